"""GPU parity of ssv_verify_attn against the fp64 oracle on the same
post-RoPE bytes (SimSD summary, section 2, temporal attention mask).

Tolerances: fp32 inputs max abs <= 1e-5; bf16 inputs with fp32 output
max abs <= 1e-2; bf16 output |err| <= 1e-2 + 2^-8 |ref| (output rounding).
Full-size workloads compare every row (decode-shaped) or every tail row
plus sampled prompt rows (prefill)."""
import numpy as np
import pytest
import torch

from diffusion_speculative_verification_gb300 import workloads as W, ssv, io as sio
import oracle.attention as oattn
from gpu_common import ensure_built, gpu_verify, compare_attn, random_attn_shape

pytestmark = pytest.mark.gpu

SMALL = {
    "tiny": lambda: W.workload_attn("tiny"),
    "ragged": lambda: W.make_attn_inputs("r", [0, 300, 129], [0, 200, 5], [1, 32, 7], 8, 2, 128, W.BF16, 31),
    "decode_gqa": lambda: W.make_attn_inputs("r", [1000, 257, 64, 1], [0] * 4, [8, 64, 3, 16], 16, 4, 128, W.BF16, 32),
    "d64": lambda: W.make_attn_inputs("r", [77, 130], [0, 40], [4, 5], 4, 4, 64, W.BF16, 33),
    "mha_prefill_small": lambda: W.make_attn_inputs("r", [0, 64], [300, 129], [16, 2], 4, 4, 128, W.BF16, 34),
    "f32_multi": lambda: W.make_attn_inputs("r", [33, 0, 200], [0, 20, 7], [4, 1, 9], 4, 2, 64, W.F32, 35),
    "empty_cache_B1": lambda: W.make_attn_inputs("r", [0], [0], [1], 2, 1, 128, W.BF16, 36),
    # B > 32 with warps whose tail rows straddle stage slot 32 (G = 4: 8 rows a warp)
    "tail_B33_B47": lambda: W.make_attn_inputs("r", [0, 100], [0, 0], [33, 47], 16, 4, 128, W.BF16, 46),
    # large query groups: an M-tile holds 4 query rows x 32 heads, or 1 row x 128 heads
    "group32": lambda: W.make_attn_inputs("r", [700, 0, 129], [0, 40, 3], [8, 5, 16], 64, 2, 128, W.BF16, 47),
    "group128": lambda: W.make_attn_inputs("r", [300, 1], [7, 0], [3, 2], 128, 1, 128, W.BF16, 48),
}


def setup_module():
    ensure_built()


@pytest.mark.parametrize("name", list(SMALL))
@pytest.mark.parametrize("out", ["f32", "bf16"])
def test_attn_small(name, out):
    a = SMALL[name]()
    if a.dtype == W.F32 and out == "bf16":
        pytest.skip("fp32 inputs produce fp32 outputs")
    got, ref, _ = gpu_verify(a, out_dtype=out)
    compare_attn(got, ref, out == "bf16", a.dtype == W.F32)


# Units split across CTAs (partials merged by the rank holding each unit's
# head): in two and three pieces, across every CTA of a head (one long unit
# per head, more than four partials) with one M-tile and with two, and a mix
# of one-tile (S double-buffered) and two-tile units, split, in one launch.
SPLIT = {
    "split2": lambda: W.make_attn_inputs("s", [4096] * 8, [0] * 8, [8] * 8, 16, 8, 128, W.BF16, 41),
    "split3": lambda: W.make_attn_inputs("s", [3000, 3100, 2900, 3333, 3050], [0] * 5, [4, 8, 2, 16, 4], 8, 8, 128,
                                         W.BF16, 42),
    "split_many": lambda: W.make_attn_inputs("s", [8192], [0], [16], 32, 8, 128, W.BF16, 43),
    "split_many_two_tiles": lambda: W.make_attn_inputs("s", [16384], [0], [32], 32, 8, 128, W.BF16, 44),
    "mixed_tiles_split": lambda: W.make_attn_inputs("s", [2500, 700, 4100, 1900, 3000, 130], [0, 0, 40, 0, 0, 0],
                                                    [32, 4, 16, 32, 8, 24], 32, 8, 128, W.BF16, 45),
}


@pytest.mark.parametrize("name", list(SPLIT))
def test_attn_split_units(name):
    a = SPLIT[name]()
    got, ref, _ = gpu_verify(a, out_dtype="bf16")
    compare_attn(got, ref, True, False)


@pytest.mark.parametrize("seed", range(8))
def test_attn_random_shapes(seed):
    a = random_attn_shape(seed)
    got, ref, _ = gpu_verify(a, out_dtype="f32")
    compare_attn(got, ref, False, False)


# fp32 inputs (exact SIMT path), head dims 64 and 128
@pytest.mark.parametrize("seed", range(4))
def test_attn_random_shapes_f32(seed):
    a = random_attn_shape(100 + seed, W.F32, 64 if seed % 2 else 128)
    got, ref, _ = gpu_verify(a)
    compare_attn(got, ref, False, True)


def test_attn_plan_tables_in_workspace():
    """130 sequences with two M-tiles: the per-sequence plan tables exceed the
    shared memory left by the pipeline and live in the workspace."""
    rng = np.random.default_rng(49)
    n = 130
    cache = [int(v) for v in rng.integers(0, 600, size=n)]
    blocks = [32 if i % 7 == 0 else int(rng.integers(1, 17)) for i in range(n)]
    a = W.make_attn_inputs("r", cache, [0] * n, blocks, 32, 8, 128, W.BF16, 49)
    got, ref, _ = gpu_verify(a, out_dtype="bf16")
    compare_attn(got, ref, True, False)


@pytest.mark.parametrize("name", ["gqa1p7b", "gqa8b", "sweep"])
def test_attn_full_decode_shapes(name):
    a = W.workload_attn(name)
    got, ref, _ = gpu_verify(a, out_dtype="f32")
    compare_attn(got, ref, False, False)


def test_attn_full_prefill_sampled():
    a = W.workload_attn("prefill")
    rows = oattn.rows_sample(a.seqs, 24, np.random.default_rng(7))
    got, ref, _ = gpu_verify(a, out_dtype="f32", rows_of=rows)
    compare_attn(got, ref, False, False)


def test_attn_bf16_output_full_gqa8b():
    a = W.workload_attn("gqa8b")
    got, ref, _ = gpu_verify(a, out_dtype="bf16")
    compare_attn(got, ref, True, False)


@pytest.mark.parametrize("dtype", [W.BF16, W.F32])
def test_no_leak_bit_identical(dtype):
    """Perturbing keys a row must not see leaves that row's output bit-identical."""
    a = W.make_attn_inputs("r", [260, 5], [0, 130], [12, 6], 8, 2, 128 if dtype == W.BF16 else 64, dtype, 37)
    t = sio.attn_to_device(a)
    o1 = ssv.verify_attn(t["q"], t["k_cache"], t["v_cache"], t["k_new"], t["v_new"], t["batch"], t["tau"])
    kn = t["k_new"].clone()
    vn = t["v_new"].clone()
    rng = np.random.default_rng(0)
    checks = []
    for b, (C, N, B, off, _kv, toff) in enumerate(a.seqs):
        tau = a.tau[toff:toff + B]
        i = int(rng.integers(0, B))                        # a mask row D~_i
        hidden = [N + j for j in range(B) if tau[j] >= tau[i]] + [N + B + j for j in range(B) if tau[j] < tau[i]]
        for r in hidden:
            kn[off + r] += 3.0
            vn[off + r] -= 2.0
        checks.append(off + N + B + i)
    o2 = ssv.verify_attn(t["q"], t["k_cache"], t["v_cache"], kn, vn, t["batch"], t["tau"])
    for r in checks:
        assert torch.equal(o1[r], o2[r])
    # fresh prompt rows never see the tail
    kn = t["k_new"].clone()
    for C, N, B, off, *_ in a.seqs:
        kn[off + N:off + N + 2 * B] += 5.0
    o3 = ssv.verify_attn(t["q"], t["k_cache"], t["v_cache"], kn, t["v_new"], t["batch"], t["tau"])
    for C, N, B, off, *_ in a.seqs:
        assert torch.equal(o1[off:off + N], o3[off:off + N])


def test_bad_tau_reports_status():
    a = W.make_attn_inputs("r", [40], [0], [4], 2, 1, 128, W.BF16, 38)
    t = sio.attn_to_device(a)
    t["tau"][:] = torch.tensor([1, 1, 2, 3], dtype=torch.int32)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    ssv.verify_attn(t["q"], t["k_cache"], t["v_cache"], t["k_new"], t["v_new"], t["batch"], t["tau"], dev_status=st)
    assert ssv.get_status(st) == ssv.SSV_ERR_BAD_TAU
    assert ssv.get_status(st) == ssv.SSV_OK          # reading clears it


def test_host_validation_on_device_buffers():
    a = W.make_attn_inputs("r", [40], [0], [4], 2, 1, 128, W.BF16, 39)
    t = sio.attn_to_device(a)
    with pytest.raises(ssv.SsvError) as e:
        ssv.verify_attn(t["q"][:, :, 1:], t["k_cache"], t["v_cache"], t["k_new"], t["v_new"], t["batch"], t["tau"])
    assert e.value.code in (ssv.SSV_ERR_INVALID, ssv.SSV_ERR_UNSUPPORTED)
