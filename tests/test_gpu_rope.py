"""GPU parity of ssv_rope_copy against the fp64 oracle (SimSD summary,
section 3: each mask slot reuses its data token's RoPE index).

fp32: max abs error <= 1e-5.
bf16: |gpu - ref| <= ulp_bf16(ref) + 2^-21 (|x_i| + |x_{i+d/2}|).  The
kernel rotates in fp32 and rounds once to bf16: the rounding is at most
half an ulp; the fp32 rotation adds at most ~4e-7 (|x_i| + |x_{i+d/2}|)
(angle reduced in fp64 then rounded to fp32: 2^-24 pi; cos/sin and the two
products: a few 2^-24), which dominates where the two terms cancel and the
output is far smaller than its inputs."""
import numpy as np
import pytest

from diffusion_speculative_verification_gb300 import workloads as W, io as sio
import oracle.rope as orope
from gpu_common import ensure_built, gpu_rope, bf16_ulp, random_attn_shape

pytestmark = pytest.mark.gpu

CASES = {
    "tiny": lambda: W.workload_attn("tiny"),
    "ragged_bf16": lambda: W.make_attn_inputs("r", [0, 300, 129], [0, 200, 5], [1, 32, 7], 8, 2, 128, W.BF16, 21),
    "d64_bf16": lambda: W.make_attn_inputs("r", [77, 130], [0, 40], [4, 5], 4, 4, 64, W.BF16, 22),
    "f32_d128": lambda: W.make_attn_inputs("r", [9000, 3], [3, 0], [64, 2], 4, 2, 128, W.F32, 23),
    "gqa1p7b": lambda: W.workload_attn("gqa1p7b"),
    "prefill": lambda: W.workload_attn("prefill"),
    "random_bf16_a": lambda: random_attn_shape(200),
    "random_bf16_b": lambda: random_attn_shape(201, W.BF16, 64),
    "random_f32": lambda: random_attn_shape(202, W.F32, 128),
}


def setup_module():
    ensure_built()


@pytest.mark.parametrize("name", list(CASES))
@pytest.mark.parametrize("in_place", [False, True])
def test_rope_parity(name, in_place):
    a = CASES[name]()
    qo, ko, _ = gpu_rope(a, in_place=in_place)
    q_ref, k_ref = orope.rope_copy_batch(a.seqs, W.values_f64(a.q_raw, a.dtype), W.values_f64(a.k_new_raw, a.dtype),
                                         a.rope_base)
    gq = W.values_f64(sio.to_numpy_storage(qo), a.dtype)
    gk = W.values_f64(sio.to_numpy_storage(ko), a.dtype)
    for got, ref, raw in ((gq, q_ref, a.q_raw), (gk, k_ref, a.k_new_raw)):
        err = np.abs(got - ref)
        if a.dtype == W.F32:
            assert err.max() <= 1e-5, err.max()
        else:
            x = np.abs(W.values_f64(raw, a.dtype))
            half = x.shape[-1] // 2
            pair = np.concatenate([x[..., :half] + x[..., half:]] * 2, axis=-1)
            bound = bf16_ulp(ref) + 2.0 ** -21 * pair
            assert np.all(err <= bound), (err / bound).max()
            assert np.mean(err <= 0.5 * bf16_ulp(ref) + 1e-12) > 0.99   # almost all correctly rounded


def test_pair_rows_bit_identical():
    a = W.make_attn_inputs("r", [100, 7], [3, 0], [16, 5], 8, 2, 128, W.BF16, 24)
    for C, N, B, off, *_ in a.seqs:
        a.q_raw[off + N + B:off + N + 2 * B] = a.q_raw[off + N:off + N + B]
        a.k_new_raw[off + N + B:off + N + 2 * B] = a.k_new_raw[off + N:off + N + B]
    qo, ko, _ = gpu_rope(a)
    q = sio.to_numpy_storage(qo)
    k = sio.to_numpy_storage(ko)
    for C, N, B, off, *_ in a.seqs:
        np.testing.assert_array_equal(q[off + N:off + N + B], q[off + N + B:off + N + 2 * B])
        np.testing.assert_array_equal(k[off + N:off + N + B], k[off + N + B:off + N + 2 * B])
