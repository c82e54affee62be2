"""Helpers shared by the GPU parity tests: build the library, run the CUDA
path through the binding, run the oracle on the same bytes, compare."""
import numpy as np

from diffusion_speculative_verification_gb300 import build, ssv, io as sio
from diffusion_speculative_verification_gb300 import workloads as W
import oracle.rope as orope
import oracle.attention as oattn
import oracle.accept as oacc

_built = False


def ensure_built():
    global _built
    if not _built:
        build.build()
        _built = True


def bf16_ulp(x):
    """Spacing of bf16 numbers at |x| (8 significant bits)."""
    ax = np.maximum(np.abs(x), 2.0 ** -126)
    return 2.0 ** (np.floor(np.log2(ax)) - 7)


def gpu_rope(a: W.AttnInputs, in_place=False):
    """Returns (q_rot, k_rot) torch tensors from ssv_rope_copy."""
    t = sio.attn_to_device(a)
    if in_place:
        ssv.rope_copy(t["q"], t["k_new"], t["batch"], a.rope_base)
        return t["q"], t["k_new"], t
    qo = t["q"].clone().zero_()
    ko = t["k_new"].clone().zero_()
    ssv.rope_copy(t["q"], t["k_new"], t["batch"], a.rope_base, q_out=qo, k_out=ko)
    return qo, ko, t


def gpu_verify(a: W.AttnInputs, out_dtype=None, rows_of=None):
    """Full GPU path rope -> attention.  Returns (O_gpu f64, oracle f64 on the GPU's post-RoPE bytes, extras)."""
    import torch
    qo, ko, t = gpu_rope(a)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    od = {None: None, "f32": torch.float32, "bf16": torch.bfloat16}[out_dtype]
    o = ssv.verify_attn(qo, t["k_cache"], t["v_cache"], ko, t["v_new"], t["batch"], t["tau"], out_dtype=od,
                        dev_status=status)
    assert ssv.get_status(status) == ssv.SSV_OK
    got = W.values_f64(sio.to_numpy_storage(o), W.BF16 if o.dtype == torch.bfloat16 else W.F32)
    q64 = W.values_f64(sio.to_numpy_storage(qo), a.dtype)
    k64 = W.values_f64(sio.to_numpy_storage(ko), a.dtype)
    ref = oattn.verify_attention(a.seqs, a.tau, q64, W.values_f64(a.k_cache, a.dtype),
                                 W.values_f64(a.v_cache, a.dtype), k64, W.values_f64(a.v_new, a.dtype),
                                 rows_of=rows_of)
    return got, ref, dict(t=t, qo=qo, ko=ko, o=o, status=status)


def compare_attn(got, ref, out_is_bf16, in_is_f32):
    """Asserts the stated tolerance on rows the oracle computed; returns max abs error."""
    m = ~np.isnan(ref)
    assert m.any()
    err = np.abs(got[m] - ref[m])
    if in_is_f32:
        tol = 1e-5
        assert err.max() <= tol, f"max abs err {err.max():.3g} > {tol}"
    elif not out_is_bf16:
        assert err.max() <= 1e-2, f"max abs err {err.max():.3g} > 1e-2"
    else:
        bound = 1e-2 + 2.0 ** -8 * np.abs(ref[m])
        assert np.all(err <= bound), f"max excess {(err - bound).max():.3g}"
    return float(err.max())


def gpu_accept(x: W.AcceptInputs, dev_status=None, workspace=None):
    d = sio.accept_to_device(x)
    n_acc, n_out, tokens = ssv.accept(d["mode"], d["T"], d["logits"], d["draft_tokens"], d["tau"], d["block"],
                                      d["gamma"], d["slot_off"], draft_logits=d["draft_logits"], noise=d["noise"],
                                      noise_row=d["noise_row"], u_accept=d["u_accept"], u_sample=d["u_sample"],
                                      max_block=d["max_block"], dev_status=dev_status, workspace=workspace)
    return n_acc.cpu().numpy(), n_out.cpu().numpy(), tokens.cpu().numpy()


REJECT_MARGIN = 1e-4        # decisions closer than this (in log space) may flip under fp32 rounding
SAMPLE_REL_TOL = 1e-5       # inverse-CDF crossing tolerance, relative to the total mass


def compare_accept(x: W.AcceptInputs, got):
    """Bit-exact n_acc / n_out / tokens; for rejection sampling the emitted
    sample may sit on a neighbouring token when u'Z lies within the stated
    rounding band of a CDF boundary (checked against the oracle's fp64 CDF).
    Returns the number of emitted samples that differ (all of them valid)."""
    n_acc, n_out, tokens = got
    ref = oacc.accept_batch(x)
    differ = 0
    for b, r in enumerate(ref["results"]):
        if x.mode == W.MODE_REJECT:
            assert all(m > REJECT_MARGIN for m in r.accept_margins), \
                f"seq {b}: decision inside the rounding band; pick another seed"
        assert n_acc[b] == r.n_acc, f"seq {b}: n_acc {n_acc[b]} vs {r.n_acc}"
        assert n_out[b] == r.n_out, f"seq {b}: n_out {n_out[b]} vs {r.n_out}"
        off, B = int(x.slot_off[b]), int(x.blocks[b])
        g = tokens[off:off + B]
        assert g[:r.n_acc].tolist() == r.tokens[:r.n_acc]
        assert np.all(g[r.n_out:] == -1)
        if r.n_out > r.n_acc:
            want = r.tokens[-1]
            have = int(g[r.n_acc])
            if r.emit_kind in ("residual", "bonus"):
                if have != want:
                    assert oacc.emission_valid(r, have, SAMPLE_REL_TOL), \
                        f"seq {b}: emitted {have}, oracle {want}, outside the band"
                    differ += 1
            else:
                assert have == want, f"seq {b}: emitted {have} vs {want}"
    return differ


def random_attn_shape(seed, dtype=None, d=128):
    """Seeded random batch: group size, tail widths (1..64), ragged caches and
    prompts, so that plans, one- and two-tile units, split units and warps whose
    rows straddle stage slot 32 vary from seed to seed."""
    import numpy as np
    from diffusion_speculative_verification_gb300 import workloads as W
    rng = np.random.default_rng(seed)
    Hkv = int(rng.choice([1, 2, 4, 8]))
    G = int(rng.choice([1, 2, 4, 8]))
    batch = int(rng.integers(1, 9))
    cache = [int(rng.choice([0, rng.integers(1, 400), rng.integers(400, 3000)])) for _ in range(batch)]
    new = [int(rng.choice([0, 0, rng.integers(1, 300)])) for _ in range(batch)]
    blocks = [int(rng.integers(1, 65)) for _ in range(batch)]
    return W.make_attn_inputs("r", cache, new, blocks, G * Hkv, Hkv, d, W.BF16 if dtype is None else dtype,
                              1000 + seed)
