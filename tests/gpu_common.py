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
                                      max_block=d["max_block"], dev_status=dev_status, workspace=workspace,
                                      noise_seed=d["noise_seed"])
    return n_acc.cpu().numpy(), n_out.cpu().numpy(), tokens.cpu().numpy()


# Rejection test u < p(d)/q(d): the device forms the ratio as
# 2^(((l_d - M_a) - (q_d - M_b)) c2) S_b / S_a with fp32 c2, an fp32-rounded
# exponent and fp32 exp2, over chunk sums of ex2.approx weights (about 2^-22
# each) merged in double-float arithmetic, then the quotient (one correction
# step) and the product in fp32 (three more roundings of 2^-24): the log
# ratio is within |arg| 2^-22 + 2^-19 + 2^-22 of the exact one, below 2.6e-5
# for |arg| <= 100.  Decisions closer than 1e-4 (log space) to the threshold
# would be inside that band; the seeded sets have none.
REJECT_MARGIN = 1e-4

# Emitted sample (residual or bonus): the device computes every weight in
# double-float arithmetic (relative error EPS_W, from the exponential's
# argument, Taylor remainder, table and product roundings) and every sum as
# a tree of at most 64 double-float additions, each within 2^-47 of its
# result (EPS_ACC).  The oracle's fp64 cumulative sum of V terms is within
# V 2^-53 of exact at either end.
EPS_W = 1e-12
EPS_ACC = 64 * 2.0 ** -47


def emission_band(res, V: int) -> float:
    """Bound, relative to the total mass Z of the sampled weights, on how far
    the device's and the oracle's normalised CDFs can lie apart; outside it
    the two must choose the same token."""
    oracle = 2.0 * V * 2.0 ** -53
    if res.emit_kind == "residual":
        zr = float(res.sample_cdf[-1])            # mass of (p - q)_+ in probability units
        eps_s = EPS_W + EPS_ACC                   # device normalisers S_a, S_b
        dev = 2.0 * ((2.0 * (EPS_W + eps_s + 2.0 ** -46) + 2.0 ** -46) / zr + EPS_ACC)
        return dev + oracle + 4.0 * (V + 3) * 2.0 ** -53 / zr + 1e-14
    return 2.0 * (EPS_W + EPS_ACC) + oracle + 1e-14


def compare_accept(x: W.AcceptInputs, got):
    """Bit-exact n_acc / n_out / tokens.  For rejection sampling every accept
    test's margin must exceed REJECT_MARGIN and every emitted sample's margin
    (oracle.accept.sample_margin) must exceed emission_band: the seeded sets
    hold no decision inside a rounding band, and the token is then unique.
    Returns the smallest emitted-sample margin / band ratio seen (inf if none)."""
    n_acc, n_out, tokens = got
    ref = oacc.accept_batch(x)
    worst = float("inf")
    for b, r in enumerate(ref["results"]):
        if x.mode == W.MODE_REJECT:
            assert all(m > REJECT_MARGIN for m in r.accept_margins), \
                f"seq {b}: accept test inside the rounding band; pick another seed"
        assert n_acc[b] == r.n_acc, f"seq {b}: n_acc {n_acc[b]} vs {r.n_acc}"
        assert n_out[b] == r.n_out, f"seq {b}: n_out {n_out[b]} vs {r.n_out}"
        off, B = int(x.slot_off[b]), int(x.blocks[b])
        g = tokens[off:off + B]
        assert g[:r.n_acc].tolist() == r.tokens[:r.n_acc]
        assert np.all(g[r.n_out:] == -1)
        if r.n_out > r.n_acc:
            if r.emit_kind in ("residual", "bonus"):
                margin, band = oacc.sample_margin(r), emission_band(r, x.V)
                assert margin > band, f"seq {b}: emitted sample {margin:.3g} from a CDF boundary, inside the " \
                                      f"rounding band {band:.3g}; pick another seed"
                worst = min(worst, margin / band)
            assert int(g[r.n_acc]) == r.tokens[-1], f"seq {b}: emitted {int(g[r.n_acc])} vs {r.tokens[-1]}"
    return worst


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
