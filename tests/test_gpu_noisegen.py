"""GPU parity of coupled-noise acceptance with the noise generated on the
device (SSV_ACCEPT_GUMBEL_GEN; SPOT review, "How it is used": one Gumbel
value per absolute output position and token, shared by drafter and
target).  Both sides evaluate the same generator (Philox4x32-10 at the
slot's position, then -L(-L(U)) in one fixed sequence of fp32 operations)
and compare identical fp32 scores, so n_acc, n_out and tokens are bit-exact.
The streaming kernel scores exactly only the tokens whose cheap upper bound
reaches the warp's best exact score; these tests check that the filter never
changes a decision (full vocabulary, small vocabularies where whole warps
hold no token, bf16 logits, unaligned rows through the general kernel)."""
import numpy as np
import pytest

from diffusion_speculative_verification_gb300 import workloads as W
from gpu_common import ensure_built, gpu_accept, compare_accept

pytestmark = pytest.mark.gpu

GEN = W.MODE_GUMBEL_GEN


def setup_module():
    ensure_built()


CASES = {
    # sweep-like: full vocabulary, blocks of 4..32, gamma = B
    "sweep_T1": dict(T=1.0, V=151936, blocks=[4, 32, 8, 16, 4, 32, 16, 8], gammas=[4, 32, 8, 16, 4, 32, 16, 8]),
    "sweep_T1.5": dict(T=1.5, V=151936, blocks=[16, 8, 32, 4], gammas=[16, 8, 32, 4]),
    "T0.7_partial_gamma": dict(T=0.7, V=50000, blocks=[8, 16, 1], gammas=[3, 16, 0]),
    "tiny_vocab": dict(T=1.0, V=100, blocks=[8, 8], gammas=[8, 5]),
    "one_token": dict(T=1.0, V=1, blocks=[3], gammas=[3]),
    "bf16_logits": dict(T=1.0, V=30000, blocks=[8, 4], gammas=[8, 2], logits_dtype=W.BF16),
    "T0_is_argmax": dict(T=0.0, V=20000, blocks=[8, 4], gammas=[8, 4]),
}


@pytest.mark.parametrize("name", list(CASES))
def test_generated_noise_parity(name):
    kw = dict(CASES[name])
    x = W.make_accept_inputs(name, GEN, kw.pop("T"), kw.pop("V"), kw.pop("blocks"), kw.pop("gammas"),
                             seed=sum(map(ord, name)) + 5000, **kw)
    compare_accept(x, gpu_accept(x))


def test_generated_noise_unaligned_rows_general_kernel():
    from test_gpu_accept import _accept_with_logits_offset
    x = W.make_accept_inputs("unal", GEN, 1.0, 20000, [8, 16, 4], [8, 16, 2], seed=5101)
    aligned = gpu_accept(x)
    shifted = _accept_with_logits_offset(x, 1)
    compare_accept(x, aligned)
    compare_accept(x, shifted)


def test_generated_noise_many_slots_general_kernel():
    blocks = [4] * 530   # 2120 slots: more than the streaming kernel lists
    gammas = [int(g) for g in np.random.default_rng(5102).integers(0, 5, size=len(blocks))]
    x = W.make_accept_inputs("many", GEN, 1.0, 640, blocks, gammas, seed=5103)
    compare_accept(x, gpu_accept(x))


@pytest.mark.parametrize("seed", range(6))
def test_generated_noise_random(seed):
    rng = np.random.default_rng(7000 + seed)
    V = int(rng.choice([int(rng.integers(1, 3000)), 8 * int(rng.integers(500, 8000))]))
    batch = int(rng.integers(1, 10))
    blocks = [int(rng.integers(1, 65)) for _ in range(batch)]
    gammas = [int(rng.integers(0, b + 1)) for b in blocks]
    T = float(rng.choice([0.5, 1.0, 1.3, 2.0]))
    dt = W.BF16 if rng.random() < 0.3 else W.F32
    x = W.make_accept_inputs(f"gen{seed}", GEN, T, V, blocks, gammas, seed=7100 + seed, logits_dtype=dt)
    compare_accept(x, gpu_accept(x))
