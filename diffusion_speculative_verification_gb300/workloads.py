"""Seeded synthetic inputs for the verification pass and the acceptance step.

This module only *draws* inputs; it holds none of the method's arithmetic
(no mask, no RoPE, no attention, no acceptance rule).  Both the CUDA path
(through the bindings) and the CPU oracle consume exactly the arrays made
here, so a parity test compares the two on identical bytes.

Shapes follow the five named workloads of the verification problem:

* ``tiny``     1 sequence, 1 head, head_dim 64, fp32, 16 cached prompt keys,
               block width B=4; acceptance over a 256-token vocabulary with
               logits ~ N(0, 2) (variance 2), T=0 and T=1 Gumbel.
* ``gqa1p7b``  8 sequences, 16 q / 8 kv heads, head_dim 128, bf16, 1024
               cached keys, B=8; greedy acceptance over 151936 tokens, gamma=8.
* ``gqa8b``    16 sequences, 32 q / 8 kv heads, 4096 cached keys, B=32;
               rejection sampling at T=1 with gamma=16, draft logits =
               target logits + N(0, 0.5^2).
* ``prefill``  4 sequences, 32 q / 8 kv heads, 8192 fresh prompt rows under
               a causal mask plus a B=16 paired tail, no cache.
* ``sweep``    64 sequences, 32 q / 8 kv heads, cache length ~ U[256, 8192],
               B drawn from {4, 8, 16, 32} per sequence; coupled-noise
               acceptance over 151936 tokens at T in {0, 1, 1.5}.

Generator: numpy PCG64 seeded per workload; normals by numpy's fp32
standard normal (scaled in fp32); bf16 values are fp32 draws rounded to
nearest-even.  Large arrays and per-row tables are drawn in pieces on worker
threads, each piece from a generator seeded by (one draw of the workload's
generator, piece index), so the values never depend on the thread count.  Uniforms that
the acceptance rule consumes (u for accept tests, u' for the emitted sample)
and the Gumbel table G = -log(-log U), U in the open interval (0, 1), are
drawn here and passed to both sides as inputs.
"""
from __future__ import annotations

import dataclasses
from typing import Dict, List, Optional

import numpy as np

F32 = "f32"
BF16 = "bf16"

MODE_ARGMAX = 0
MODE_GUMBEL = 1
MODE_REJECT = 2
MODE_GUMBEL_GEN = 3
MODE_NAMES = {"argmax": MODE_ARGMAX, "gumbel": MODE_GUMBEL, "reject": MODE_REJECT, "gumbel_gen": MODE_GUMBEL_GEN}

#: Per-sequence record, same field order as ``ssv_seq`` in include/ssv.h.
SEQ_FIELDS = ("cache_len", "new_len", "block", "q_off", "kv_off", "tau_off")


# --------------------------------------------------------------------------
# bf16 helpers (storage format only)
# --------------------------------------------------------------------------
def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round fp32 values to bf16 (nearest-even); returns the uint16 bit patterns."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    lsb = (u >> np.uint32(16)) & np.uint32(1)
    return ((u + np.uint32(0x7FFF) + lsb) >> np.uint32(16)).astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.ascontiguousarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def values_f64(arr: np.ndarray, dtype: str) -> np.ndarray:
    """Exact float64 values of a stored array (bf16 bits or fp32)."""
    if dtype == BF16:
        return bf16_bits_to_f32(arr).astype(np.float64)
    return np.asarray(arr, dtype=np.float32).astype(np.float64)


def _store(x32: np.ndarray, dtype: str) -> np.ndarray:
    return f32_to_bf16_bits(x32) if dtype == BF16 else np.ascontiguousarray(x32, dtype=np.float32)


def _normal(rng: np.random.Generator, shape, std: float = 1.0) -> np.ndarray:
    x = rng.standard_normal(size=shape, dtype=np.float32)
    if std != 1.0:
        x *= np.float32(std)
    return x


#: arrays above this many elements are drawn in fixed-size pieces on worker
#: threads, each piece from its own generator seeded by (a draw of the parent
#: generator, piece index): the values depend only on the seed, never on the
#: thread count.
_PIECE = 1 << 22


def _pool():
    import concurrent.futures as cf
    import os
    return cf.ThreadPoolExecutor(max_workers=max(1, min(16, os.cpu_count() or 1)))


def _normal_store(rng: np.random.Generator, shape, dtype: str, std: float = 1.0) -> np.ndarray:
    """N(0, std^2) fp32 draws stored as `dtype` (bf16 bits or fp32)."""
    n = int(np.prod(shape))
    if n <= _PIECE:
        return _store(_normal(rng, shape, std), dtype)
    seed = int(rng.integers(0, 1 << 63))
    out = np.empty(n, np.uint16 if dtype == BF16 else np.float32)

    def piece(i):
        lo, hi = i * _PIECE, min(n, (i + 1) * _PIECE)
        out[lo:hi] = _store(_normal(np.random.default_rng([seed, i]), hi - lo, std), dtype)

    with _pool() as ex:
        list(ex.map(piece, range((n + _PIECE - 1) // _PIECE)))
    return out.reshape(shape)


def _rows_parallel(rng: np.random.Generator, rows: int, fn) -> None:
    """fn(row, generator) for every row, each row with its own generator
    seeded from one draw of `rng` (thread-count independent)."""
    seed = int(rng.integers(0, 1 << 63))
    with _pool() as ex:
        list(ex.map(lambda r: fn(r, np.random.default_rng([seed, r])), range(rows)))


def open_uniform(rng: np.random.Generator, shape) -> np.ndarray:
    """fp64 uniforms strictly inside (0, 1): (k + 0.5) / 2^53."""
    k = rng.integers(0, 1 << 53, size=shape, dtype=np.uint64)
    return (k.astype(np.float64) + 0.5) * (1.0 / float(1 << 53))


def gumbel_table(rng: np.random.Generator, rows: int, V: int) -> np.ndarray:
    """Gumbel(0,1) noise table, fp64 transform rounded to fp32, row by row."""
    out = np.empty((rows, V), dtype=np.float32)

    def row(r, g):
        out[r] = (-np.log(-np.log(open_uniform(g, V)))).astype(np.float32)

    _rows_parallel(rng, rows, row)
    return out


def uniform01_f32(rng: np.random.Generator, shape) -> np.ndarray:
    """fp32 uniforms in [0, 1) on a 2^-24 grid (exactly representable)."""
    return (rng.integers(0, 1 << 24, size=shape, dtype=np.int64).astype(np.float64) / float(1 << 24)).astype(np.float32)


# --------------------------------------------------------------------------
# layout
# --------------------------------------------------------------------------
def seq_table(cache_lens, new_lens, blocks) -> np.ndarray:
    """int32 [batch, 6] table of ``ssv_seq`` records with packed offsets."""
    cache_lens = np.asarray(cache_lens, np.int64)
    new_lens = np.asarray(new_lens, np.int64)
    blocks = np.asarray(blocks, np.int64)
    batch = len(blocks)
    rows = new_lens + 2 * blocks
    t = np.zeros((batch, 6), np.int32)
    t[:, 0] = cache_lens
    t[:, 1] = new_lens
    t[:, 2] = blocks
    t[:, 3] = np.concatenate([[0], np.cumsum(rows)[:-1]]) if batch else []
    t[:, 4] = np.concatenate([[0], np.cumsum(cache_lens)[:-1]]) if batch else []
    t[:, 5] = np.concatenate([[0], np.cumsum(blocks)[:-1]]) if batch else []
    return t


def random_tau(rng: np.random.Generator, B: int) -> np.ndarray:
    """Stage map: a uniformly random permutation of 1..B (slot k -> stage tau[k])."""
    return (rng.permutation(B) + 1).astype(np.int32)


@dataclasses.dataclass
class AttnInputs:
    name: str
    dtype: str
    Hq: int
    Hkv: int
    d: int
    rope_base: float
    seqs: np.ndarray          # int32 [batch, 6]
    tau: np.ndarray           # int32 [sum B], 1..B per sequence
    q_raw: np.ndarray         # [rows, Hq, d]  (pre-RoPE), bf16 bits or fp32
    k_new_raw: np.ndarray     # [rows, Hkv, d] (pre-RoPE)
    v_new: np.ndarray         # [rows, Hkv, d]
    k_cache: np.ndarray       # [sum C, Hkv, d] (already rotated by the caller)
    v_cache: np.ndarray       # [sum C, Hkv, d]

    @property
    def batch(self) -> int:
        return int(self.seqs.shape[0])

    @property
    def total_rows(self) -> int:
        return int(self.q_raw.shape[0])

    @property
    def total_cache(self) -> int:
        return int(self.k_cache.shape[0])


@dataclasses.dataclass
class AcceptInputs:
    name: str
    mode: int
    T: float
    V: int
    logits_dtype: str
    blocks: np.ndarray        # int32 [batch]
    gammas: np.ndarray        # int32 [batch], 0 <= gamma <= B
    slot_off: np.ndarray      # int32 [batch], first slot of each sequence
    tau: np.ndarray           # int32 [sum B]
    logits: np.ndarray        # [sum B, V] target logits of the mask slots, slot order
    draft_logits: Optional[np.ndarray]   # [sum B, V] same storage as logits (reject mode)
    draft_tokens: np.ndarray  # int32 [sum B], draft token of each slot
    noise: Optional[np.ndarray]          # [n_noise, V] fp32 Gumbel table (gumbel mode)
    noise_row: np.ndarray     # int32 [sum B], table row per slot
    u_accept: np.ndarray      # fp32 [sum B], uniforms for the accept tests
    u_sample: np.ndarray      # fp32 [batch], uniform for the emitted sample
    noise_seed: int = 0       # generated coupled noise: key of the generator (noise_row holds positions)

    @property
    def batch(self) -> int:
        return int(self.blocks.shape[0])


# --------------------------------------------------------------------------
# generators
# --------------------------------------------------------------------------
def make_attn_inputs(name: str, cache_lens, new_lens, blocks, Hq: int, Hkv: int, d: int,
                     dtype: str, seed: int, rope_base: float = 10000.0) -> AttnInputs:
    rng = np.random.default_rng(seed)
    seqs = seq_table(cache_lens, new_lens, blocks)
    rows = int(np.sum(np.asarray(new_lens) + 2 * np.asarray(blocks)))
    total_c = int(np.sum(cache_lens))
    tau = np.concatenate([random_tau(rng, int(b)) for b in blocks]).astype(np.int32) \
        if len(blocks) else np.zeros(0, np.int32)
    q = _normal_store(rng, (rows, Hq, d), dtype)
    kn = _normal_store(rng, (rows, Hkv, d), dtype)
    vn = _normal_store(rng, (rows, Hkv, d), dtype)
    kc = _normal_store(rng, (total_c, Hkv, d), dtype)
    vc = _normal_store(rng, (total_c, Hkv, d), dtype)
    return AttnInputs(name, dtype, Hq, Hkv, d, rope_base, seqs, tau, q, kn, vn, kc, vc)


PLANT_LOGIT = 40.0


def make_accept_inputs(name: str, mode: int, T: float, V: int, blocks, gammas, seed: int,
                       logits_dtype: str = F32, logit_std: float = 2.0 ** 0.5,
                       draft_noise_std: float = 0.5, tau: Optional[np.ndarray] = None) -> AcceptInputs:
    """Acceptance inputs with planted agreement.

    For each sequence a cut stage c is drawn uniformly in 1..gamma+1.  Greedy
    and coupled-noise modes: at stages before c the draft token's target
    logit is raised to PLANT_LOGIT, which makes it the winner with
    overwhelming probability; other stages carry uniform random draft tokens.
    Reject mode: at stages before c the draft row is an exact copy of the
    target row (ratio exactly 1), later stages use target + N(0, 0.5^2).
    Planting only shapes the distribution of accepted lengths; both sides
    compute the outcome from the same bytes.
    """
    rng = np.random.default_rng(seed)
    blocks = np.asarray(blocks, np.int32)
    gammas = np.asarray(gammas, np.int32)
    batch = len(blocks)
    S = int(blocks.sum())
    slot_off = np.concatenate([[0], np.cumsum(blocks)[:-1]]).astype(np.int32) if batch else np.zeros(0, np.int32)
    if tau is None:
        tau = np.concatenate([random_tau(rng, int(b)) for b in blocks]).astype(np.int32) if batch else np.zeros(0, np.int32)
    logits32 = np.empty((S, V), np.float32)

    def logit_row(r, g):
        logits32[r] = _normal(g, V, logit_std)

    _rows_parallel(rng, S, logit_row)
    draft_tokens = rng.integers(0, V, size=S).astype(np.int32)
    draft32 = None
    if mode == MODE_REJECT:
        draft32 = np.empty((S, V), np.float32)
    for b in range(batch):
        B, g, off = int(blocks[b]), int(gammas[b]), int(slot_off[b])
        cut = int(rng.integers(1, g + 2))
        slot_of_stage = np.empty(B, np.int64)
        slot_of_stage[tau[off:off + B] - 1] = np.arange(B)
        for s in range(1, B + 1):
            k = off + int(slot_of_stage[s - 1])
            if mode == MODE_REJECT:
                if s < cut:
                    draft32[k] = logits32[k]
                else:
                    draft32[k] = logits32[k] + _normal(rng, V, draft_noise_std)
            elif s < cut:
                logits32[k, draft_tokens[k]] = PLANT_LOGIT
    logits = _store(logits32, logits_dtype)
    draft = None if draft32 is None else _store(draft32, logits_dtype)
    noise = None
    noise_row = np.zeros(S, np.int32)
    noise_seed = 0
    if mode == MODE_GUMBEL:
        noise_row = rng.permutation(S).astype(np.int32)
        noise = gumbel_table(rng, S, V)
    elif mode == MODE_GUMBEL_GEN:
        # one position per slot (distinct, any 32-bit pattern), one generator key
        noise_row = (int(rng.integers(0, 1 << 30)) + rng.permutation(S)).astype(np.int32)
        noise_seed = int(rng.integers(0, 1 << 63))
    u_accept = uniform01_f32(rng, S)
    u_sample = uniform01_f32(rng, batch)
    return AcceptInputs(name, mode, float(T), V, logits_dtype, blocks, gammas, slot_off, tau,
                        logits, draft, draft_tokens, noise, noise_row, u_accept, u_sample, noise_seed)


# --------------------------------------------------------------------------
# named workloads
# --------------------------------------------------------------------------
VOCAB = 151936

WORKLOADS: Dict[str, dict] = {
    "tiny": dict(batch=1, Hq=1, Hkv=1, d=64, dtype=F32, seed=1001,
                 accept=[("argmax", 0.0), ("gumbel", 1.0)], V=256, gamma="B"),
    "gqa1p7b": dict(batch=8, Hq=16, Hkv=8, d=128, dtype=BF16, seed=1002,
                    accept=[("argmax", 0.0)], V=VOCAB, gamma="B"),
    "gqa8b": dict(batch=16, Hq=32, Hkv=8, d=128, dtype=BF16, seed=1003,
                  accept=[("reject", 1.0)], V=VOCAB, gamma=16),
    "prefill": dict(batch=4, Hq=32, Hkv=8, d=128, dtype=BF16, seed=1004,
                    accept=[], V=VOCAB, gamma="B"),
    "sweep": dict(batch=64, Hq=32, Hkv=8, d=128, dtype=BF16, seed=1005,
                  accept=[("gumbel", 0.0), ("gumbel", 1.0), ("gumbel", 1.5)], V=VOCAB, gamma="B"),
}


def workload_lengths(name: str, seed: Optional[int] = None):
    """(cache_lens, new_lens, blocks) of a named workload."""
    w = WORKLOADS[name]
    seed = w["seed"] if seed is None else seed
    b = w["batch"]
    if name == "tiny":
        return [16], [0], [4]
    if name == "gqa1p7b":
        return [1024] * b, [0] * b, [8] * b
    if name == "gqa8b":
        return [4096] * b, [0] * b, [32] * b
    if name == "prefill":
        return [0] * b, [8192] * b, [16] * b
    if name == "sweep":
        rng = np.random.default_rng(seed + 7919)
        cache = rng.integers(256, 8192 + 1, size=b).tolist()
        blocks = rng.choice([4, 8, 16, 32], size=b).tolist()
        return cache, [0] * b, blocks
    raise KeyError(name)


def workload_attn(name: str, seed: Optional[int] = None) -> AttnInputs:
    w = WORKLOADS[name]
    seed = w["seed"] if seed is None else seed
    c, n, b = workload_lengths(name, seed)
    return make_attn_inputs(name, c, n, b, w["Hq"], w["Hkv"], w["d"], w["dtype"], seed)


def workload_gammas(name: str, blocks) -> List[int]:
    g = WORKLOADS[name]["gamma"]
    return [int(x) if g == "B" else min(int(g), int(x)) for x in blocks]


def workload_accept(name: str, which: int = 0, seed: Optional[int] = None,
                    tau: Optional[np.ndarray] = None) -> AcceptInputs:
    w = WORKLOADS[name]
    seed = w["seed"] if seed is None else seed
    mode_name, T = w["accept"][which]
    _, _, blocks = workload_lengths(name, seed)
    return make_accept_inputs(f"{name}/{mode_name}/T={T}", MODE_NAMES[mode_name], T, w["V"], blocks,
                              workload_gammas(name, blocks), seed + 100 * (which + 1), tau=tau)


@dataclasses.dataclass
class CommitInputs:
    """Inputs of the commit step: the pass's fresh rows (from an AttnInputs),
    accepted-stage counts, and destination caches laid out with room."""
    attn: AttnInputs
    n_acc: np.ndarray         # int32 [batch], 0..B
    dst_off: np.ndarray       # int32 [batch], first destination row of each sequence
    dst_cap: np.ndarray       # int32 [batch], rows of room from dst_off
    k_dst: np.ndarray         # [dst_rows, Hkv, d] prior contents (same storage as the fresh rows)
    v_dst: np.ndarray


def commit_layout(a: AttnInputs, seed: int, slack: int = 3):
    """Destination layout of the commit step: each sequence gets C + N + B +
    slack rows of room, with a gap of `slack` rows between sequences; accepted
    counts are uniform on 0..B.  Returns (n_acc, dst_off, dst_cap, dst_rows)
    and the generator, positioned for the destination contents."""
    rng = np.random.default_rng(seed)
    C = a.seqs[:, 0].astype(np.int64)
    N = a.seqs[:, 1].astype(np.int64)
    B = a.seqs[:, 2].astype(np.int64)
    cap = C + N + B + slack
    off = np.concatenate([[slack], slack + np.cumsum(cap + slack)[:-1]]) if len(cap) else np.zeros(0, np.int64)
    rows = int(off[-1] + cap[-1] + slack) if len(cap) else 1
    n_acc = np.array([rng.integers(0, int(b) + 1) for b in B], np.int32)
    return n_acc, off.astype(np.int32), cap.astype(np.int32), rows, rng


def make_commit_inputs(a: AttnInputs, seed: int, slack: int = 3) -> CommitInputs:
    """commit_layout plus destination rows holding seeded random values (so
    rows the commit must not touch can be checked)."""
    n_acc, off, cap, rows, rng = commit_layout(a, seed, slack)
    shape = (rows, a.Hkv, a.d)
    k_dst = _normal_store(rng, shape, a.dtype)
    v_dst = _normal_store(rng, shape, a.dtype)
    return CommitInputs(a, n_acc, off, cap, k_dst, v_dst)


# --------------------------------------------------------------------------
# fused LM head + acceptance
# --------------------------------------------------------------------------
@dataclasses.dataclass
class LmheadInputs:
    """Inputs of the fused LM head + acceptance: the acceptance metadata (an
    AcceptInputs whose logits are None) plus the final hidden states of the
    mask slots and the LM head."""
    acc: AcceptInputs
    hidden: int
    h: np.ndarray             # bf16 bits [total_slots, hidden], row = slot (slot order)
    w: np.ndarray             # bf16 bits [V, hidden]


#: hidden width, acceptance mode and temperature of the fused LM head per
#: named workload (hidden = query heads x head_dim of the workload's layer)
LMHEAD: Dict[str, tuple] = {
    "tiny": (64, "gumbel", 1.0),
    "gqa1p7b": (2048, "argmax", 0.0),
    "gqa8b": (4096, "argmax", 0.0),
    "sweep": (4096, "gumbel", 1.0),
}


def lm_head_matrix(rng: np.random.Generator, V: int, hidden: int) -> np.ndarray:
    """Synthetic LM head [V, hidden] as bf16 bit patterns drawn directly: a
    random sign, a random 7-bit mantissa and exponent 2^-1 or 2^0, i.e.
    |x| uniform over the bf16 values in [0.5, 2) (mean 0, E x^2 about 1.46).
    Drawn in row blocks to bound the temporaries."""
    w = np.empty((V, hidden), np.uint16)
    step = max(1, (1 << 26) // max(hidden, 1))
    for r0 in range(0, V, step):
        r1 = min(V, r0 + step)
        n = (r1 - r0) * hidden
        u = rng.integers(0, 1 << 32, size=(n + 1) // 2, dtype=np.uint32).view(np.uint16)[:n].reshape(r1 - r0, hidden)
        # bit 15 sign, bit 8 picks exponent 126 or 127 (moved to bit 7), bits 0..6 mantissa
        e = u & np.uint16(0x0100)
        e >>= np.uint16(1)
        u &= np.uint16(0x807F)
        u |= np.uint16(0x3F00)
        u |= e
        w[r0:r1] = u
    return w


def make_lmhead_inputs(name: str, mode: int, T: float, V: int, hidden: int, blocks, gammas, seed: int,
                       plant: float = 64.0, tau: Optional[np.ndarray] = None,
                       w: Optional[np.ndarray] = None) -> LmheadInputs:
    """Hidden states with planted agreement.

    Rows are h = z + (plant / |w_t|^2) w_t with z ~ N(0, 1/hidden) per entry
    and w_t row t of the stored LM head (lm_head_matrix), so that the score
    of token t sits near `plant` while the others are about N(0, 1.5).  Per
    sequence a cut stage c is drawn uniformly in 1..gamma+1: stages before c
    plant the slot's draft token; stage c (if c <= B) plants a different
    random token; later stages are z alone.  Planting only shapes the accepted
    lengths; both sides compute the outcome from the same bytes.  `w` reuses
    an LM head drawn earlier (same V and hidden)."""
    rng = np.random.default_rng(seed)
    blocks = np.asarray(blocks, np.int32)
    gammas = np.asarray(gammas, np.int32)
    batch = len(blocks)
    S = int(blocks.sum())
    slot_off = np.concatenate([[0], np.cumsum(blocks)[:-1]]).astype(np.int32) if batch else np.zeros(0, np.int32)
    if tau is None:
        tau = np.concatenate([random_tau(rng, int(b)) for b in blocks]).astype(np.int32) if batch else np.zeros(0, np.int32)
    if w is None:
        w = lm_head_matrix(rng, V, hidden)
    assert w.shape == (V, hidden)
    h32 = _normal(rng, (S, hidden), 1.0 / np.sqrt(hidden))
    draft_tokens = rng.integers(0, V, size=S).astype(np.int32)
    for b in range(batch):
        B, g, off = int(blocks[b]), int(gammas[b]), int(slot_off[b])
        cut = int(rng.integers(1, g + 2))
        slot_of_stage = np.empty(B, np.int64)
        slot_of_stage[tau[off:off + B] - 1] = np.arange(B)
        for s in range(1, min(cut, B) + 1):
            k = off + int(slot_of_stage[s - 1])
            t = int(draft_tokens[k])
            if s == cut:
                t = int((t + 1 + rng.integers(0, V - 1)) % V) if V > 1 else t
            wt = bf16_bits_to_f32(w[t])
            h32[k] += np.float32(plant / float(np.dot(wt.astype(np.float64), wt))) * wt
    h = f32_to_bf16_bits(h32)
    noise = None
    noise_row = np.zeros(S, np.int32)
    if mode == MODE_GUMBEL:
        noise_row = rng.permutation(S).astype(np.int32)
        noise = gumbel_table(rng, S, V)
    acc = AcceptInputs(name, mode, float(T), V, F32, blocks, gammas, slot_off, tau, None, None, draft_tokens,
                       noise, noise_row, uniform01_f32(rng, S), uniform01_f32(rng, batch))
    return LmheadInputs(acc, hidden, h, w)


def workload_lmhead(name: str, seed: Optional[int] = None, w: Optional[np.ndarray] = None) -> LmheadInputs:
    """The named workload's verified slots under the fused LM head."""
    wl = WORKLOADS[name]
    seed = wl["seed"] if seed is None else seed
    hidden, mode_name, T = LMHEAD[name]
    _, _, blocks = workload_lengths(name, seed)
    V = wl["V"]
    return make_lmhead_inputs(f"{name}/lmhead/{mode_name}/T={T}", MODE_NAMES[mode_name], T, V, hidden, blocks,
                              workload_gammas(name, blocks), seed + 500, w=w)


# --------------------------------------------------------------------------
# tree (state-set) verification
# --------------------------------------------------------------------------
#: Per-sequence record of a tree batch, field order of ssv_tree_seq in include/ssv.h.
TREE_FIELDS = ("cache_len", "new_len", "block", "n_edges", "q_off", "k_off", "kv_off", "edge_off", "o_off")


@dataclasses.dataclass
class TreeInputs:
    """One draft tree per sequence over a block of B positions, with the
    attention inputs of the tree pass and (optionally) planted acceptance
    inputs.  Layout: query rows N + B per sequence (fresh prompt rows, then
    one mask-slot row per position) at q_off; new key/value rows N + E + B
    (fresh rows, one data row per edge, one mask row per position) at k_off;
    output and logits rows N + (E + 1) B at o_off (fresh rows, then node-major
    (node, position))."""
    name: str
    dtype: str
    Hq: int
    Hkv: int
    d: int
    seqs: np.ndarray          # int32 [batch, 9] (TREE_FIELDS)
    parent: np.ndarray        # int32 [sum E], -1 = root
    pos: np.ndarray           # int32 [sum E]
    token: np.ndarray         # int32 [sum E]
    q: np.ndarray             # [sum (N + B), Hq, d] (post-RoPE), bf16 bits or fp32
    k_new: np.ndarray         # [sum (N + E + B), Hkv, d]
    v_new: np.ndarray
    k_cache: np.ndarray       # [sum C, Hkv, d]
    v_cache: np.ndarray
    # acceptance (None when not drawn)
    mode: int = MODE_ARGMAX
    T: float = 0.0
    V: int = 0
    logits: Optional[np.ndarray] = None   # fp32 [sum (N + (E+1) B), V]
    noise: Optional[np.ndarray] = None    # fp32 [sum B, V] (coupled noise)
    noise_row: Optional[np.ndarray] = None  # int32 [sum B]
    pos_off: Optional[np.ndarray] = None  # int32 [batch]: first noise_row entry of each sequence
    planted: Optional[list] = None        # per sequence: (edges of the planted path, planted emission (p, v) or None)

    @property
    def batch(self) -> int:
        return int(self.seqs.shape[0])

    @property
    def total_out(self) -> int:
        s = self.seqs
        return int(np.sum(s[:, 1] + (s[:, 3] + 1) * s[:, 2])) if len(s) else 0


def random_tree(rng: np.random.Generator, B: int, E: int):
    """E edges over a block of B positions: each edge hangs under a random
    earlier node (half the time the newest one, so paths grow deep) and commits
    a random position still undecided there.  Returns (parent, pos) int32."""
    committed = [0]
    parent, pos = [], []
    for e in range(E):
        for _ in range(64):
            par = e - 1 if (e > 0 and rng.random() < 0.5) else int(rng.integers(-1, e))
            und = [p for p in range(B) if not (committed[par + 1] >> p) & 1]
            if und:
                break
        else:
            par, und = -1, list(range(B))
        p = int(rng.choice(und))
        parent.append(par)
        pos.append(p)
        committed.append(committed[par + 1] | (1 << p))
    return np.asarray(parent, np.int32), np.asarray(pos, np.int32)


def make_tree_inputs(name: str, cache_lens, new_lens, blocks, n_edges, Hq: int, Hkv: int, d: int, dtype: str,
                     seed: int, V: int = 0, mode: int = MODE_ARGMAX, T: float = 0.0) -> TreeInputs:
    """Seeded tree-pass inputs; with V > 0 also acceptance inputs with a
    planted target path: per sequence a cut depth is drawn; along the tree
    from the root, while above the cut, one existing child edge is made the
    target's transition (its token's logit raised to 40 in the row of its
    position, which makes it both the decision and the most confident
    position); at the cut node a transition outside the tree is planted the
    same way.  Planting only shapes the accepted lengths."""
    rng = np.random.default_rng(seed)
    C = np.asarray(cache_lens, np.int64)
    N = np.asarray(new_lens, np.int64)
    B = np.asarray(blocks, np.int64)
    E = np.asarray(n_edges, np.int64)
    batch = len(B)
    cum = lambda x: np.concatenate([[0], np.cumsum(x)[:-1]]) if batch else np.zeros(0, np.int64)  # noqa: E731
    seqs = np.zeros((batch, 9), np.int32)
    seqs[:, 0], seqs[:, 1], seqs[:, 2], seqs[:, 3] = C, N, B, E
    seqs[:, 4] = cum(N + B)
    seqs[:, 5] = cum(N + E + B)
    seqs[:, 6] = cum(C)
    seqs[:, 7] = cum(E)
    seqs[:, 8] = cum(N + (E + 1) * B)
    parent, pos = [], []
    for b in range(batch):
        pa, po = random_tree(rng, int(B[b]), int(E[b]))
        parent.append(pa)
        pos.append(po)
    parent = np.concatenate(parent).astype(np.int32) if batch else np.zeros(0, np.int32)
    pos = np.concatenate(pos).astype(np.int32) if batch else np.zeros(0, np.int32)
    token = rng.integers(0, max(V, 1), size=len(parent)).astype(np.int32)
    q = _normal_store(rng, (int(np.sum(N + B)), Hq, d), dtype)
    kn = _normal_store(rng, (int(np.sum(N + E + B)), Hkv, d), dtype)
    vn = _normal_store(rng, (int(np.sum(N + E + B)), Hkv, d), dtype)
    kc = _normal_store(rng, (int(np.sum(C)), Hkv, d), dtype)
    vc = _normal_store(rng, (int(np.sum(C)), Hkv, d), dtype)
    t = TreeInputs(name, dtype, Hq, Hkv, d, seqs, parent, pos, token, q, kn, vn, kc, vc)
    if V <= 0:
        return t
    total_out = t.total_out
    logits = np.empty((total_out, V), np.float32)

    def row(r, g):
        logits[r] = _normal(g, V, 2.0 ** 0.5)

    _rows_parallel(rng, total_out, row)
    planted = []
    for b in range(batch):
        Bb, Eb, e0, o0, Nb = int(B[b]), int(E[b]), int(seqs[b, 7]), int(seqs[b, 8]), int(N[b])
        pa, po, tk = parent[e0:e0 + Eb], pos[e0:e0 + Eb], token[e0:e0 + Eb]
        cut = int(rng.integers(0, Bb + 1))
        n, committed, depth = 0, 0, 0
        path, emit = [], None
        while True:
            und = [p for p in range(Bb) if not (committed >> p) & 1]
            if not und:
                break
            kids = [e for e in range(Eb) if int(pa[e]) + 1 == n]
            if depth < cut and kids:
                e = int(rng.choice(kids))
                logits[o0 + Nb + n * Bb + int(po[e]), int(tk[e])] = 40.0
                committed |= 1 << int(po[e])
                path.append(e)
                n, depth = e + 1, depth + 1
                continue
            # a transition outside the tree: a position and token no child has
            p = int(rng.choice(und))
            bad = {int(tk[e]) for e in kids if int(po[e]) == p}
            v = int(rng.integers(0, V))
            if V > len(bad):
                while v in bad:
                    v = int(rng.integers(0, V))
            logits[o0 + Nb + n * Bb + p, v] = 40.0
            emit = (p, v)
            break
        planted.append((path, emit))
    t.mode, t.T, t.V, t.logits, t.planted = mode, float(T), V, logits, planted
    if mode == MODE_GUMBEL:
        t.pos_off = cum(B).astype(np.int32)
        t.noise_row = rng.permutation(int(np.sum(B))).astype(np.int32)
        t.noise = gumbel_table(rng, int(np.sum(B)), V)
    return t
