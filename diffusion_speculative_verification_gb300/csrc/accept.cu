// ssv_accept: acceptance in temporal order with the longest accepted prefix
// (the shared records, arithmetic and completion steps are in accept.cuh).
//
// Reduce kernels:
//   accept_stream   (accept_stream.cu) the default: persistent, one CTA per
//                   SM, rows streamed through a shared-memory ring by bulk
//                   copies.  Needs 16-byte aligned rows and at most
//                   kStrMaxRows slots.
//   accept_reduce   (below) any shape: grid = slots x vocab chunks, one
//                   streaming pass of register loads per (row, chunk).
// Both write one AccPartial per (verified row, chunk) and finish through the
// row-merge / sequence-walk steps.
//   accept_emit_norm, accept_sample   (rejection sampling only, below)
//                   the emitted token in double-float arithmetic: the
//                   emission row's normalisers, then its chunk masses and
//                   the inverse-CDF search.
#include "accept.cuh"
#include "dfloat.cuh"

namespace ssv {

constexpr int kAccThreads = 256;
constexpr int kAccVec = 4;                                 // elements per vector access
constexpr int kAccIters = 8;                               // vector accesses per thread per stream
constexpr int kAccPerThread = kAccVec * kAccIters;         // 32
static_assert(kAccThreads * kAccPerThread == kAccChunk, "one chunk per CTA");

// 4 consecutive elements starting at i (i % 4 == 0, row base suitably aligned), streaming load
template <typename T>
__device__ __forceinline__ void ld_vec4(const void* base, size_t i, float* out) {
  if constexpr (sizeof(T) == 4) {
    const float4 v = __ldcs(reinterpret_cast<const float4*>(static_cast<const float*>(base) + i));
    out[0] = v.x; out[1] = v.y; out[2] = v.z; out[3] = v.w;
  } else {
    const uint2 v = __ldcs(reinterpret_cast<const uint2*>(static_cast<const __nv_bfloat16*>(base) + i));
    out[0] = __uint_as_float(v.x << 16); out[1] = __uint_as_float(v.x & 0xffff0000u);
    out[2] = __uint_as_float(v.y << 16); out[3] = __uint_as_float(v.y & 0xffff0000u);
  }
}

// Loads this thread's kAccPerThread entries of a chunk: entry (it, k) is vocab
// index c0 + (it * kAccThreads + tid) * 4 + k, so a thread's indices increase
// with (it, k).  Entries past V read as `fill`.
template <typename T>
__device__ __forceinline__ void ld_chunk(const void* base, size_t rbase, int c0, int V, bool vec, float fill,
                                         float* x) {
  const int tid = threadIdx.x;
#pragma unroll
  for (int it = 0; it < kAccIters; ++it) {
    const int e = c0 + (it * kAccThreads + tid) * kAccVec;
    if (vec && e + kAccVec <= V) {
      ld_vec4<T>(base, rbase + e, x + it * kAccVec);
    } else {
#pragma unroll
      for (int k = 0; k < kAccVec; ++k) x[it * kAccVec + k] = (e + k < V) ? ld_logit<T>(base, rbase + e + k) : fill;
    }
  }
}

__device__ __forceinline__ int chunk_index(int c0, int j) {  // vocab index of a thread's j-th entry
  return c0 + ((j / kAccVec) * kAccThreads + (int)threadIdx.x) * kAccVec + (j % kAccVec);
}

// ---- block reductions (256 threads) ---------------------------------------

// result valid in thread 0
__device__ void block_argmax(float& v, int& i) {
  __shared__ float sv[kAccThreads / 32];
  __shared__ int si[kAccThreads / 32];
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1)
    argmax_combine(v, i, __shfl_xor_sync(0xffffffffu, v, o), __shfl_xor_sync(0xffffffffu, i, o));
  if (lane == 0) { sv[wid] = v; si[wid] = i; }
  __syncthreads();
  if (threadIdx.x == 0) {
    for (int w = 1; w < kAccThreads / 32; ++w) argmax_combine(v, i, sv[w], si[w]);
  }
}

// all threads receive the maxima
__device__ void block_max2(float& a, float& b) {
  __shared__ float sa[kAccThreads / 32], sb[kAccThreads / 32];
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, o));
    b = fmaxf(b, __shfl_xor_sync(0xffffffffu, b, o));
  }
  if (lane == 0) { sa[wid] = a; sb[wid] = b; }
  __syncthreads();
  a = sa[0];
  b = sb[0];
#pragma unroll
  for (int w = 1; w < kAccThreads / 32; ++w) { a = fmaxf(a, sa[w]); b = fmaxf(b, sb[w]); }
}

// compensated sums of two (hi, lo) pairs, fixed order; result valid in thread 0
__device__ void block_sum2x2(float& h1, float& l1, float& h2, float& l2) {
  __shared__ float s[4][kAccThreads / 32];
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float a = __shfl_xor_sync(0xffffffffu, h1, o), b = __shfl_xor_sync(0xffffffffu, l1, o);
    const float c = __shfl_xor_sync(0xffffffffu, h2, o), d = __shfl_xor_sync(0xffffffffu, l2, o);
    two_sum_acc(h1, l1, a, b);
    two_sum_acc(h2, l2, c, d);
  }
  if (lane == 0) { s[0][wid] = h1; s[1][wid] = l1; s[2][wid] = h2; s[3][wid] = l2; }
  __syncthreads();
  if (threadIdx.x == 0) {
    for (int w = 1; w < kAccThreads / 32; ++w) {
      two_sum_acc(h1, l1, s[0][w], s[1][w]);
      two_sum_acc(h2, l2, s[2][w], s[3][w]);
    }
  }
}

template <int MODE, typename T>
__global__ void __launch_bounds__(kAccThreads)
accept_reduce_kernel(const AcceptParams p) {
  __shared__ int s_ok;
  __shared__ WalkSmem s_walk;
  const int slot = blockIdx.x / p.nchunks;
  const int chunk = blockIdx.x % p.nchunks;
  const int b = find_seq_by_slot(p.slot_off, p.batch, slot);
  if (b < 0) return;
  const int off = p.slot_off[b];
  const int B = p.block[b], g = p.gamma[b];
  if (B < 1 || slot - off >= B) return;
  const int need = min(g + 1, B);
  const int st = p.tau[slot];
  if (st < 1 || st > need) return;  // not a verified row (a bad map is reported below)
  const int tid = threadIdx.x;
  const size_t rbase = (size_t)slot * p.V;
  const int c0 = chunk * kAccChunk;
  const bool vec = p.vec != 0;

  // ---- streaming loads first (all in flight), validation overlaps them
  float xa[kAccPerThread], xb[kAccPerThread];
  const bool draft = (MODE == SSV_ACCEPT_REJECT) && st <= g;
  const float* nrow = nullptr;
  bool nrow_ok = true;
  if (MODE == SSV_ACCEPT_GUMBEL) {
    const int nr = p.noise_row[slot];
    nrow_ok = nr >= 0 && nr < p.n_noise_rows;
    nrow = p.noise + (size_t)(nrow_ok ? nr : 0) * p.V;
  }
  ld_chunk<T>(p.logits, rbase, c0, p.V, vec, -INFINITY, xa);
  if (MODE == SSV_ACCEPT_GUMBEL) ld_chunk<float>(nrow, 0, c0, p.V, vec, 0.f, xb);
  if (draft) ld_chunk<T>(p.draft_logits, rbase, c0, p.V, vec, -INFINITY, xb);
  if (tid < 32) {
    const bool ok = warp_seq_valid(p, b);
    if (tid == 0) {
      s_ok = ok && nrow_ok;
      if (!ok && slot == off + 0 && chunk == 0) report(p.dev_status, SSV_ERR_BAD_TAU);
      if (!nrow_ok && chunk == 0) report(p.dev_status, SSV_ERR_INVALID);
    }
  }
  __syncthreads();
  if (!s_ok) return;

  AccPartial out;
  if (MODE == SSV_ACCEPT_GUMBEL_GEN) {
    // every entry's noise generated here: entries (it, 0..3) are 4 consecutive
    // tokens, one generator call
    const bool unit_t = p.T == 1.0f;
    const uint32_t pos = (uint32_t)p.noise_row[slot];
#pragma unroll
    for (int it = 0; it < kAccIters; ++it) {
      const int e = chunk_index(c0, it * kAccVec);
      const uint4 w = noise::philox4x32_10(make_uint4((uint32_t)e >> 2, pos, 0u, 0u), (uint32_t)p.noise_seed,
                                           (uint32_t)(p.noise_seed >> 32));
      const uint32_t wq[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
      for (int k = 0; k < kAccVec; ++k) xa[it * kAccVec + k] = gen_score(xa[it * kAccVec + k], wq[k], p.T, unit_t);
    }
  }
  if (MODE != SSV_ACCEPT_REJECT) {
    if (MODE == SSV_ACCEPT_GUMBEL) {
      const bool unit_t = p.T == 1.0f;  // l / 1 is exact
#pragma unroll
      for (int j = 0; j < kAccPerThread; ++j)
        xa[j] = __fadd_rn(unit_t ? xa[j] : __fdiv_rn(xa[j], p.T), xb[j]);
    }
    float best = -INFINITY;
    int bi = INT_MAX;
#pragma unroll
    for (int j = 0; j < kAccPerThread; ++j) {
      const int e = chunk_index(c0, j);
      if (e < p.V && (xa[j] > best || bi == INT_MAX)) { best = xa[j]; bi = e; }
    }
    block_argmax(best, bi);
    out.val = best; out.idx = bi;
    out.m_a = out.m_b = out.sa_hi = out.sa_lo = out.sb_hi = out.sb_lo = 0.f;
  } else {
    float ma = -INFINITY, mb = -INFINITY;
#pragma unroll
    for (int j = 0; j < kAccPerThread; ++j) {
      ma = fmaxf(ma, xa[j]);
      if (draft) mb = fmaxf(mb, xb[j]);
    }
    block_max2(ma, mb);
    const float nma = -ma * p.c2, nmb = -mb * p.c2;
    float sa = 0.f, ca = 0.f, sb = 0.f, cb = 0.f;
#pragma unroll
    for (int j = 0; j < kAccPerThread; ++j) {
      kahan_add(sa, ca, ex2f(fmaf(xa[j], p.c2, nma)));
      if (draft) kahan_add(sb, cb, ex2f(fmaf(xb[j], p.c2, nmb)));
    }
    float la = -ca, lb = -cb;
    block_sum2x2(sa, la, sb, lb);
    out.m_a = ma; out.m_b = mb;
    out.sa_hi = sa; out.sa_lo = la; out.sb_hi = sb; out.sb_lo = lb;
    out.val = 0.f; out.idx = 0;
  }
  if (tid == 0) p.part[(size_t)slot * p.nchunks + chunk] = out;
  if (tid < 32)
    warp_rows_done<MODE, T>(p, b, slot, 1, __ldcg(&p.tau[slot]), p.slot_off[b], p.block[b], p.gamma[b], s_walk,
                            nullptr);
}

// ---- rejection sampling: emitted token ------------------------------------
// The emitted token is the smallest v whose cumulative weight exceeds u' Z
// (inverse CDF).  It is computed in double-float arithmetic (dfloat.cuh):
// every weight to about 5e-13 relative and every sum as a tree of depth
// below 32 double-float additions, so the token can differ from the exact
// one only when u' Z lies within about 1e-12 Z of a CDF boundary (for a
// residual sample, that divided by the residual's total mass).  The row is
// cut into sub-chunks of kEmitSub entries, one CTA each, 8 consecutive
// entries per thread:
//   accept_emit_norm   for a residual sample, each sub-chunk's sums of
//                      e_a = 2^((l - m_a) c2) and e_b = 2^((ql - m_b) c2)
//                      (unnormalised p and q).
//   accept_sample      every CTA of sequence b adds the sub-chunk sums in the
//                      same fixed order (S_a, S_b), forms the weights
//                      w = (e_a S_b - e_b S_a)_+ (the residual (p - q)_+ scaled
//                      by S_a S_b) and e_a (p scaled by S_a), and writes its
//                      masses per warp and per sub-chunk; the last CTA finds
//                      the sub-chunk, then the warp, then (one warp, one
//                      thread's 8 entries per lane) the entry where the
//                      cumulative mass passes u' Z (fp64 prefix sums of the
//                      exact pair values; the residual unless it vanished,
//                      then p).

struct EmitCtx {
  bool residual;
  float ma, mb;  // row maxima of the logits and the draft logits
  dfx c2;        // log2(e) / T
  dfx sa, sb;    // S_a, S_b (residual only)
};

// residual weight (e_a S_b - e_b S_a)_+ and p weight e_a of one entry
__device__ __forceinline__ void emit_weights(const EmitCtx& c, float la, float lb, const float2* tab, dfx& wr,
                                             dfx& wp) {
  const dfx ea = dfx_exp2_diff(la, c.ma, c.c2, tab);
  wp = ea;
  wr = dfx{0.f, 0.f};
  if (c.residual) {
    const dfx eb = dfx_exp2_diff(lb, c.mb, c.c2, tab);
    const dfx d = dfx_add(dfx_mul(ea, c.sb), dfx_mul(dfx{-eb.hi, -eb.lo}, c.sa));
    if (d.hi > 0.f) wr = d;
  }
}

__device__ __forceinline__ dfx shfl_xor_dfx(dfx a, int o) {
  return dfx{__shfl_xor_sync(0xffffffffu, a.hi, o), __shfl_xor_sync(0xffffffffu, a.lo, o)};
}

// The 8 consecutive entries [e0, e0 + 8) of a row (fill -inf past V).
template <typename T>
__device__ __forceinline__ void ld_run8(const void* base, size_t rbase, int e0, int V, bool vec, float* x) {
  if (vec && e0 + 8 <= V) {
    if constexpr (sizeof(T) == 4) {
      const float4* p4 = reinterpret_cast<const float4*>(static_cast<const float*>(base) + rbase + e0);
      const float4 a = __ldcg(p4), b = __ldcg(p4 + 1);
      x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w; x[4] = b.x; x[5] = b.y; x[6] = b.z; x[7] = b.w;
    } else {  // rows are 8-byte aligned (V % 4 == 0): two 4-entry loads
      const uint2* p2 = reinterpret_cast<const uint2*>(static_cast<const __nv_bfloat16*>(base) + rbase + e0);
      const uint2 u = __ldcg(p2), v = __ldcg(p2 + 1);
      const uint32_t w[4] = {u.x, u.y, v.x, v.y};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        x[2 * i] = __uint_as_float(w[i] << 16);
        x[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
      }
    }
  } else {
#pragma unroll
    for (int i = 0; i < 8; ++i) x[i] = (e0 + i < V) ? ld_logit<T>(base, rbase + e0 + i) : -INFINITY;
  }
}

// Common prologue of the two emission kernels: validity of sequence b (reads
// only the call's inputs, so it runs before the wait), the 2^(j/256) table
// into shared memory, then the wait for the reduce kernel's records.
__device__ __forceinline__ bool emit_prologue(const AcceptParams& p, int b, float2* s_tab, int* s_ok) {
  const int tid = threadIdx.x;
  if (tid < 32) {
    const bool ok = warp_seq_valid(p, b);
    if (tid == 0) *s_ok = ok;
  }
  dfx_exp2_table(p.e2pow, s_tab, tid);  // kAccThreads == 256 entries
  __syncthreads();
  pdl_wait();  // emission records, accepted lengths and row normalisers
  pdl_trigger();
  return *s_ok != 0;
}

static_assert(kAccThreads == 256 && kEmitSub == 8 * kAccThreads, "one table entry and 8 row entries per thread");

template <typename T>
__global__ void __launch_bounds__(kAccThreads)
accept_emit_norm_kernel(const AcceptParams p) {
  __shared__ int s_ok;
  __shared__ float2 s_tab[256];
  __shared__ float4 s_w[kAccThreads / 32];
  const int b = blockIdx.x / p.nsub;
  const int sub = blockIdx.x % p.nsub;
  // A sequence whose stage map or sizes were rejected never ran its walk,
  // so its emission record may be stale: skip it.
  if (!emit_prologue(p, b, s_tab, &s_ok)) return;
  const int eslot = p.emit[2 * b];
  const int soff = p.slot_off[b];
  if (eslot < soff || eslot >= soff + p.block[b] || p.emit[2 * b + 1] == 0) return;  // bonus: no normaliser needed
  const SlotNorm nm = p.norm[eslot];
  const dfx c2{p.c2_hi, p.c2_lo};
  const size_t rbase = (size_t)eslot * p.V;
  const int e0 = sub * kEmitSub + threadIdx.x * 8;
  float xa[8], xb[8];
  ld_run8<T>(p.logits, rbase, e0, p.V, p.vec != 0, xa);
  ld_run8<T>(p.draft_logits, rbase, e0, p.V, p.vec != 0, xb);
  dfx sa{0.f, 0.f}, sb{0.f, 0.f};
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    sa = dfx_add(sa, dfx_exp2_diff(xa[j], nm.m_a, c2, s_tab));
    sb = dfx_add(sb, dfx_exp2_diff(xb[j], nm.m_b, c2, s_tab));
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    sa = dfx_add(sa, shfl_xor_dfx(sa, o));
    sb = dfx_add(sb, shfl_xor_dfx(sb, o));
  }
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  if (lane == 0) s_w[wid] = make_float4(sa.hi, sa.lo, sb.hi, sb.lo);
  __syncthreads();
  if (threadIdx.x == 0) {
    for (int w = 1; w < kAccThreads / 32; ++w) {
      sa = dfx_add(sa, dfx{s_w[w].x, s_w[w].y});
      sb = dfx_add(sb, dfx{s_w[w].z, s_w[w].w});
    }
    p.enorm[(size_t)b * p.nsub + sub] = make_float4(sa.hi, sa.lo, sb.hi, sb.lo);
  }
}

template <typename T>
__global__ void __launch_bounds__(kAccThreads)
accept_sample_kernel(const AcceptParams p) {
  __shared__ int s_ok, s_last;
  __shared__ float2 s_tab[256];
  __shared__ float4 s_w[kAccThreads / 32];
  __shared__ float4 s_S;
  const int b = blockIdx.x / p.nsub;
  const int sub = blockIdx.x % p.nsub;
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  if (!emit_prologue(p, b, s_tab, &s_ok)) return;
  const int eslot = p.emit[2 * b];
  const int soff = p.slot_off[b];
  const int nacc = p.n_acc[b];
  if (eslot < soff || eslot >= soff + p.block[b] || nacc < 0 || nacc >= p.block[b]) return;
  const SlotNorm nm = p.norm[eslot];
  EmitCtx c;
  c.residual = p.emit[2 * b + 1] != 0;
  c.ma = nm.m_a;
  c.mb = nm.m_b;
  c.c2 = dfx{p.c2_hi, p.c2_lo};
  c.sa = c.sb = dfx{0.f, 0.f};
  if (c.residual) {
    // S_a, S_b: warp 0 adds the sub-chunk sums, lane l over sub-chunks l, l + 32, ...,
    // then a butterfly; the same fixed order in every CTA of the sequence
    if (wid == 0) {
      const float4* en = p.enorm + (size_t)b * p.nsub;
      dfx a{0.f, 0.f}, bb{0.f, 0.f};
      for (int k = lane; k < p.nsub; k += 32) {
        const float4 v = __ldcg(en + k);
        a = dfx_add(a, dfx{v.x, v.y});
        bb = dfx_add(bb, dfx{v.z, v.w});
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        a = dfx_add(a, shfl_xor_dfx(a, o));
        bb = dfx_add(bb, shfl_xor_dfx(bb, o));
      }
      if (lane == 0) s_S = make_float4(a.hi, a.lo, bb.hi, bb.lo);
    }
    __syncthreads();
    c.sa = dfx{s_S.x, s_S.y};
    c.sb = dfx{s_S.z, s_S.w};
  }
  const size_t rbase = (size_t)eslot * p.V;
  const bool vec = p.vec != 0;
  {
    const int e0 = sub * kEmitSub + tid * 8;
    float xa[8], xb[8];
    ld_run8<T>(p.logits, rbase, e0, p.V, vec, xa);
    if (c.residual) ld_run8<T>(p.draft_logits, rbase, e0, p.V, vec, xb);
    dfx mr{0.f, 0.f}, mp{0.f, 0.f};
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      dfx wr, wp;
      emit_weights(c, xa[j], c.residual ? xb[j] : -INFINITY, s_tab, wr, wp);
      mr = dfx_add(mr, wr);
      mp = dfx_add(mp, wp);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      mr = dfx_add(mr, shfl_xor_dfx(mr, o));
      mp = dfx_add(mp, shfl_xor_dfx(mp, o));
    }
    if (lane == 0) {
      const float4 m4 = make_float4(mr.hi, mr.lo, mp.hi, mp.lo);
      s_w[wid] = m4;
      p.wmass[((size_t)b * p.nsub + sub) * 8 + wid] = m4;
    }
    __syncthreads();
    if (tid == 0) {
      for (int w = 1; w < kAccThreads / 32; ++w) {
        mr = dfx_add(mr, dfx{s_w[w].x, s_w[w].y});
        mp = dfx_add(mp, dfx{s_w[w].z, s_w[w].w});
      }
      p.smass[(size_t)b * p.nsub + sub] = make_float4(mr.hi, mr.lo, mp.hi, mp.lo);
      __threadfence();
      const int prev = atomicAdd(&p.cnt_sample[b], 1);
      s_last = (prev == p.nsub - 1);
    }
  }
  __syncthreads();
  if (!s_last || wid != 0) return;
  __threadfence();

  // ---- last CTA of sequence b, warp 0: locate u' * Z ---------------------------
  const float4* sm = p.smass + (size_t)b * p.nsub;
  double zr = 0.0, zp = 0.0;
  for (int k = lane; k < p.nsub; k += 32) {
    const float4 v = __ldcg(sm + k);
    zr += (double)v.x + (double)v.y;
    zp += (double)v.z + (double)v.w;
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    zr += __shfl_xor_sync(0xffffffffu, zr, o);
    zp += __shfl_xor_sync(0xffffffffu, zp, o);
  }
  const bool use_res = c.residual && zr > 0.0;  // (p - q)_+ vanished: sample p
  const double t = (double)p.u_sample[b] * (use_res ? zr : zp);
  auto mass = [&](const float4& v) -> double { return use_res ? (double)v.x + (double)v.y : (double)v.z + (double)v.w; };
  // level 1: the first sub-chunk whose running mass passes t (else the last non-empty one)
  double before = 0.0, before_last = 0.0, base = 0.0;
  int cs = -1, last_nz = 0;
  for (int r0 = 0; r0 < p.nsub; r0 += 32) {
    const int k = r0 + lane;
    const double m = (k < p.nsub) ? mass(__ldcg(sm + k)) : 0.0;
    double incl = m;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const double y = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += y;
    }
    const double excl = incl - m;
    const unsigned cross = __ballot_sync(0xffffffffu, k < p.nsub && base + incl > t);
    const unsigned nz = __ballot_sync(0xffffffffu, k < p.nsub && m > 0.0);
    if (cs < 0 && cross) {
      const int f = __ffs(cross) - 1;
      cs = r0 + f;
      before = base + __shfl_sync(0xffffffffu, excl, f);
    }
    if (nz) {
      const int l = 31 - __clz(nz);
      last_nz = r0 + l;
      before_last = base + __shfl_sync(0xffffffffu, excl, l);
    }
    base += __shfl_sync(0xffffffffu, incl, 31);
  }
  if (cs < 0) { cs = last_nz; before = before_last; }  // rounding left t at the very end
  // level 2: the warp of that sub-chunk (lanes 0..7 hold the 8 warp masses)
  int wsel;
  {
    const double m = (lane < 8) ? mass(__ldcg(p.wmass + ((size_t)b * p.nsub + cs) * 8 + lane)) : 0.0;
    double incl = m;
#pragma unroll
    for (int o = 1; o < 8; o <<= 1) {
      const double y = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += y;
    }
    const double excl = incl - m;
    const unsigned cross = __ballot_sync(0xffffffffu, lane < 8 && before + incl > t);
    const unsigned nz = __ballot_sync(0xffffffffu, lane < 8 && m > 0.0);
    wsel = cross ? __ffs(cross) - 1 : (nz ? 31 - __clz(nz) : 7);
    before += __shfl_sync(0xffffffffu, excl, wsel);
  }
  // level 3: that warp's 256 entries, 8 consecutive per lane
  const int e0 = cs * kEmitSub + wsel * 256 + lane * 8;
  float ya[8], yb[8];
  ld_run8<T>(p.logits, rbase, e0, p.V, vec, ya);
  if (c.residual) ld_run8<T>(p.draft_logits, rbase, e0, p.V, vec, yb);
  dfx w8[8];
  dfx run{0.f, 0.f};
  int last_pos = -1;
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    dfx wr, wp;
    emit_weights(c, ya[k], c.residual ? yb[k] : -INFINITY, s_tab, wr, wp);
    w8[k] = use_res ? wr : wp;
    run = dfx_add(run, w8[k]);
    if (w8[k].hi > 0.f) last_pos = e0 + k;
  }
  const double rm = dfx_to_double(run);
  double incl = rm;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const double y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  const double rel = t - (before + (incl - rm));  // mass still to cross at the start of this lane's run
  dfx acc{0.f, 0.f};
  int pick = INT_MAX;
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    acc = dfx_add(acc, w8[k]);
    if (pick == INT_MAX && w8[k].hi > 0.f && dfx_to_double(acc) > rel) pick = e0 + k;
  }
  // lanes are in vocabulary order: the first lane with a crossing holds the token
  const unsigned has = __ballot_sync(0xffffffffu, pick != INT_MAX);
  const int v_pick = has ? __shfl_sync(0xffffffffu, pick, __ffs(has) - 1) : INT_MAX;
  const unsigned anyw = __ballot_sync(0xffffffffu, last_pos >= 0);
  const int v_last = anyw ? __shfl_sync(0xffffffffu, last_pos, 31 - __clz(anyw)) : -1;
  if (lane == 0) {
    int v = v_pick != INT_MAX ? v_pick : v_last;
    if (v < 0) v = 0;
    p.tokens[soff + nacc] = v;
    p.cnt_sample[b] = 0;
  }
}

template <int MODE, typename T>
static cudaError_t launch_reduce_t(const AcceptParams& p, cudaStream_t st) {
  const long long g1 = (long long)p.total_slots * p.nchunks;
  if (g1 > 0x7fffffffLL) return cudaErrorInvalidValue;
  accept_reduce_kernel<MODE, T><<<(unsigned)g1, kAccThreads, 0, st>>>(p);
  return cudaGetLastError();
}

// Reduce (streaming kernel where the rows allow it) then, for rejection
// sampling, the emitted-token pass.
static cudaError_t launch_accept(const AcceptParams& p, int mode, bool bf, cudaStream_t st) {
  cudaError_t e;
  if (accept_stream_supported(p, mode, bf)) {
    e = launch_accept_stream(p, mode, bf, st);
  } else {
    switch (mode) {
      case SSV_ACCEPT_ARGMAX:
        e = bf ? launch_reduce_t<SSV_ACCEPT_ARGMAX, __nv_bfloat16>(p, st) : launch_reduce_t<SSV_ACCEPT_ARGMAX, float>(p, st);
        break;
      case SSV_ACCEPT_GUMBEL:
        e = bf ? launch_reduce_t<SSV_ACCEPT_GUMBEL, __nv_bfloat16>(p, st) : launch_reduce_t<SSV_ACCEPT_GUMBEL, float>(p, st);
        break;
      case SSV_ACCEPT_GUMBEL_GEN:
        e = bf ? launch_reduce_t<SSV_ACCEPT_GUMBEL_GEN, __nv_bfloat16>(p, st)
               : launch_reduce_t<SSV_ACCEPT_GUMBEL_GEN, float>(p, st);
        break;
      default:
        e = bf ? launch_reduce_t<SSV_ACCEPT_REJECT, __nv_bfloat16>(p, st) : launch_reduce_t<SSV_ACCEPT_REJECT, float>(p, st);
        break;
    }
  }
  if (e != cudaSuccess || mode != SSV_ACCEPT_REJECT) return e;
  const long long g2 = (long long)p.batch * p.nsub;
  if (g2 > 0x7fffffffLL) return cudaErrorInvalidValue;
  if (bf) {
    e = launch_pdl(accept_emit_norm_kernel<__nv_bfloat16>, dim3((unsigned)g2), dim3(kAccThreads), 0, st, p);
    if (e != cudaSuccess) return e;
    return launch_pdl(accept_sample_kernel<__nv_bfloat16>, dim3((unsigned)g2), dim3(kAccThreads), 0, st, p);
  }
  e = launch_pdl(accept_emit_norm_kernel<float>, dim3((unsigned)g2), dim3(kAccThreads), 0, st, p);
  if (e != cudaSuccess) return e;
  return launch_pdl(accept_sample_kernel<float>, dim3((unsigned)g2), dim3(kAccThreads), 0, st, p);
}

}  // namespace ssv

using namespace ssv;

static ssv_status accept_check(const ssv_accept_args* a, int* nchunks) {
  if (!a) return SSV_ERR_INVALID;
  if (a->mode != SSV_ACCEPT_ARGMAX && a->mode != SSV_ACCEPT_GUMBEL && a->mode != SSV_ACCEPT_REJECT &&
      a->mode != SSV_ACCEPT_GUMBEL_GEN)
    return SSV_ERR_INVALID;
  if (!isfinite(a->T) || a->T < 0.f) return SSV_ERR_NOT_FINITE;
  if (a->V < 1 || a->batch < 0 || a->total_slots < 0) return SSV_ERR_INVALID;
  if (a->max_block < 1 || a->max_block > 64) return SSV_ERR_INVALID;
  if (a->logits_dtype != SSV_F32 && a->logits_dtype != SSV_BF16) return SSV_ERR_INVALID;
  *nchunks = (a->V + kAccChunk - 1) / kAccChunk;
  if (a->batch == 0) return SSV_OK;
  if (!a->logits || !a->draft_tokens || !a->tau || !a->block || !a->gamma || !a->slot_off || !a->n_acc ||
      !a->n_out || !a->tokens)
    return SSV_ERR_INVALID;
  if (a->mode == SSV_ACCEPT_REJECT) {
    if (!(a->T > 0.f)) return SSV_ERR_INVALID;
    if (!a->draft_logits || !a->u_accept || !a->u_sample) return SSV_ERR_INVALID;
  }
  if (a->mode == SSV_ACCEPT_GUMBEL && a->T > 0.f) {
    if (!a->noise || !a->noise_row || a->n_noise_rows < 1) return SSV_ERR_INVALID;
  }
  if (a->mode == SSV_ACCEPT_GUMBEL_GEN && a->T > 0.f && !a->noise_row) return SSV_ERR_INVALID;
  return SSV_OK;
}

// Parameter block over a workspace laid out by accept_layout.  Returns the
// effective mode: coupled noise at T = 0 is the plain argmax.
static int fill_params(const ssv_accept_args* a, char* w, const AccWorkspaceLayout& L, int nchunks,
                       AcceptParams* out) {
  AcceptParams& p = *out;
  p.mode = a->mode;
  p.T = a->T;
  p.c2 = a->T > 0.f ? (float)(1.4426950408889634 / (double)a->T) : 0.f;
  p.V = a->V;
  p.vec = ((a->V % 4) == 0 && ((uintptr_t)a->logits & 15u) == 0 && ((uintptr_t)a->draft_logits & 15u) == 0 &&
           ((uintptr_t)a->noise & 15u) == 0) ? 1 : 0;
  p.batch = a->batch;
  p.total_slots = a->total_slots;
  p.nchunks = nchunks;
  p.logits = a->logits;
  p.draft_logits = a->draft_logits;
  p.draft_tokens = a->draft_tokens;
  p.tau = a->tau;
  p.block = a->block;
  p.gamma = a->gamma;
  p.slot_off = a->slot_off;
  p.noise = a->noise;
  p.n_noise_rows = a->n_noise_rows;
  p.noise_row = a->noise_row;
  p.u_accept = a->u_accept;
  p.u_sample = a->u_sample;
  p.n_acc = a->n_acc;
  p.n_out = a->n_out;
  p.tokens = a->tokens;
  p.dev_status = a->dev_status;
  p.early = 0;
  p.cnt_seq = reinterpret_cast<int32_t*>(w + L.cnt_seq);
  p.cnt_sample = reinterpret_cast<int32_t*>(w + L.cnt_sample);
  p.cnt_row = reinterpret_cast<int32_t*>(w + L.cnt_row);
  p.emit = reinterpret_cast<int32_t*>(w + L.emit);
  p.part = reinterpret_cast<AccPartial*>(w + L.part);
  p.norm = reinterpret_cast<SlotNorm*>(w + L.norm);
  p.rowres = reinterpret_cast<RowResult*>(w + L.rowres);
  p.nsub = nchunks * (kAccChunk / kEmitSub);
  p.enorm = reinterpret_cast<float4*>(w + L.enorm);
  p.smass = reinterpret_cast<float4*>(w + L.smass);
  p.wmass = reinterpret_cast<float4*>(w + L.wmass);
  // double-float constants of the emitted sample: log2(e) / T and 2^(2^i / 256)
  const double c2d = a->T > 0.f ? 1.4426950408889634074 / (double)a->T : 0.0;
  p.c2_hi = (float)c2d;
  p.c2_lo = (float)(c2d - (double)p.c2_hi);
  for (int i = 0; i < 8; ++i) {
    const double v = exp2((double)(1 << i) / 256.0);
    p.e2pow[i].x = (float)v;
    p.e2pow[i].y = (float)(v - (double)(float)v);
  }
  const FaultSetting f = fault_for(SSV_FAULT_ACCEPT);
  p.wait_budget = f.budget;
  p.fault_skip = f.skip;
  p.noise_seed = a->noise_seed;
  int mode = a->mode;
  if ((mode == SSV_ACCEPT_GUMBEL || mode == SSV_ACCEPT_GUMBEL_GEN) && a->T == 0.f)
    mode = SSV_ACCEPT_ARGMAX;  // T = 0 ignores the noise
  p.mode = mode;
  return mode;
}

extern "C" ssv_status ssv_accept_workspace(const ssv_accept_args* a, size_t* bytes) {
  if (!bytes) return SSV_ERR_INVALID;
  int nchunks = 0;
  const ssv_status st = accept_check(a, &nchunks);
  if (st != SSV_OK) return st;
  *bytes = accept_layout(a->batch, a->total_slots, nchunks).total;
  return SSV_OK;
}

namespace ssv {

ssv_status accept_validate(const ssv_accept_args* a, void* ws, size_t ws_bytes) {
  int nchunks = 0;
  const ssv_status st = accept_check(a, &nchunks);
  if (st != SSV_OK) return st;
  if (a->batch == 0 || a->total_slots == 0) return SSV_OK;
  const AccWorkspaceLayout L = accept_layout(a->batch, a->total_slots, nchunks);
  if (!ws || ((uintptr_t)ws & 255u) || ws_bytes < L.total) return SSV_ERR_WORKSPACE;
  return SSV_OK;
}

ssv_status accept_run(const ssv_accept_args* a, void* ws, size_t ws_bytes, cudaStream_t s, int early) {
  const ssv_status st = accept_validate(a, ws, ws_bytes);
  if (st != SSV_OK) return st;
  if (a->batch == 0 || a->total_slots == 0) return SSV_OK;
  int nchunks = 0;
  accept_check(a, &nchunks);
  const AccWorkspaceLayout L = accept_layout(a->batch, a->total_slots, nchunks);
  AcceptParams p;
  const int mode = fill_params(a, static_cast<char*>(ws), L, nchunks, &p);
  p.early = early;
  const cudaError_t e = launch_accept(p, mode, a->logits_dtype == SSV_BF16, s);
  return e == cudaSuccess ? SSV_OK : SSV_ERR_CUDA;
}

}  // namespace ssv

extern "C" ssv_status ssv_accept(const ssv_accept_args* a, void* ws, size_t ws_bytes, void* stream) {
  return ssv::accept_run(a, ws, ws_bytes, static_cast<cudaStream_t>(stream), 0);
}

// ---------------------------------------------------------------------------
// ssv_accept_noalloc: ssv_accept with its scratch in a fixed device array.
//
// For callers that cannot allocate device memory themselves.  The scratch
// lives in one file-scope array per device (kNoAllocScratchBytes, reserved
// by every GPU that loads this library until the process exits).  Host code
// cannot use the array's name as a device address, so the first call in each
// CUDA context looks the address up with cudaGetSymbolAddress while that
// context is current and caches it per device, together with the context it
// belongs to: a call from another context on the same device (after
// cudaDeviceReset, or with a context the caller made current) looks it up
// again.  Every call shares the array: calls that overlap on the GPU (other
// streams, other host threads) race and must be serialised by the caller.
// The arrival counters are cleared with a memset at each call.
// ---------------------------------------------------------------------------
#include <cuda.h>
#include <mutex>

namespace {

constexpr size_t kNoAllocScratchBytes = size_t(4) << 20;  // 4 MiB
constexpr int kNoAllocMaxDevices = 64;

static __device__ __align__(256) unsigned char g_accept_scratch[kNoAllocScratchBytes];

struct ScratchEntry {
  CUcontext ctx;
  void* addr;
};

std::mutex g_scratch_mu;
ScratchEntry g_scratch[kNoAllocMaxDevices] = {};

using CtxGetCurrentFn = CUresult (*)(CUcontext*);

CtxGetCurrentFn ctx_get_current() {
  static CtxGetCurrentFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<CtxGetCurrentFn>(f);
  });
  return fn;
}

ssv_status noalloc_scratch_address(void** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return SSV_ERR_CUDA;
  if (dev >= kNoAllocMaxDevices) return SSV_ERR_INVALID;
  CUcontext ctx = nullptr;
  const CtxGetCurrentFn get = ctx_get_current();
  if (!get || get(&ctx) != CUDA_SUCCESS) return SSV_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  ScratchEntry& e = g_scratch[dev];
  if (!ctx || !e.addr || e.ctx != ctx) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_accept_scratch) != cudaSuccess || !p) return SSV_ERR_CUDA;
    // with no context current, the lookup above made the device's primary one current
    if (!ctx && (get(&ctx) != CUDA_SUCCESS || !ctx)) return SSV_ERR_CUDA;
    e.ctx = ctx;
    e.addr = p;
  }
  *out = e.addr;
  return SSV_OK;
}

}  // namespace

extern "C" ssv_status ssv_accept_noalloc(const ssv_accept_args* a, void* stream) {
  int nchunks = 0;
  ssv_status st = accept_check(a, &nchunks);
  if (st != SSV_OK) return st;
  if (a->batch == 0 || a->total_slots == 0) return SSV_OK;
  const AccWorkspaceLayout L = accept_layout(a->batch, a->total_slots, nchunks);
  if (L.total > kNoAllocScratchBytes) return SSV_ERR_WORKSPACE;
  void* scratch = nullptr;
  st = noalloc_scratch_address(&scratch);
  if (st != SSV_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // The arrival counters (cnt_seq, cnt_sample, cnt_row: the front of the
  // layout, up to emit) must start at zero.
  if (cudaMemsetAsync(scratch, 0, L.emit, s) != cudaSuccess) return SSV_ERR_CUDA;
  AcceptParams p;
  const int mode = fill_params(a, static_cast<char*>(scratch), L, nchunks, &p);
  const cudaError_t e = launch_accept(p, mode, a->logits_dtype == SSV_BF16, s);
  return e == cudaSuccess ? SSV_OK : SSV_ERR_CUDA;
}
