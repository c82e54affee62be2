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

#include <algorithm>

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
//                      (unnormalised p and q); where the workspace holds
//                      room for them (eexp), also every entry's e_a and e_b
//                      and the p masses (sums of e_a) per warp and sub-chunk.
//   accept_sample      every CTA of sequence b adds the sub-chunk sums in the
//                      same fixed order (S_a, S_b), forms the weights
//                      w = (e_a S_b - e_b S_a)_+ (the residual (p - q)_+ scaled
//                      by S_a S_b) and e_a (p scaled by S_a) -- from the stored
//                      exponentials when there are any, the same values --
//                      and writes its masses per warp and per sub-chunk.
//   accept_locate      one CTA per sequence finds the sub-chunk, then the
//                      warp, then the entry where the cumulative mass passes
//                      u' Z (double-float prefix sums; the residual unless it
//                      vanished, then p).
// fp64 is avoided throughout: it is a narrow pipe on this part (tens of
// cycles per dependent operation).

struct EmitCtx {
  bool residual;
  float ma, mb;  // row maxima of the logits and the draft logits
  dfx c2;        // log2(e) / T
  dfx sa, sb;    // S_a, S_b (residual only)
};

// residual weight (e_a S_b - e_b S_a)_+ of one entry
__device__ __forceinline__ dfx residual_weight(const EmitCtx& c, dfx ea, dfx eb) {
  const dfx d = dfx_add(dfx_mul(ea, c.sb), dfx_mul(dfx{-eb.hi, -eb.lo}, c.sa));
  return d.hi > 0.f ? d : dfx{0.f, 0.f};
}

// residual weight and p weight e_a of one entry, from its two logits
__device__ __forceinline__ void emit_weights(const EmitCtx& c, float la, float lb, const float2* tab, dfx& wr,
                                             dfx& wp) {
  const dfx ea = dfx_exp2_diff(la, c.ma, c.c2, tab);
  wp = ea;
  wr = dfx{0.f, 0.f};
  if (c.residual) wr = residual_weight(c, ea, dfx_exp2_diff(lb, c.mb, c.c2, tab));
}

__device__ __forceinline__ dfx shfl_xor_dfx(dfx a, int o) {
  return dfx{__shfl_xor_sync(0xffffffffu, a.hi, o), __shfl_xor_sync(0xffffffffu, a.lo, o)};
}
__device__ __forceinline__ dfx shfl_up_dfx(dfx a, int o) {
  return dfx{__shfl_up_sync(0xffffffffu, a.hi, o), __shfl_up_sync(0xffffffffu, a.lo, o)};
}
__device__ __forceinline__ dfx shfl_dfx(dfx a, int src) {
  return dfx{__shfl_sync(0xffffffffu, a.hi, src), __shfl_sync(0xffffffffu, a.lo, src)};
}
__device__ __forceinline__ dfx dfx_neg(dfx a) { return dfx{-a.hi, -a.lo}; }
// a > b, decided on the sign of the renormalised difference
__device__ __forceinline__ bool dfx_gt(dfx a, dfx b) { return dfx_add(a, dfx_neg(b)).hi > 0.f; }
// inclusive prefix sum over the lanes (Hillis-Steele, 5 double-float additions deep)
__device__ __forceinline__ dfx warp_incl_scan(dfx x, int lane) {
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const dfx y = shfl_up_dfx(x, o);
    if (lane >= o) x = dfx_add(x, y);
  }
  return x;
}

// exclusive prefix from the inclusive one (every lane takes part in the shuffle)
__device__ __forceinline__ dfx warp_excl_of(dfx incl, int lane) {
  const dfx y = shfl_up_dfx(incl, 1);
  return lane ? y : dfx{0.f, 0.f};
}

constexpr int kEmitLane = 4;  // sub-chunk masses per lane in the level-1 search

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

// The normaliser pass takes its work as items (sequence, sub-chunk) of the
// sequences that sample the residual this call, dealt round-robin over a
// grid sized to be resident at once, so that no SM idles on a sequence
// without work.  The emission records are authoritative: the pass before the
// walks set every sequence's record to "none" (emit[2b] = -1), and the walk
// of each valid sequence wrote its own.
constexpr int kEmitList = 2048;  // sequences listed per round (8 KB of shared memory)

// The emitting sequences among b in [b0, b0 + kEmitList), in increasing b,
// into s_seq (emission slot | residual << 31 in s_rec); returns their count.
// Called by every thread of the CTA (barriers inside).
__device__ int emit_list(const AcceptParams& p, int b0, bool residual_only, int* s_seq, int* s_rec, int* s_wc) {
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  int total = 0;
  const int end = min(p.batch, b0 + kEmitList);
  for (int base = b0; base < end; base += kAccThreads) {
    const int b = base + tid;
    int es = -1, res = 0;
    if (b < end) {
      es = __ldcg(p.emit + 2 * b);
      res = __ldcg(p.emit + 2 * b + 1);
    }
    const bool v = es >= 0 && es < p.total_slots && (!residual_only || res != 0);
    const unsigned bal = __ballot_sync(0xffffffffu, v);
    if (lane == 0) s_wc[wid] = __popc(bal);
    __syncthreads();
    int before = total, sum = 0;
#pragma unroll
    for (int w = 0; w < kAccThreads / 32; ++w) {
      const int c = s_wc[w];
      before += (w < wid) ? c : 0;
      sum += c;
    }
    if (v) {
      const int pos = before + __popc(bal & ((1u << lane) - 1u));
      s_seq[pos] = b;
      s_rec[pos] = (int)((unsigned)es | ((res != 0 ? 1u : 0u) << 31));
    }
    total += sum;
    __syncthreads();
  }
  return total;
}

// The 2^(j/256) table into shared memory (inputs only, before the wait),
// then the wait for the walks' emission records, accepted lengths and row
// maxima (normaliser pass).
__device__ __forceinline__ void emit_prologue(const AcceptParams& p, float2* s_tab) {
  dfx_exp2_table(p.e2pow, s_tab, threadIdx.x);  // kAccThreads == 256 entries
  __syncthreads();
  pdl_wait();
  pdl_trigger();
}

static_assert(kAccThreads == 256 && kEmitSub == 8 * kAccThreads, "one table entry and 8 row entries per thread");

template <typename T>
__global__ void __launch_bounds__(kAccThreads)
accept_emit_norm_kernel(const AcceptParams p) {
  __shared__ float2 s_tab[256];
  __shared__ float4 s_w[kAccThreads / 32];
  __shared__ int s_seq[kEmitList], s_rec[kEmitList], s_wc[kAccThreads / 32];
  emit_prologue(p, s_tab);
  const dfx c2{p.c2_hi, p.c2_lo};
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  long long it0 = 0;  // items of earlier rounds
  for (int b0 = 0; b0 < p.batch; b0 += kEmitList) {
    const int n = emit_list(p, b0, true, s_seq, s_rec, s_wc);
    const long long items = (long long)n * p.nsub;
    // this CTA's items of the round: global item indices congruent to blockIdx.x
    long long first = ((long long)blockIdx.x - it0 % gridDim.x + gridDim.x) % gridDim.x;
    for (long long it = first; it < items; it += gridDim.x) {
      const int b = s_seq[it / p.nsub];
      const int sub = (int)(it % p.nsub);
      const int eslot = s_rec[it / p.nsub] & 0x7fffffff;
      const SlotNorm nm = p.norm[eslot];
      const size_t rbase = (size_t)eslot * p.V;
      const int e0 = sub * kEmitSub + threadIdx.x * 8;
      float xa[8], xb[8];
      ld_run8<T>(p.logits, rbase, e0, p.V, p.vec != 0, xa);
      ld_run8<T>(p.draft_logits, rbase, e0, p.V, p.vec != 0, xb);
      const size_t cta = (size_t)b * p.nsub + sub;
      float4* ex = p.eexp ? p.eexp + cta * kEmitSub + threadIdx.x : nullptr;
      dfx sa{0.f, 0.f}, sb{0.f, 0.f};
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const dfx ea = dfx_exp2_diff(xa[j], nm.m_a, c2, s_tab);
        const dfx eb = dfx_exp2_diff(xb[j], nm.m_b, c2, s_tab);
        if (ex) __stcg(ex + j * kAccThreads, make_float4(ea.hi, ea.lo, eb.hi, eb.lo));
        sa = dfx_add(sa, ea);
        sb = dfx_add(sb, eb);
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        sa = dfx_add(sa, shfl_xor_dfx(sa, o));
        sb = dfx_add(sb, shfl_xor_dfx(sb, o));
      }
      // With the exponentials stored, the p masses (the fallback when the
      // residual vanishes) are these sums of e_a, in the sampling pass's order.
      if (lane == 0) {
        s_w[wid] = make_float4(sa.hi, sa.lo, sb.hi, sb.lo);
        if (ex) __stcg(reinterpret_cast<float2*>(p.wmass + cta * 8 + wid) + 1, make_float2(sa.hi, sa.lo));
      }
      __syncthreads();
      if (threadIdx.x == 0) {
        for (int w = 1; w < kAccThreads / 32; ++w) {
          sa = dfx_add(sa, dfx{s_w[w].x, s_w[w].y});
          sb = dfx_add(sb, dfx{s_w[w].z, s_w[w].w});
        }
        p.enorm[cta] = make_float4(sa.hi, sa.lo, sb.hi, sb.lo);
        if (ex) __stcg(reinterpret_cast<float2*>(p.smass + cta) + 1, make_float2(sa.hi, sa.lo));
      }
      __syncthreads();  // s_w is reused by the next item
    }
    it0 += items;
  }
}

// S_a, S_b of sequence b from its sub-chunk sums (one warp): kEmitLane
// consecutive sums per lane (one round of loads for nsub <= 128), then a
// butterfly.  The same fixed order wherever it is formed (the sampling CTAs
// and the locating CTA must agree to the last bit).
__device__ __forceinline__ float4 warp_emit_norms(const AcceptParams& p, int b) {
  const int lane = threadIdx.x & 31;
  const float4* en = p.enorm + (size_t)b * p.nsub;
  dfx a{0.f, 0.f}, bb{0.f, 0.f};
  for (int k0 = 0; k0 < p.nsub; k0 += 32 * kEmitLane) {
    float4 v[kEmitLane];
#pragma unroll
    for (int k = 0; k < kEmitLane; ++k) {
      const int i = k0 + lane * kEmitLane + k;
      v[k] = i < p.nsub ? __ldcg(en + i) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll
    for (int k = 0; k < kEmitLane; ++k) {
      a = dfx_add(a, dfx{v[k].x, v[k].y});
      bb = dfx_add(bb, dfx{v[k].z, v[k].w});
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    a = dfx_add(a, shfl_xor_dfx(a, o));
    bb = dfx_add(bb, shfl_xor_dfx(bb, o));
  }
  return make_float4(a.hi, a.lo, bb.hi, bb.lo);
}

// Emission context of sequence b from its records, or false when it emits
// nothing this call.
__device__ __forceinline__ bool emit_ctx(const AcceptParams& p, int b, int& eslot, EmitCtx& c) {
  eslot = __ldcg(p.emit + 2 * b);
  if (eslot < 0 || eslot >= p.total_slots) return false;
  c.residual = __ldcg(p.emit + 2 * b + 1) != 0;
  const float2 nm = __ldcg(reinterpret_cast<const float2*>(p.norm + eslot));  // m_a, m_b
  c.ma = nm.x;
  c.mb = nm.y;
  c.c2 = dfx{p.c2_hi, p.c2_lo};
  c.sa = c.sb = dfx{0.f, 0.f};
  return true;
}

// Sampling pass: one CTA per (sequence, sub-chunk); the masses of the
// sampled weights per warp and per sub-chunk.
template <typename T>
__global__ void __launch_bounds__(kAccThreads)
accept_sample_kernel(const AcceptParams p) {
  __shared__ float2 s_tab[256];
  __shared__ float4 s_w[kAccThreads / 32];
  __shared__ float4 s_S;
  const int b = blockIdx.x / p.nsub;
  const int sub = blockIdx.x % p.nsub;
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  // Before the wait: the emission record and row maxima (the row merges
  // wrote them, and they completed before the normaliser pass let this
  // kernel start) and the exponential table.
  int eslot;
  EmitCtx c;
  if (!emit_ctx(p, b, eslot, c)) return;
  dfx_exp2_table(p.e2pow, s_tab, tid);  // kAccThreads == 256 entries
  __syncthreads();
  pdl_wait();  // the normalisers and stored exponentials
  pdl_trigger();
  if (c.residual) {
    if (wid == 0) {
      const float4 S = warp_emit_norms(p, b);
      if (lane == 0) s_S = S;
    }
    __syncthreads();
    c.sa = dfx{s_S.x, s_S.y};
    c.sb = dfx{s_S.z, s_S.w};
  }
  const size_t rbase = (size_t)eslot * p.V;
  const bool vec = p.vec != 0;
  // stored exponentials of the residual's row (the normaliser pass wrote them
  // and this sub-chunk's p masses): only the residual weights are formed here
  const bool stored = c.residual && p.eexp != nullptr;
  {
    const size_t cta = (size_t)b * p.nsub + sub;
    dfx mr{0.f, 0.f}, mp{0.f, 0.f};
    if (stored) {
      const float4* ex = p.eexp + cta * kEmitSub + tid;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const float4 v = __ldcg(ex + j * kAccThreads);
        mr = dfx_add(mr, residual_weight(c, dfx{v.x, v.y}, dfx{v.z, v.w}));
      }
    } else {
      const int e0 = sub * kEmitSub + tid * 8;
      float xa[8], xb[8];
      ld_run8<T>(p.logits, rbase, e0, p.V, vec, xa);
      if (c.residual) ld_run8<T>(p.draft_logits, rbase, e0, p.V, vec, xb);
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        dfx wr, wp;
        emit_weights(c, xa[j], c.residual ? xb[j] : -INFINITY, s_tab, wr, wp);
        mr = dfx_add(mr, wr);
        mp = dfx_add(mp, wp);
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      mr = dfx_add(mr, shfl_xor_dfx(mr, o));
      if (!stored) mp = dfx_add(mp, shfl_xor_dfx(mp, o));
    }
    if (lane == 0) {
      const float4 m4 = make_float4(mr.hi, mr.lo, mp.hi, mp.lo);
      s_w[wid] = m4;
      if (stored) __stcg(reinterpret_cast<float2*>(p.wmass + cta * 8 + wid), make_float2(mr.hi, mr.lo));
      else p.wmass[cta * 8 + wid] = m4;
    }
    __syncthreads();
    if (tid == 0) {
      for (int w = 1; w < kAccThreads / 32; ++w) {
        mr = dfx_add(mr, dfx{s_w[w].x, s_w[w].y});
        if (!stored) mp = dfx_add(mp, dfx{s_w[w].z, s_w[w].w});
      }
      if (stored) __stcg(reinterpret_cast<float2*>(p.smass + cta), make_float2(mr.hi, mr.lo));
      else p.smass[cta] = make_float4(mr.hi, mr.lo, mp.hi, mp.lo);
    }
  }
}

// Locating pass: one CTA per sequence, once every mass is written: the
// token where the cumulative mass passes t = u' Z.
template <typename T>
__global__ void __launch_bounds__(kAccThreads)
accept_locate_kernel(const AcceptParams p) {
  __shared__ float2 s_tab[256];
  __shared__ int s_cs, s_use_res, s_wsel;
  __shared__ float4 s_S;
  __shared__ float2 s_t, s_before;
  const int b = blockIdx.x;
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  // Before the wait: everything but the masses -- the emission record, row
  // maxima, normalisers and stored exponentials were complete before the
  // sampling pass let this kernel start -- and the exponential table.
  int eslot;
  EmitCtx c;
  if (!emit_ctx(p, b, eslot, c)) return;
  const size_t rbase = (size_t)eslot * p.V;
  const bool vec = p.vec != 0;
  const bool stored = c.residual && p.eexp != nullptr;
  if (wid == 1 && c.residual) {  // the normalisers (residual weights of level 3)
    const float4 S = warp_emit_norms(p, b);
    if (lane == 0) s_S = S;
  }
  dfx_exp2_table(p.e2pow, s_tab, tid);  // kAccThreads == 256 entries
  __syncthreads();
  pdl_wait();  // the masses
  pdl_trigger();
  // Level 1 (warp 0): the sub-chunk masses, kEmitLane consecutive per lane
  // in registers (one round of loads for nsub <= 128), the total Z and
  // t = u' Z, then the first sub-chunk whose cumulative mass passes t (else,
  // rounding having left t at the very end, the last non-empty one).  All
  // in double-float arithmetic.
  const float4* sm = p.smass + (size_t)b * p.nsub;
  if (wid == 0) {
    constexpr int kBlk = 32 * kEmitLane;
    const int nblk = (p.nsub + kBlk - 1) / kBlk;
    float4 v[kEmitLane];
    auto load_blk = [&](int blk) {
#pragma unroll
      for (int k = 0; k < kEmitLane; ++k) {
        const int i = blk * kBlk + lane * kEmitLane + k;
        v[k] = (i < p.nsub) ? __ldcg(sm + i) : make_float4(0.f, 0.f, 0.f, 0.f);
      }
    };
    dfx zr{0.f, 0.f}, zp{0.f, 0.f};
    for (int blk = 0; blk < nblk; ++blk) {
      load_blk(blk);
#pragma unroll
      for (int k = 0; k < kEmitLane; ++k) {
        zr = dfx_add(zr, dfx{v[k].x, v[k].y});
        zp = dfx_add(zp, dfx{v[k].z, v[k].w});
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      zr = dfx_add(zr, shfl_xor_dfx(zr, o));
      zp = dfx_add(zp, shfl_xor_dfx(zp, o));
    }
    const bool use_res = c.residual && zr.hi > 0.f;  // (p - q)_+ vanished: sample p
    const dfx t = dfx_mul(use_res ? zr : zp, dfx{p.u_sample[b], 0.f});
    dfx base{0.f, 0.f}, before{0.f, 0.f}, before_last{0.f, 0.f};
    int cs = -1, last_nz = 0;
    for (int blk = 0; blk < nblk; ++blk) {
      if (nblk > 1) load_blk(blk);  // a single block is still in registers
      dfx pre[kEmitLane];  // this lane's inclusive prefix over its sub-chunks
      dfx run{0.f, 0.f};
#pragma unroll
      for (int k = 0; k < kEmitLane; ++k) {
        run = dfx_add(run, use_res ? dfx{v[k].x, v[k].y} : dfx{v[k].z, v[k].w});
        pre[k] = run;
      }
      const dfx incl = warp_incl_scan(run, lane);
      const dfx start = dfx_add(base, warp_excl_of(incl, lane));  // before this lane's first
      int kc = -1, kz = -1;
#pragma unroll
      for (int k = 0; k < kEmitLane; ++k) {
        const int i = blk * kBlk + lane * kEmitLane + k;
        const bool nonzero = (use_res ? v[k].x : v[k].z) > 0.f;
        if (i < p.nsub && nonzero) kz = k;
        if (kc < 0 && i < p.nsub && dfx_gt(dfx_add(start, pre[k]), t)) kc = k;
      }
      const unsigned cross = __ballot_sync(0xffffffffu, kc >= 0);
      const unsigned nz = __ballot_sync(0xffffffffu, kz >= 0);
      // cumulative mass before sub-chunk k of this lane
      auto before_k = [&](int k) {
        dfx r = start;
#pragma unroll
        for (int j = 1; j < kEmitLane; ++j)
          if (j == k) r = dfx_add(start, pre[j - 1]);
        return r;
      };
      if (cs < 0 && cross) {
        const int f = __ffs(cross) - 1;
        const dfx bk = before_k(kc);
        cs = __shfl_sync(0xffffffffu, blk * kBlk + lane * kEmitLane + kc, f);
        before = shfl_dfx(bk, f);
      }
      if (nz) {
        const int l = 31 - __clz(nz);
        const dfx bk = before_k(kz);
        last_nz = __shfl_sync(0xffffffffu, blk * kBlk + lane * kEmitLane + kz, l);
        before_last = shfl_dfx(bk, l);
      }
      base = dfx_add(base, shfl_dfx(incl, 31));
    }
    if (cs < 0) { cs = last_nz; before = before_last; }
    if (lane == 0) {
      s_cs = cs;
      s_use_res = use_res;
      s_t = make_float2(t.hi, t.lo);
      s_before = make_float2(before.hi, before.lo);
    }
  }
  __syncthreads();
  const int cs = s_cs;
  const bool use_res = s_use_res;
  const dfx t{s_t.x, s_t.y};
  if (c.residual) {
    c.sa = dfx{s_S.x, s_S.y};
    c.sb = dfx{s_S.z, s_S.w};
  }
  // Every warp forms the weights of its 256 entries of sub-chunk cs (lane:
  // 8 consecutive entries) while warp 0 finds the warp that holds t (level
  // 2, from the sub-chunk's 8 warp masses).
  const int e0 = cs * kEmitSub + wid * 256 + lane * 8;
  float4 wm = make_float4(0.f, 0.f, 0.f, 0.f);
  if (wid == 0 && lane < 8) wm = __ldcg(p.wmass + ((size_t)b * p.nsub + cs) * 8 + lane);
  dfx w8[8];
  if (stored) {  // entry e0 + k is [k][32 wid + lane] of sub-chunk cs
    const float4* ex = p.eexp + ((size_t)b * p.nsub + cs) * kEmitSub + wid * 32 + lane;
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const float4 v = __ldcg(ex + k * kAccThreads);
      const dfx ea{v.x, v.y};
      w8[k] = use_res ? residual_weight(c, ea, dfx{v.z, v.w}) : ea;
    }
  } else {
    float ya[8], yb[8];
    ld_run8<T>(p.logits, rbase, e0, p.V, vec, ya);
    if (c.residual) ld_run8<T>(p.draft_logits, rbase, e0, p.V, vec, yb);
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      dfx wr, wp;
      emit_weights(c, ya[k], c.residual ? yb[k] : -INFINITY, s_tab, wr, wp);
      w8[k] = use_res ? wr : wp;
    }
  }
  if (wid == 0) {
    const dfx m = use_res ? dfx{wm.x, wm.y} : dfx{wm.z, wm.w};  // zero past lane 7
    const dfx incl = warp_incl_scan(m, lane);
    const dfx before{s_before.x, s_before.y};
    const unsigned cross = __ballot_sync(0xffffffffu, lane < 8 && dfx_gt(dfx_add(before, incl), t));
    const unsigned nz = __ballot_sync(0xffffffffu, lane < 8 && m.hi > 0.f);
    const int wsel = cross ? __ffs(cross) - 1 : (nz ? 31 - __clz(nz) : 7);
    const dfx b2 = dfx_add(before, shfl_dfx(warp_excl_of(incl, lane), wsel));
    if (lane == 0) {
      s_wsel = wsel;
      s_before = make_float2(b2.hi, b2.lo);
    }
  }
  __syncthreads();
  if (wid == s_wsel) {
    // Level 3 (warp wsel): the entry where the cumulative mass passes t
    dfx run{0.f, 0.f};
    int last_pos = -1;
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      run = dfx_add(run, w8[k]);
      if (w8[k].hi > 0.f) last_pos = e0 + k;
    }
    const dfx incl = warp_incl_scan(run, lane);
    // mass still to cross at the start of this lane's run
    const dfx rel = dfx_add(t, dfx_neg(dfx_add(dfx{s_before.x, s_before.y}, warp_excl_of(incl, lane))));
    dfx acc{0.f, 0.f};
    int pick = INT_MAX;
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      acc = dfx_add(acc, w8[k]);
      if (pick == INT_MAX && w8[k].hi > 0.f && dfx_gt(acc, rel)) pick = e0 + k;
    }
    // lanes are in vocabulary order: the first lane with a crossing holds the token
    const unsigned has = __ballot_sync(0xffffffffu, pick != INT_MAX);
    const int v_pick = has ? __shfl_sync(0xffffffffu, pick, __ffs(has) - 1) : INT_MAX;
    const unsigned anyw = __ballot_sync(0xffffffffu, last_pos >= 0);
    const int v_last = anyw ? __shfl_sync(0xffffffffu, last_pos, 31 - __clz(anyw)) : -1;
    if (lane == 0) {
      int v = v_pick != INT_MAX ? v_pick : v_last;
      if (v < 0) v = 0;
      p.tokens[p.slot_off[b] + p.n_acc[b]] = v;
    }
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
    // every emission record to "none" (-1); the walks write the valid sequences' own
    if (mode == SSV_ACCEPT_REJECT && cudaMemsetAsync(p.emit, 0xff, sizeof(int32_t) * 2 * (size_t)p.batch, st) != cudaSuccess)
      return cudaGetLastError();
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
  // emission passes: the normalisers over a grid that is resident at once
  // (five CTAs per SM beside the row merges still running), its items dealt
  // round-robin; the masses, one CTA per (sequence, sub-chunk); the token,
  // one CTA per sequence
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return cudaErrorInvalidDevice;
  const long long items = (long long)p.batch * p.nsub;
  if (items > 0x7fffffffLL) return cudaErrorInvalidValue;
  const unsigned g_norm = (unsigned)std::min<long long>(items, 5LL * sms);
  if (bf) {
    e = launch_pdl(accept_emit_norm_kernel<__nv_bfloat16>, dim3(g_norm), dim3(kAccThreads), 0, st, p);
    if (e == cudaSuccess)
      e = launch_pdl(accept_sample_kernel<__nv_bfloat16>, dim3((unsigned)items), dim3(kAccThreads), 0, st, p);
    if (e == cudaSuccess)
      e = launch_pdl(accept_locate_kernel<__nv_bfloat16>, dim3((unsigned)p.batch), dim3(kAccThreads), 0, st, p);
    return e;
  }
  e = launch_pdl(accept_emit_norm_kernel<float>, dim3(g_norm), dim3(kAccThreads), 0, st, p);
  if (e == cudaSuccess) e = launch_pdl(accept_sample_kernel<float>, dim3((unsigned)items), dim3(kAccThreads), 0, st, p);
  if (e == cudaSuccess) e = launch_pdl(accept_locate_kernel<float>, dim3((unsigned)p.batch), dim3(kAccThreads), 0, st, p);
  return e;
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
  p.unit_ctr = reinterpret_cast<int32_t*>(w + L.unit_ctr);
  p.cnt_seq = reinterpret_cast<int32_t*>(w + L.cnt_seq);
  p.cnt_row = reinterpret_cast<int32_t*>(w + L.cnt_row);
  p.emit = reinterpret_cast<int32_t*>(w + L.emit);
  p.part = reinterpret_cast<AccPartial*>(w + L.part);
  p.norm = reinterpret_cast<SlotNorm*>(w + L.norm);
  p.rowres = reinterpret_cast<RowResult*>(w + L.rowres);
  p.nsub = nchunks * (kAccChunk / kEmitSub);
  p.enorm = reinterpret_cast<float4*>(w + L.enorm);
  p.smass = reinterpret_cast<float4*>(w + L.smass);
  p.wmass = reinterpret_cast<float4*>(w + L.wmass);
  p.eexp = L.total > L.eexp ? reinterpret_cast<float4*>(w + L.eexp) : nullptr;
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
  *bytes = accept_layout(a->batch, a->total_slots, nchunks, a->mode == SSV_ACCEPT_REJECT).total;
  return SSV_OK;
}

namespace ssv {

ssv_status accept_validate(const ssv_accept_args* a, void* ws, size_t ws_bytes) {
  int nchunks = 0;
  const ssv_status st = accept_check(a, &nchunks);
  if (st != SSV_OK) return st;
  if (a->batch == 0 || a->total_slots == 0) return SSV_OK;
  const AccWorkspaceLayout L = accept_layout(a->batch, a->total_slots, nchunks, a->mode == SSV_ACCEPT_REJECT);
  if (!ws || ((uintptr_t)ws & 255u) || ws_bytes < L.total) return SSV_ERR_WORKSPACE;
  return SSV_OK;
}

ssv_status accept_run(const ssv_accept_args* a, void* ws, size_t ws_bytes, cudaStream_t s, int early) {
  const ssv_status st = accept_validate(a, ws, ws_bytes);
  if (st != SSV_OK) return st;
  if (a->batch == 0 || a->total_slots == 0) return SSV_OK;
  int nchunks = 0;
  accept_check(a, &nchunks);
  const AccWorkspaceLayout L = accept_layout(a->batch, a->total_slots, nchunks, a->mode == SSV_ACCEPT_REJECT);
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
  // rejection sampling stores the emitted rows' exponentials where they fit,
  // else its sampling pass forms them again
  AccWorkspaceLayout L = accept_layout(a->batch, a->total_slots, nchunks, a->mode == SSV_ACCEPT_REJECT);
  if (L.total > kNoAllocScratchBytes) L = accept_layout(a->batch, a->total_slots, nchunks, false);
  if (L.total > kNoAllocScratchBytes) return SSV_ERR_WORKSPACE;
  void* scratch = nullptr;
  st = noalloc_scratch_address(&scratch);
  if (st != SSV_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // The arrival counters (unit_ctr, cnt_seq, cnt_row: the front of the
  // layout, up to emit) must start at zero.
  if (cudaMemsetAsync(scratch, 0, L.emit, s) != cudaSuccess) return SSV_ERR_CUDA;
  AcceptParams p;
  const int mode = fill_params(a, static_cast<char*>(scratch), L, nchunks, &p);
  const cudaError_t e = launch_accept(p, mode, a->logits_dtype == SSV_BF16, s);
  return e == cudaSuccess ? SSV_OK : SSV_ERR_CUDA;
}
