// ssv_accept: acceptance in temporal order with the longest accepted prefix.
//
// SimSD summary, section 4 "Acceptance": standard rejection sampling in the
// temporal order the draft induces; the longest accepted prefix is kept.
// SPOT review, section "How it is used": state equality (exact at T = 0) and
// the coupled-noise match argmax(l/T + G[position]) with a Gumbel table
// shared by drafter and target (Proposition 2).
//
// Two kernels, each finishing with a "last CTA of the sequence" step (a
// per-sequence arrival counter in the workspace, no spinning):
//   accept_reduce   grid = verified rows x vocab chunks.  One streaming pass
//                   over each needed logits row (plus noise or draft row):
//                   per chunk the (max, first argmax) of the decision score,
//                   or for rejection sampling the chunk max and the
//                   compensated sum of exp of l/T and of draft/T.  The last
//                   CTA of a sequence merges the chunks, walks the stages in
//                   tau order, writes n_acc / n_out / tokens and, for
//                   rejection sampling, which row to sample from.
//   accept_sample   (rejection sampling only) grid = vocab chunks x batch.
//                   Chunk masses of (p - q)_+ and of p for the emission
//                   row; the last CTA finds the chunk holding u' * Z and
//                   scans it in vocabulary order (fp64 prefix sums).
#include "ssv_internal.cuh"

#include <limits.h>
#include <math.h>

namespace ssv {

constexpr int kAccThreads = 256;
constexpr int kAccVec = 4;                                 // elements per vector access
constexpr int kAccIters = 8;                               // vector accesses per thread per stream
constexpr int kAccPerThread = kAccVec * kAccIters;         // 32
constexpr int kAccChunk = kAccThreads * kAccPerThread;     // 8192 vocab entries per CTA

struct AccPartial {
  float m_a, m_b;          // chunk max of the raw logits and of the draft logits  (reject)
  float sa_hi, sa_lo;      // compensated sum over the chunk of 2^((l - m_a) c2)   (reject)
  float sb_hi, sb_lo;      // same for the draft row                              (reject)
  float val;               // best decision score                                  (argmax / gumbel)
  int idx;                 // its first index
};

struct SlotNorm {  // p_v = 2^((l_v - m_a) c2) / s_a, q likewise
  float m_a, m_b;
  double s_a, s_b;
};

__device__ __forceinline__ float ex2f(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

struct AcceptParams {
  int mode;
  float T;
  float c2;                // log2(e) / T: rejection-sampling weights are 2^((l - max) * c2)
  int V;
  int vec;                 // rows allow 4-element vector accesses
  int batch;
  int total_slots;
  int nchunks;
  const void* logits;
  const void* draft_logits;
  const int32_t* draft_tokens;
  const int32_t* tau;
  const int32_t* block;
  const int32_t* gamma;
  const int32_t* slot_off;
  const float* noise;
  int n_noise_rows;
  const int32_t* noise_row;
  const float* u_accept;
  const float* u_sample;
  int32_t* n_acc;
  int32_t* n_out;
  int32_t* tokens;
  int32_t* dev_status;
  // workspace carve-up
  int32_t* cnt_reduce;  // [batch]
  int32_t* cnt_sample;  // [batch]
  int32_t* emit;        // [batch][2] : emission slot (or -1), 1 = residual / 0 = p
  AccPartial* part;     // [total_slots][nchunks]
  SlotNorm* norm;       // [total_slots]
  float* smass;         // [batch][nchunks][4] : residual mass (hi, lo), p mass (hi, lo)
};

struct AccWorkspaceLayout {
  size_t cnt_reduce, cnt_sample, emit, part, norm, smass, total;
};

static AccWorkspaceLayout accept_layout(int batch, int total_slots, int nchunks) {
  AccWorkspaceLayout L;
  size_t o = 0;
  L.cnt_reduce = o; o = align_up(o + sizeof(int32_t) * (size_t)batch, 256);
  L.cnt_sample = o; o = align_up(o + sizeof(int32_t) * (size_t)batch, 256);
  L.emit = o;       o = align_up(o + sizeof(int32_t) * 2 * (size_t)batch, 256);
  L.part = o;       o = align_up(o + sizeof(AccPartial) * (size_t)total_slots * nchunks, 256);
  L.norm = o;       o = align_up(o + sizeof(SlotNorm) * (size_t)total_slots, 256);
  L.smass = o;      o = align_up(o + sizeof(float) * 4 * (size_t)batch * nchunks, 256);
  L.total = o;
  return L;
}

template <typename T>
__device__ __forceinline__ float ld_logit(const void* base, size_t i) {
  return Elem<T>::to_f32(static_cast<const T*>(base)[i]);
}

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

__device__ __forceinline__ void kahan_add(float& s, float& c, float x) {
  const float y = x - c;
  const float t = s + y;
  c = (t - s) - y;
  s = t;
}

// (h1, l1) += (h2, l2) with an error-free transformation of the leading terms
__device__ __forceinline__ void two_sum_acc(float& h1, float& l1, float h2, float l2) {
  const float s = h1 + h2;
  const float bb = s - h1;
  const float err = (h1 - (s - bb)) + (h2 - bb);
  h1 = s;
  l1 = l1 + l2 + err;
}

// ---- block reductions (256 threads) ---------------------------------------
__device__ __forceinline__ void argmax_combine(float& v, int& i, float ov, int oi) {
  if (ov > v || (ov == v && oi < i)) { v = ov; i = oi; }
}

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

// Exclusive prefix sum over the block (thread order), fp64.
__device__ double block_exclusive_scan(double v) {
  __shared__ double sw[kAccThreads / 32];
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  double incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const double y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) sw[wid] = incl;
  __syncthreads();
  double before = 0.0;
  for (int w = 0; w < wid; ++w) before += sw[w];
  __syncthreads();
  return before + incl - v;
}

// ---- per-sequence validity, checked by warp 0 (all 32 lanes) -----------------
__device__ bool warp_seq_valid(const AcceptParams& p, int b) {
  const int B = p.block[b], g = p.gamma[b];
  bool ok = B >= 1 && B <= 64 && g >= 0 && g <= B && p.slot_off[b] + B <= p.total_slots;
  if (ok) ok = warp_tau_is_permutation(p.tau + p.slot_off[b], B);
  return ok;
}

// ---- finalize: merge chunks, walk stages, write outputs --------------------
template <int MODE, typename T>
__device__ void accept_finalize(const AcceptParams& p, int b) {
  __shared__ int s_slot[64];
  __shared__ int s_dec[64];
  __shared__ int s_ok[64];
  const int off = p.slot_off[b], B = p.block[b], g = p.gamma[b];
  const int need = min(g + 1, B);
  const int tid = threadIdx.x;
  if (tid < B) s_slot[p.tau[off + tid] - 1] = tid;
  __syncthreads();
  if (tid < need) {
    const int k = off + s_slot[tid];
    const AccPartial* pp = p.part + (size_t)k * p.nchunks;
    if (MODE != SSV_ACCEPT_REJECT) {
      float v = -INFINITY;
      int i = INT_MAX;
      for (int c = 0; c < p.nchunks; ++c) argmax_combine(v, i, __ldcg(&pp[c].val), __ldcg(&pp[c].idx));
      s_dec[tid] = i;
      s_ok[tid] = (tid < g) && (p.draft_tokens[k] == i);
    } else {
      const bool with_draft = tid < g;  // the draft row is read only for tested stages
      float ma = -INFINITY, mb = -INFINITY;
      for (int c = 0; c < p.nchunks; ++c) {
        ma = fmaxf(ma, __ldcg(&pp[c].m_a));
        if (with_draft) mb = fmaxf(mb, __ldcg(&pp[c].m_b));
      }
      const double c2 = (double)p.c2;
      double sa = 0.0, sb = 0.0;
      for (int c = 0; c < p.nchunks; ++c) {
        sa += ((double)__ldcg(&pp[c].sa_hi) + (double)__ldcg(&pp[c].sa_lo)) *
              exp2(((double)__ldcg(&pp[c].m_a) - (double)ma) * c2);
        if (with_draft)
          sb += ((double)__ldcg(&pp[c].sb_hi) + (double)__ldcg(&pp[c].sb_lo)) *
                exp2(((double)__ldcg(&pp[c].m_b) - (double)mb) * c2);
      }
      SlotNorm nm;
      nm.m_a = ma; nm.m_b = mb; nm.s_a = sa; nm.s_b = sb;
      p.norm[k] = nm;
      s_dec[tid] = -1;
      int ok = 0;
      if (with_draft) {
        const int d = p.draft_tokens[k];
        if (d >= 0 && d < p.V) {
          const double ld = ld_logit<T>(p.logits, (size_t)k * p.V + d);
          const double qd = ld_logit<T>(p.draft_logits, (size_t)k * p.V + d);
          // p(d)/q(d) = 2^(((l_d - M_a) - (q_d - M_b)) c2) * S_b / S_a
          const double ratio = exp2(((ld - (double)ma) - (qd - (double)mb)) * c2) * (sb / sa);
          ok = (double)p.u_accept[k] < ratio;
        } else {
          report(p.dev_status, SSV_ERR_INVALID);
        }
      }
      s_ok[tid] = ok;
    }
  }
  __syncthreads();
  if (tid == 0) {
    int n = 0;
    while (n < g && s_ok[n]) ++n;
    for (int i = 0; i < n; ++i) p.tokens[off + i] = p.draft_tokens[off + s_slot[i]];
    for (int i = n; i < B; ++i) p.tokens[off + i] = -1;
    int nout = n;
    int eslot = -1, ekind = 0;
    if (n + 1 <= B) {
      nout = n + 1;
      if (MODE != SSV_ACCEPT_REJECT) {
        p.tokens[off + n] = s_dec[n];
      } else {
        eslot = off + s_slot[n];
        ekind = (n + 1 <= g) ? 1 : 0;
      }
    }
    p.n_acc[b] = n;
    p.n_out[b] = nout;
    if (MODE == SSV_ACCEPT_REJECT) {
      p.emit[2 * b] = eslot;
      p.emit[2 * b + 1] = ekind;
    }
  }
}

template <int MODE, typename T>
__global__ void __launch_bounds__(kAccThreads)
accept_reduce_kernel(const AcceptParams p) {
  __shared__ int s_ok, s_last;
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
  if (tid == 0) {
    p.part[(size_t)slot * p.nchunks + chunk] = out;
    __threadfence();
    const int prev = atomicAdd(&p.cnt_reduce[b], 1);
    s_last = (prev == need * p.nchunks - 1);
  }
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  accept_finalize<MODE, T>(p, b);
  __syncthreads();
  if (tid == 0) p.cnt_reduce[b] = 0;
}

// ---- rejection sampling: emitted token ------------------------------------
// Weight of vocab entry e: p_e = exp(l_e / T - M_a) / S_a and, for a residual
// sample, (p_e - q_e)_+ with q likewise.  The same expression serves the chunk
// masses and the final in-chunk scan.
__device__ __forceinline__ void sample_weight(float c2, float nma, float nmb, float la, float lb, float inv_sa,
                                              float inv_sb, bool residual, float& wr, float& wp) {
  const float pv = ex2f(fmaf(la, c2, nma)) * inv_sa;
  const float qv = residual ? ex2f(fmaf(lb, c2, nmb)) * inv_sb : 0.f;
  wp = pv;
  wr = residual ? fmaxf(pv - qv, 0.f) : 0.f;
}

template <typename T>
__global__ void __launch_bounds__(kAccThreads)
accept_sample_kernel(const AcceptParams p) {
  __shared__ int s_ok, s_last;
  const int b = blockIdx.x / p.nchunks;
  const int chunk = blockIdx.x % p.nchunks;
  const int tid = threadIdx.x;
  // A sequence whose stage map or sizes were rejected never ran its finalize
  // step, so its emission record may be stale: skip it.
  if (tid < 32) {
    const bool ok = warp_seq_valid(p, b);
    if (tid == 0) s_ok = ok;
  }
  __syncthreads();
  if (!s_ok) return;
  const int eslot = p.emit[2 * b];
  const int soff = p.slot_off[b];
  const int nacc = p.n_acc[b];
  if (eslot < soff || eslot >= soff + p.block[b] || nacc < 0 || nacc >= p.block[b]) return;
  const bool residual = p.emit[2 * b + 1] != 0;
  const SlotNorm nm = p.norm[eslot];
  const float inv_sa = (float)(1.0 / nm.s_a);
  const float inv_sb = residual ? (float)(1.0 / nm.s_b) : 0.f;
  const float nma = -nm.m_a * p.c2, nmb = -nm.m_b * p.c2;
  const size_t rbase = (size_t)eslot * p.V;
  const int c0 = chunk * kAccChunk;
  const bool vec = p.vec != 0;
  float xa[kAccPerThread], xb[kAccPerThread];
  ld_chunk<T>(p.logits, rbase, c0, p.V, vec, -INFINITY, xa);
  if (residual) ld_chunk<T>(p.draft_logits, rbase, c0, p.V, vec, -INFINITY, xb);
  float wr[kAccPerThread], wp[kAccPerThread];
  float sr = 0.f, cr = 0.f, sp = 0.f, cp = 0.f;
#pragma unroll
  for (int j = 0; j < kAccPerThread; ++j) {
    sample_weight(p.c2, nma, nmb, xa[j], residual ? xb[j] : -INFINITY, inv_sa, inv_sb, residual, wr[j], wp[j]);
    kahan_add(sr, cr, wr[j]);
    kahan_add(sp, cp, wp[j]);
  }
  float lr = -cr, lp = -cp;
  block_sum2x2(sr, lr, sp, lp);
  if (tid == 0) {
    float* sm = p.smass + ((size_t)b * p.nchunks + chunk) * 4;
    sm[0] = sr; sm[1] = lr; sm[2] = sp; sm[3] = lp;
    __threadfence();
    const int prev = atomicAdd(&p.cnt_sample[b], 1);
    s_last = (prev == p.nchunks - 1);
  }
  __syncthreads();
  if (!s_last) return;
  __threadfence();

  // ---- last CTA of sequence b: locate u' * Z --------------------------------
  __shared__ int s_chunk;
  __shared__ double s_before, s_thresh;
  __shared__ int s_use_res;
  if (tid == 0) {
    const float* sm = p.smass + (size_t)b * p.nchunks * 4;
    double zr = 0.0, zp = 0.0;
    for (int c = 0; c < p.nchunks; ++c) {
      zr += (double)__ldcg(&sm[4 * c]) + (double)__ldcg(&sm[4 * c + 1]);
      zp += (double)__ldcg(&sm[4 * c + 2]) + (double)__ldcg(&sm[4 * c + 3]);
    }
    const int use_res = residual && zr > 0.0;
    const double Z = use_res ? zr : zp;
    const double t = (double)p.u_sample[b] * Z;
    double cum = 0.0, before = 0.0, before_last = 0.0;
    int cs = -1, last_nz = 0;
    for (int c = 0; c < p.nchunks; ++c) {
      const double m = use_res ? (double)__ldcg(&sm[4 * c]) + (double)__ldcg(&sm[4 * c + 1])
                               : (double)__ldcg(&sm[4 * c + 2]) + (double)__ldcg(&sm[4 * c + 3]);
      if (m > 0.0) { last_nz = c; before_last = cum; }
      if (cs < 0 && cum + m > t) { cs = c; before = cum; }
      cum += m;
    }
    if (cs < 0) { cs = last_nz; before = before_last; }
    s_chunk = cs; s_before = before; s_thresh = t; s_use_res = use_res;
  }
  __syncthreads();
  const int cs = s_chunk;
  const bool use_res = s_use_res != 0;
  // Weights of the crossing chunk in vocabulary order, through shared memory
  // (index i stored at i + i / 32 so that the contiguous runs read below are
  // free of bank conflicts).
  __shared__ float s_w[kAccChunk + kAccChunk / 32];
  {
    const int cc0 = cs * kAccChunk;
    if (cs != chunk) {
      ld_chunk<T>(p.logits, rbase, cc0, p.V, vec, -INFINITY, xa);
      if (residual) ld_chunk<T>(p.draft_logits, rbase, cc0, p.V, vec, -INFINITY, xb);
#pragma unroll
      for (int j = 0; j < kAccPerThread; ++j)
        sample_weight(p.c2, nma, nmb, xa[j], residual ? xb[j] : -INFINITY, inv_sa, inv_sb, residual, wr[j], wp[j]);
    }
#pragma unroll
    for (int j = 0; j < kAccPerThread; ++j) {
      const int li = chunk_index(0, j);  // index within the chunk
      s_w[li + li / 32] = (cc0 + li < p.V) ? (use_res ? wr[j] : wp[j]) : 0.f;
    }
  }
  __syncthreads();
  // each thread: a contiguous run of kAccPerThread entries
  const int r0 = tid * kAccPerThread;
  float local = 0.f;
  int last_pos = -1;
#pragma unroll
  for (int j = 0; j < kAccPerThread; ++j) {
    const float w = s_w[(r0 + j) + (r0 + j) / 32];
    local += w;
    if (w > 0.f) last_pos = cs * kAccChunk + r0 + j;
  }
  const double excl = block_exclusive_scan((double)local);
  __shared__ int s_pick, s_last_nz;
  if (tid == 0) { s_pick = INT_MAX; s_last_nz = -1; }
  __syncthreads();
  // remaining mass to cross inside this run, then an fp32 scan of the run
  const float rel = (float)(s_thresh - (s_before + excl));
  float acc = 0.f;
  int pick = INT_MAX;
#pragma unroll
  for (int j = 0; j < kAccPerThread; ++j) {
    const float w = s_w[(r0 + j) + (r0 + j) / 32];
    acc += w;
    if (pick == INT_MAX && w > 0.f && acc > rel) pick = cs * kAccChunk + r0 + j;
  }
  if (pick != INT_MAX) atomicMin(&s_pick, pick);
  if (last_pos >= 0) atomicMax(&s_last_nz, last_pos);
  __syncthreads();
  if (tid == 0) {
    int v = s_pick != INT_MAX ? s_pick : s_last_nz;
    if (v < 0) v = 0;
    p.tokens[soff + nacc] = v;
    p.cnt_sample[b] = 0;
  }
}

template <int MODE, typename T>
static cudaError_t launch_accept_t(const AcceptParams& p, cudaStream_t st) {
  const long long g1 = (long long)p.total_slots * p.nchunks;
  if (g1 > 0x7fffffffLL) return cudaErrorInvalidValue;
  accept_reduce_kernel<MODE, T><<<(unsigned)g1, kAccThreads, 0, st>>>(p);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  if (MODE == SSV_ACCEPT_REJECT) {
    const long long g2 = (long long)p.batch * p.nchunks;
    accept_sample_kernel<T><<<(unsigned)g2, kAccThreads, 0, st>>>(p);
    e = cudaGetLastError();
  }
  return e;
}

}  // namespace ssv

using namespace ssv;

static ssv_status accept_check(const ssv_accept_args* a, int* nchunks) {
  if (!a) return SSV_ERR_INVALID;
  if (a->mode != SSV_ACCEPT_ARGMAX && a->mode != SSV_ACCEPT_GUMBEL && a->mode != SSV_ACCEPT_REJECT)
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
  return SSV_OK;
}

extern "C" ssv_status ssv_accept_workspace(const ssv_accept_args* a, size_t* bytes) {
  if (!bytes) return SSV_ERR_INVALID;
  int nchunks = 0;
  const ssv_status st = accept_check(a, &nchunks);
  if (st != SSV_OK) return st;
  *bytes = accept_layout(a->batch, a->total_slots, nchunks).total;
  return SSV_OK;
}

extern "C" ssv_status ssv_accept(const ssv_accept_args* a, void* ws, size_t ws_bytes, void* stream) {
  int nchunks = 0;
  const ssv_status st = accept_check(a, &nchunks);
  if (st != SSV_OK) return st;
  if (a->batch == 0 || a->total_slots == 0) return SSV_OK;
  const AccWorkspaceLayout L = accept_layout(a->batch, a->total_slots, nchunks);
  if (!ws || ((uintptr_t)ws & 255u) || ws_bytes < L.total) return SSV_ERR_WORKSPACE;
  char* w = static_cast<char*>(ws);
  AcceptParams p;
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
  p.cnt_reduce = reinterpret_cast<int32_t*>(w + L.cnt_reduce);
  p.cnt_sample = reinterpret_cast<int32_t*>(w + L.cnt_sample);
  p.emit = reinterpret_cast<int32_t*>(w + L.emit);
  p.part = reinterpret_cast<AccPartial*>(w + L.part);
  p.norm = reinterpret_cast<SlotNorm*>(w + L.norm);
  p.smass = reinterpret_cast<float*>(w + L.smass);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const bool bf = a->logits_dtype == SSV_BF16;
  int mode = a->mode;
  if (mode == SSV_ACCEPT_GUMBEL && a->T == 0.f) mode = SSV_ACCEPT_ARGMAX;   // T = 0 ignores the noise
  cudaError_t e;
  switch (mode) {
    case SSV_ACCEPT_ARGMAX:
      e = bf ? launch_accept_t<SSV_ACCEPT_ARGMAX, __nv_bfloat16>(p, s) : launch_accept_t<SSV_ACCEPT_ARGMAX, float>(p, s);
      break;
    case SSV_ACCEPT_GUMBEL:
      e = bf ? launch_accept_t<SSV_ACCEPT_GUMBEL, __nv_bfloat16>(p, s) : launch_accept_t<SSV_ACCEPT_GUMBEL, float>(p, s);
      break;
    default:
      e = bf ? launch_accept_t<SSV_ACCEPT_REJECT, __nv_bfloat16>(p, s) : launch_accept_t<SSV_ACCEPT_REJECT, float>(p, s);
      break;
  }
  return e == cudaSuccess ? SSV_OK : SSV_ERR_CUDA;
}

// ---------------------------------------------------------------------------
// ssv_accept_noalloc: ssv_accept with its scratch in a fixed device array.
//
// For callers that cannot allocate device memory themselves.  The scratch
// lives in one file-scope array per device (kNoAllocScratchBytes, reserved
// by every GPU that loads this library until the process exits).  Host code
// cannot use the array's name as a device address, so the first call on each
// device looks the address up with cudaGetSymbolAddress while that device is
// current and caches it.  Every call shares the array: calls that overlap on
// the GPU (other streams, other host threads) race and must be serialised by
// the caller.  The arrival counters are cleared with a memset at each call.
// ---------------------------------------------------------------------------
#include <mutex>

namespace {

constexpr size_t kNoAllocScratchBytes = size_t(4) << 20;  // 4 MiB
constexpr int kNoAllocMaxDevices = 64;

static __device__ __align__(256) unsigned char g_accept_scratch[kNoAllocScratchBytes];

std::mutex g_scratch_mu;
void* g_scratch_addr[kNoAllocMaxDevices] = {};

ssv_status noalloc_scratch_address(void** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kNoAllocMaxDevices) return SSV_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (!g_scratch_addr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_accept_scratch) != cudaSuccess || !p) return SSV_ERR_CUDA;
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
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
  // The counters [cnt_reduce, cnt_sample] must start at zero.
  if (cudaMemsetAsync(scratch, 0, L.emit, s) != cudaSuccess) return SSV_ERR_CUDA;
  char* w = static_cast<char*>(scratch);
  AcceptParams p;
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
  p.cnt_reduce = reinterpret_cast<int32_t*>(w + L.cnt_reduce);
  p.cnt_sample = reinterpret_cast<int32_t*>(w + L.cnt_sample);
  p.emit = reinterpret_cast<int32_t*>(w + L.emit);
  p.part = reinterpret_cast<AccPartial*>(w + L.part);
  p.norm = reinterpret_cast<SlotNorm*>(w + L.norm);
  p.smass = reinterpret_cast<float*>(w + L.smass);
  const bool bf = a->logits_dtype == SSV_BF16;
  int mode = a->mode;
  if (mode == SSV_ACCEPT_GUMBEL && a->T == 0.f) mode = SSV_ACCEPT_ARGMAX;
  cudaError_t e;
  switch (mode) {
    case SSV_ACCEPT_ARGMAX:
      e = bf ? launch_accept_t<SSV_ACCEPT_ARGMAX, __nv_bfloat16>(p, s) : launch_accept_t<SSV_ACCEPT_ARGMAX, float>(p, s);
      break;
    case SSV_ACCEPT_GUMBEL:
      e = bf ? launch_accept_t<SSV_ACCEPT_GUMBEL, __nv_bfloat16>(p, s) : launch_accept_t<SSV_ACCEPT_GUMBEL, float>(p, s);
      break;
    default:
      e = bf ? launch_accept_t<SSV_ACCEPT_REJECT, __nv_bfloat16>(p, s) : launch_accept_t<SSV_ACCEPT_REJECT, float>(p, s);
      break;
  }
  return e == cudaSuccess ? SSV_OK : SSV_ERR_CUDA;
}
