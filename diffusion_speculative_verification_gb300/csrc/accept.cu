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
constexpr int kAccPerThread = 16;
constexpr int kAccChunk = kAccThreads * kAccPerThread;  // 4096 vocab entries per CTA

struct AccPartial {
  float m_a, m_b;    // chunk max of l/T and of draft/T          (reject)
  double s_a, s_b;   // sum over the chunk of exp(x - chunk max)  (reject)
  float val;         // best decision score                       (argmax / gumbel)
  int idx;           // its first index
};

struct SlotNorm {
  float m_a, m_b;
  double s_a, s_b;
};

struct AcceptParams {
  int mode;
  float T;
  int V;
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
  double* smass;        // [batch][nchunks][2] : residual mass, p mass
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
  L.smass = o;      o = align_up(o + sizeof(double) * 2 * (size_t)batch * nchunks, 256);
  L.total = o;
  return L;
}

template <typename T>
__device__ __forceinline__ float ld_logit(const void* base, size_t i) {
  return Elem<T>::to_f32(static_cast<const T*>(base)[i]);
}

__device__ __forceinline__ void kahan_add(float& s, float& c, float x) {
  const float y = x - c;
  const float t = s + y;
  c = (t - s) - y;
  s = t;
}

// ---- block reductions (256 threads) ---------------------------------------
__device__ __forceinline__ void argmax_combine(float& v, int& i, float ov, int oi) {
  if (ov > v || (ov == v && oi < i)) { v = ov; i = oi; }
}

__device__ void block_argmax(float& v, int& i) {
  __shared__ float sv[kAccThreads / 32];
  __shared__ int si[kAccThreads / 32];
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1)
    argmax_combine(v, i, __shfl_xor_sync(0xffffffffu, v, o), __shfl_xor_sync(0xffffffffu, i, o));
  if (lane == 0) { sv[wid] = v; si[wid] = i; }
  __syncthreads();
  if (wid == 0) {
    v = lane < kAccThreads / 32 ? sv[lane] : -INFINITY;
    i = lane < kAccThreads / 32 ? si[lane] : INT_MAX;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
      argmax_combine(v, i, __shfl_xor_sync(0xffffffffu, v, o), __shfl_xor_sync(0xffffffffu, i, o));
  }
  __syncthreads();
}

__device__ float block_max(float v) {
  __shared__ float sv[kAccThreads / 32];
  __shared__ float res;
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  if (lane == 0) sv[wid] = v;
  __syncthreads();
  if (threadIdx.x == 0) {
    float m = sv[0];
    for (int w = 1; w < kAccThreads / 32; ++w) m = fmaxf(m, sv[w]);
    res = m;
  }
  __syncthreads();
  const float r = res;
  __syncthreads();
  return r;
}

// Sum in a fixed order (lane tree, then warps in order): deterministic.
__device__ double block_sum(double v) {
  __shared__ double sv[kAccThreads / 32];
  __shared__ double res;
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  if (lane == 0) sv[wid] = v;
  __syncthreads();
  if (threadIdx.x == 0) {
    double s = 0.0;
    for (int w = 0; w < kAccThreads / 32; ++w) s += sv[w];
    res = s;
  }
  __syncthreads();
  const double r = res;
  __syncthreads();
  return r;
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

// ---- per-sequence validity (uniform over the block) ------------------------
__device__ bool seq_valid(const AcceptParams& p, int b) {
  __shared__ int s_ok;
  if (threadIdx.x < 32) {
    const int B = p.block[b], g = p.gamma[b];
    bool ok = B >= 1 && B <= 64 && g >= 0 && g <= B && p.slot_off[b] + B <= p.total_slots;
    ok = __all_sync(0xffffffffu, ok);
    if (ok) ok = warp_tau_is_permutation(p.tau + p.slot_off[b], B);
    if (threadIdx.x == 0) s_ok = ok;
  }
  __syncthreads();
  const bool ok = s_ok;
  __syncthreads();
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
      float ma = -INFINITY, mb = -INFINITY;
      for (int c = 0; c < p.nchunks; ++c) { ma = fmaxf(ma, __ldcg(&pp[c].m_a)); mb = fmaxf(mb, __ldcg(&pp[c].m_b)); }
      double sa = 0.0, sb = 0.0;
      for (int c = 0; c < p.nchunks; ++c) {
        sa += __ldcg(&pp[c].s_a) * exp((double)__ldcg(&pp[c].m_a) - (double)ma);
        sb += __ldcg(&pp[c].s_b) * exp((double)__ldcg(&pp[c].m_b) - (double)mb);
      }
      SlotNorm nm;
      nm.m_a = ma; nm.m_b = mb; nm.s_a = sa; nm.s_b = sb;
      p.norm[k] = nm;
      s_dec[tid] = -1;
      int ok = 0;
      if (tid < g) {
        const int d = p.draft_tokens[k];
        if (d >= 0 && d < p.V) {
          const float ad = __fdiv_rn(ld_logit<T>(p.logits, (size_t)k * p.V + d), p.T);
          const float bd = __fdiv_rn(ld_logit<T>(p.draft_logits, (size_t)k * p.V + d), p.T);
          // p(d)/q(d) = exp((a_d - M_a) - (b_d - M_b)) * S_b / S_a
          const double ratio = exp(((double)ad - (double)ma) - ((double)bd - (double)mb)) * (sb / sa);
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
  const int slot = blockIdx.x / p.nchunks;
  const int chunk = blockIdx.x % p.nchunks;
  const int b = find_seq_by_slot(p.slot_off, p.batch, slot);
  if (b < 0) return;
  const int off = p.slot_off[b];
  if (slot - off >= p.block[b]) return;
  if (!seq_valid(p, b)) {
    if (threadIdx.x == 0 && slot == off && chunk == 0) report(p.dev_status, SSV_ERR_BAD_TAU);
    return;
  }
  const int B = p.block[b];
  const int need = min(p.gamma[b] + 1, B);
  if (p.tau[slot] > need) return;

  const int tid = threadIdx.x;
  const size_t rbase = (size_t)slot * p.V;
  const int c0 = chunk * kAccChunk;
  AccPartial out;
  if (MODE != SSV_ACCEPT_REJECT) {
    const float* nrow = nullptr;
    if (MODE == SSV_ACCEPT_GUMBEL) {
      const int nr = p.noise_row[slot];
      if (nr < 0 || nr >= p.n_noise_rows) {
        if (tid == 0) report(p.dev_status, SSV_ERR_INVALID);
        return;
      }
      nrow = p.noise + (size_t)nr * p.V;
    }
    float best = -INFINITY;
    int bi = INT_MAX;
    float x[kAccPerThread];
#pragma unroll
    for (int it = 0; it < kAccPerThread; ++it) {
      const int e = c0 + it * kAccThreads + tid;
      x[it] = e < p.V ? ld_logit<T>(p.logits, rbase + e) : -INFINITY;
    }
    if (MODE == SSV_ACCEPT_GUMBEL) {
#pragma unroll
      for (int it = 0; it < kAccPerThread; ++it) {
        const int e = c0 + it * kAccThreads + tid;
        if (e < p.V) x[it] = __fadd_rn(__fdiv_rn(x[it], p.T), nrow[e]);
      }
    }
#pragma unroll
    for (int it = 0; it < kAccPerThread; ++it) {
      const int e = c0 + it * kAccThreads + tid;
      if (e < p.V && x[it] > best) { best = x[it]; bi = e; }
    }
    block_argmax(best, bi);
    out.val = best; out.idx = bi;
    out.m_a = out.m_b = 0.f; out.s_a = out.s_b = 0.0;
  } else {
    float xa[kAccPerThread], xb[kAccPerThread];
#pragma unroll
    for (int it = 0; it < kAccPerThread; ++it) {
      const int e = c0 + it * kAccThreads + tid;
      xa[it] = e < p.V ? __fdiv_rn(ld_logit<T>(p.logits, rbase + e), p.T) : -INFINITY;
      xb[it] = e < p.V ? __fdiv_rn(ld_logit<T>(p.draft_logits, rbase + e), p.T) : -INFINITY;
    }
    float ma = -INFINITY, mb = -INFINITY;
#pragma unroll
    for (int it = 0; it < kAccPerThread; ++it) { ma = fmaxf(ma, xa[it]); mb = fmaxf(mb, xb[it]); }
    ma = block_max(ma);
    mb = block_max(mb);
    float sa = 0.f, ca = 0.f, sb = 0.f, cb = 0.f;
#pragma unroll
    for (int it = 0; it < kAccPerThread; ++it) {
      kahan_add(sa, ca, expf(xa[it] - ma));
      kahan_add(sb, cb, expf(xb[it] - mb));
    }
    out.m_a = ma; out.m_b = mb;
    out.s_a = block_sum((double)sa - (double)ca);
    out.s_b = block_sum((double)sb - (double)cb);
    out.val = 0.f; out.idx = 0;
  }
  __shared__ int s_last;
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
template <typename T>
__device__ __forceinline__ void sample_weights(const AcceptParams& p, const SlotNorm& nm, size_t rbase, int e,
                                               float inv_sa, float inv_sb, bool residual, float& wr, float& wp) {
  const float pv = expf(__fdiv_rn(ld_logit<T>(p.logits, rbase + e), p.T) - nm.m_a) * inv_sa;
  float qv = 0.f;
  if (residual) qv = expf(__fdiv_rn(ld_logit<T>(p.draft_logits, rbase + e), p.T) - nm.m_b) * inv_sb;
  wp = pv;
  wr = residual ? fmaxf(pv - qv, 0.f) : 0.f;
}

template <typename T>
__global__ void __launch_bounds__(kAccThreads)
accept_sample_kernel(const AcceptParams p) {
  const int b = blockIdx.x / p.nchunks;
  const int chunk = blockIdx.x % p.nchunks;
  // A sequence whose stage map or sizes were rejected never ran its finalize
  // step, so its emission record may be stale: skip it.
  if (!seq_valid(p, b)) return;
  const int eslot = p.emit[2 * b];
  const int soff = p.slot_off[b];
  const int nacc = p.n_acc[b];
  if (eslot < soff || eslot >= soff + p.block[b] || nacc < 0 || nacc >= p.block[b]) return;
  const bool residual = p.emit[2 * b + 1] != 0;
  const SlotNorm nm = p.norm[eslot];
  const float inv_sa = (float)(1.0 / nm.s_a);
  const float inv_sb = residual ? (float)(1.0 / nm.s_b) : 0.f;
  const size_t rbase = (size_t)eslot * p.V;
  const int tid = threadIdx.x;
  const int c0 = chunk * kAccChunk;
  float sr = 0.f, cr = 0.f, sp = 0.f, cp = 0.f;
#pragma unroll 4
  for (int it = 0; it < kAccPerThread; ++it) {
    const int e = c0 + it * kAccThreads + tid;
    if (e < p.V) {
      float wr, wp;
      sample_weights<T>(p, nm, rbase, e, inv_sa, inv_sb, residual, wr, wp);
      kahan_add(sr, cr, wr);
      kahan_add(sp, cp, wp);
    }
  }
  const double mr = block_sum((double)sr - (double)cr);
  const double mp = block_sum((double)sp - (double)cp);
  __shared__ int s_last;
  if (tid == 0) {
    double* sm = p.smass + ((size_t)b * p.nchunks + chunk) * 2;
    sm[0] = mr;
    sm[1] = mp;
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
    const double* sm = p.smass + (size_t)b * p.nchunks * 2;
    double zr = 0.0, zp = 0.0;
    for (int c = 0; c < p.nchunks; ++c) { zr += __ldcg(&sm[2 * c]); zp += __ldcg(&sm[2 * c + 1]); }
    const int use_res = residual && zr > 0.0;
    const int w = use_res ? 0 : 1;
    const double Z = use_res ? zr : zp;
    const double t = (double)p.u_sample[b] * Z;
    double cum = 0.0;
    int cs = -1, last_nz = 0;
    double before = 0.0, before_last = 0.0;
    for (int c = 0; c < p.nchunks; ++c) {
      const double m = __ldcg(&sm[2 * c + w]);
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
  // contiguous run of kAccPerThread entries per thread, vocabulary order
  const int e0 = cs * kAccChunk + tid * kAccPerThread;
  double run[kAccPerThread];
  double local = 0.0;
  int last_pos = -1;
#pragma unroll
  for (int j = 0; j < kAccPerThread; ++j) {
    const int e = e0 + j;
    double w = 0.0;
    if (e < p.V) {
      float wr, wp;
      sample_weights<T>(p, nm, rbase, e, inv_sa, inv_sb, residual, wr, wp);
      w = use_res ? (double)wr : (double)wp;
    }
    if (w > 0.0) last_pos = e;
    run[j] = w;
    local += w;
  }
  const double excl = block_exclusive_scan(local);
  __shared__ int s_pick, s_last_nz;
  if (tid == 0) { s_pick = INT_MAX; s_last_nz = -1; }
  __syncthreads();
  double acc = s_before + excl;
  int pick = INT_MAX;
#pragma unroll
  for (int j = 0; j < kAccPerThread; ++j) {
    acc += run[j];
    if (pick == INT_MAX && run[j] > 0.0 && acc > s_thresh) pick = e0 + j;
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
  p.V = a->V;
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
  p.smass = reinterpret_cast<double*>(w + L.smass);
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
  p.V = a->V;
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
  p.smass = reinterpret_cast<double*>(w + L.smass);
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
