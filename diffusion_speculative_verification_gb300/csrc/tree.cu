// Tree (state-set) verification: the attention pass over a draft tree of
// block states and the acceptance by state equality.
//
// SPOT review, "How it works" (a tree of candidate block states, each edge
// committing one position with one token) and "How it is used" (an edge is
// accepted only if the target's next state from its parent equals the
// edge's child, so the accepted set is one path); SimSD summary section 2
// (in a block state, the mask slot of an undecided position sees the
// committed data tokens and the undecided mask slots).
//
// ssv_tree_verify_attn: one CTA of 8 warps per (query row, kv head, group of
// up to 8 of its query heads), fp32 FMA; each key's K and V are loaded once
// for all the group's heads.  A fresh prompt row is causal over cache and
// fresh prompt.  The prompt keys are cut into 8 contiguous ranges, one per
// warp, and the warps' partial softmax states merged.  A mask-slot row M_p
// runs once over the whole prompt (cache + fresh) that way, then, for every
// node n where p is undecided (nodes dealt to the warps in turn), continues a
// copy of the merged state over the node's tail keys -- the data rows of the
// edges on the path to n and the mask rows of the positions undecided at n --
// and writes output row (n, p).  The tree is checked and its per-node bitmasks
// (committed positions, path edges) built in shared memory once per CTA.
//
// ssv_tree_accept: a reduce kernel over (row, vocabulary chunk) records each
// chunk's decision (first argmax of l or of fl(fl(l/T) + G)) and its
// max and sum of 2^((l - max) log2 e); a row kernel (one warp per row) forms
// every row's decision token and confidence l[dec] - logsumexp(l) (the sum
// in double-float); a walk kernel (one warp per sequence) takes, at each node
// of the walk, the most confident undecided position (ties: lowest) and
// follows the edge with that (position, token) (lowest such edge), or emits
// the transition.
#include "ssv_internal.cuh"
#include "accept.cuh"
#include "attn.cuh"
#include "tc_ptx.cuh"

#include <limits.h>
#include <math.h>
#include <string.h>

namespace ssv {
namespace {

constexpr int kTreeMaxB = 64;
constexpr int kTreeMaxE = 63;   // nodes 0..63 fit one 64-bit path mask per node
constexpr int kTreeWarps = 8;   // warps sharing one (row, kv head) task's prompt keys
constexpr int kTreeHeads = 8;   // most query heads a warp serves together

struct TreeAttnParams {
  const void* q;
  const void* k_cache;
  const void* v_cache;
  const void* k_new;
  const void* v_new;
  void* o;
  int Hq, Hkv, d;
  float scale;
  const ssv_tree_seq* seqs;
  int batch;
  const int32_t* parent;
  const int32_t* pos;
  int total_q, total_k, total_cache, total_edges, total_out;
  int max_cache;
  int32_t* dev_status;
  // when set: the prompt part of every query row already done (tensor-core
  // prompt pass): normalised output [total_q][Hq][d] and its log2-sum-exp2
  // [total_q][Hq] (scores scaled by scale * log2 e)
  const float* pre_o;
  const float* pre_lse;
};

// sequence whose rows [key(s), key(s) + span) hold `row` (sequences in increasing order)
template <typename KeyFn>
__device__ __forceinline__ int find_tree_seq(const ssv_tree_seq* seqs, int batch, int row, KeyFn key) {
  int lo = 0, hi = batch - 1, ans = -1;
  while (lo <= hi) {
    const int mid = (lo + hi) >> 1;
    if (key(seqs[mid]) <= row) { ans = mid; lo = mid + 1; } else { hi = mid - 1; }
  }
  return ans;
}

__device__ __forceinline__ bool tree_seq_ok(const ssv_tree_seq& s, int total_q, int total_k, int total_cache,
                                            int total_edges, int total_out) {
  return s.cache_len >= 0 && s.new_len >= 0 && s.block >= 1 && s.block <= kTreeMaxB && s.n_edges >= 0 &&
         s.n_edges <= kTreeMaxE && s.q_off >= 0 && (long long)s.q_off + s.new_len + s.block <= total_q &&
         s.k_off >= 0 && (long long)s.k_off + s.new_len + s.n_edges + s.block <= total_k && s.kv_off >= 0 &&
         (long long)s.kv_off + s.cache_len <= total_cache && s.edge_off >= 0 &&
         (long long)s.edge_off + s.n_edges <= total_edges && s.o_off >= 0 &&
         (long long)s.o_off + s.new_len + (long long)(s.n_edges + 1) * s.block <= total_out;
}

// Lane 0 checks the tree of sequence s and fills, per node n = 0..E, the
// committed-position mask cm[n] and the path-edge mask pm[n]; the answer is
// returned on every lane.  An edge must hang under an earlier node and
// commit a position in 0..B-1 still undecided there.
__device__ __forceinline__ bool build_tree_masks(const ssv_tree_seq& s, const int32_t* parent, const int32_t* pos,
                                                 unsigned long long* cm, unsigned long long* pm) {
  // every edge's (parent, position) loaded at once, two per lane (E <= 63)
  const int lane = threadIdx.x & 31;
  const int pa0 = lane < s.n_edges ? parent[s.edge_off + lane] : 0;
  const int po0 = lane < s.n_edges ? pos[s.edge_off + lane] : 0;
  const int pa1 = lane + 32 < s.n_edges ? parent[s.edge_off + lane + 32] : 0;
  const int po1 = lane + 32 < s.n_edges ? pos[s.edge_off + lane + 32] : 0;
  int ok = 1;
  if (lane == 0) {
    cm[0] = 0ull;
    pm[0] = 0ull;
  }
  __syncwarp();
  for (int e = 0; e < s.n_edges; ++e) {  // warp-uniform walk; lane 0 writes
    const int a0 = __shfl_sync(0xffffffffu, pa0, e & 31), a1 = __shfl_sync(0xffffffffu, pa1, e & 31);
    const int b0 = __shfl_sync(0xffffffffu, po0, e & 31), b1 = __shfl_sync(0xffffffffu, po1, e & 31);
    const int par = e < 32 ? a0 : a1, p = e < 32 ? b0 : b1;
    if (par < -1 || par >= e || p < 0 || p >= s.block) { ok = 0; break; }
    const unsigned long long c = cm[par + 1];
    if ((c >> p) & 1ull) { ok = 0; break; }
    __syncwarp();
    if (lane == 0) {
      cm[e + 1] = c | (1ull << p);
      pm[e + 1] = pm[par + 1] | (1ull << e);
    }
    __syncwarp();
  }
  __syncwarp();
  return ok != 0;
}

template <typename T, int E>
__device__ __forceinline__ void load_lane(const T* p, float* out) {
  if constexpr (sizeof(T) == 4) {
    if constexpr (E == 4) {
      const float4 v = *reinterpret_cast<const float4*>(p);
      out[0] = v.x; out[1] = v.y; out[2] = v.z; out[3] = v.w;
    } else {
      const float2 v = *reinterpret_cast<const float2*>(p);
      out[0] = v.x; out[1] = v.y;
    }
  } else {
    if constexpr (E == 4) {
      const uint2 v = *reinterpret_cast<const uint2*>(p);
      out[0] = __uint_as_float(v.x << 16); out[1] = __uint_as_float(v.x & 0xffff0000u);
      out[2] = __uint_as_float(v.y << 16); out[3] = __uint_as_float(v.y & 0xffff0000u);
    } else {
      const uint32_t v = *reinterpret_cast<const uint32_t*>(p);
      out[0] = __uint_as_float(v << 16); out[1] = __uint_as_float(v & 0xffff0000u);
    }
  }
}

// Running softmax (log2 domain) of up to GH heads, the lane's E columns.
template <int E, int GH>
struct RunState {
  float m[GH], l[GH], acc[GH][E];
};

// One key (k, v rows of this lane) into the running state of the warp's gh <= GH heads.
template <int E, int GH>
__device__ __forceinline__ void add_key(RunState<E, GH>& st, const float (*q)[E], const float* kk, const float* vv,
                                        int gh) {
  float sc[GH];
#pragma unroll
  for (int h = 0; h < GH; ++h) {
    float part = 0.f;
    if (h < gh) {
#pragma unroll
      for (int e = 0; e < E; ++e) part = fmaf(q[h][e], kk[e], part);
    }
    sc[h] = part;
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
#pragma unroll
    for (int h = 0; h < GH; ++h) sc[h] += __shfl_xor_sync(0xffffffffu, sc[h], o);
  }
#pragma unroll
  for (int h = 0; h < GH; ++h) {
    if (h >= gh) continue;
    const float mx = fmaxf(st.m[h], sc[h]);
    const float corr = exp2f(st.m[h] - mx);
    const float pk = exp2f(sc[h] - mx);
    st.l[h] = st.l[h] * corr + pk;
#pragma unroll
    for (int e = 0; e < E; ++e) st.acc[h][e] = fmaf(pk, vv[e], st.acc[h][e] * corr);
    st.m[h] = mx;
  }
}

// NK keys at once into the running state: the NK dot products reduce across
// the warp side by side, and the state is rescaled once per NK keys.
template <int E, int GH, int NK = 4>
__device__ __forceinline__ void add_keys4(RunState<E, GH>& st, const float (*q)[E], const float (*kk)[E],
                                          const float (*vv)[E], int gh) {
  float sc[NK][GH];
#pragma unroll
  for (int k = 0; k < NK; ++k)
#pragma unroll
    for (int h = 0; h < GH; ++h) {
      float part = 0.f;
      if (h < gh) {
#pragma unroll
        for (int e = 0; e < E; ++e) part = fmaf(q[h][e], kk[k][e], part);
      }
      sc[k][h] = part;
    }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1)
#pragma unroll
    for (int k = 0; k < NK; ++k)
#pragma unroll
      for (int h = 0; h < GH; ++h) sc[k][h] += __shfl_xor_sync(0xffffffffu, sc[k][h], o);
#pragma unroll
  for (int h = 0; h < GH; ++h) {
    if (h >= gh) continue;
    float mx = st.m[h];
#pragma unroll
    for (int k = 0; k < NK; ++k) mx = fmaxf(mx, sc[k][h]);
    const float corr = exp2f(st.m[h] - mx);
    float pk[NK], ps = 0.f;
#pragma unroll
    for (int k = 0; k < NK; ++k) {
      pk[k] = exp2f(sc[k][h] - mx);
      ps += pk[k];
    }
    st.l[h] = st.l[h] * corr + ps;
#pragma unroll
    for (int e = 0; e < E; ++e) {
      float a = st.acc[h][e] * corr;
#pragma unroll
      for (int k = 0; k < NK; ++k) a = fmaf(pk[k], vv[k][e], a);
      st.acc[h][e] = a;
    }
    st.m[h] = mx;
  }
}

template <typename OutT, int E, int GH>
__device__ __forceinline__ void store_row(const RunState<E, GH>& st, OutT* o, int h0, int gh, int lane) {
#pragma unroll
  for (int h = 0; h < GH; ++h) {
    if (h >= gh) continue;
    const float inv = 1.f / st.l[h];
    OutT* dst = o + (size_t)(h0 + h) * (size_t)(E * 32) + lane * E;
#pragma unroll
    for (int e = 0; e < E; ++e) dst[e] = Elem<OutT>::from_f32(st.acc[h][e] * inv);
  }
}

template <typename T, typename OutT, int D, int GH>
__global__ void __launch_bounds__(kTreeWarps * 32) tree_attn_kernel(const TreeAttnParams p) {
  constexpr int E = D / 32;
  __shared__ unsigned long long s_cm[kTreeMaxE + 1], s_pm[kTreeMaxE + 1];
  __shared__ float s_ml[kTreeWarps][2][GH];       // each warp's running max and sum per head
  __shared__ float s_acc[kTreeWarps][GH][D];      // and its unnormalised output
  __shared__ int s_ok;
  __shared__ int s_keys[kTreeWarps][kTreeMaxE + kTreeMaxB];  // a node's tail-key rows, per warp
  const int lane = threadIdx.x & 31, wl = threadIdx.x >> 5;
  const int G = p.Hq / p.Hkv;
  const int nhc = (G + GH - 1) / GH;
  // one CTA per (query row, kv head, group of heads): every early return below is CTA-uniform
  const long long w = blockIdx.x;
  if (w >= (long long)p.total_q * p.Hkv * nhc) return;
  const int qr = (int)(w / ((long long)p.Hkv * nhc));
  const int g = (int)((w / nhc) % p.Hkv), hc = (int)(w % nhc);
  const int b = find_tree_seq(p.seqs, p.batch, qr, [](const ssv_tree_seq& s) { return s.q_off; });
  if (b < 0) return;
  const ssv_tree_seq s = p.seqs[b];
  if (!tree_seq_ok(s, p.total_q, p.total_k, p.total_cache, p.total_edges, p.total_out) || s.cache_len > p.max_cache) {
    if (threadIdx.x == 0) report(p.dev_status, SSV_ERR_INVALID);
    return;
  }
  const int i = qr - s.q_off;
  if (i >= s.new_len + s.block) return;
  if (wl == 0) {
    const bool ok = build_tree_masks(s, p.parent, p.pos, s_cm, s_pm);
    if (lane == 0) {
      s_ok = ok ? 1 : 0;
      if (!ok) report(p.dev_status, SSV_ERR_INVALID);
    }
  }
  __syncthreads();
  if (!s_ok) return;
  const unsigned long long* cm = s_cm;
  const unsigned long long* pm = s_pm;
  const int h0 = g * G + hc * GH;
  const int gh = min(GH, G - hc * GH);
  const T* Q = static_cast<const T*>(p.q);
  const T* Kc = static_cast<const T*>(p.k_cache);
  const T* Vc = static_cast<const T*>(p.v_cache);
  const T* Kn = static_cast<const T*>(p.k_new);
  const T* Vn = static_cast<const T*>(p.v_new);
  OutT* O = static_cast<OutT*>(p.o);
  const float qs = p.scale * 1.4426950408889634f;  // fold log2(e)
  float q[GH][E];
#pragma unroll
  for (int h = 0; h < GH; ++h) {
    if (h < gh) {
      load_lane<T, E>(Q + ((size_t)qr * p.Hq + h0 + h) * D + lane * E, q[h]);
#pragma unroll
      for (int e = 0; e < E; ++e) q[h][e] *= qs;
    }
  }
  RunState<E, GH> st;
#pragma unroll
  for (int h = 0; h < GH; ++h) {
    st.m[h] = -INFINITY;
    st.l[h] = 0.f;
#pragma unroll
    for (int e = 0; e < E; ++e) st.acc[h][e] = 0.f;
  }
  auto key_cache = [&](int j, float* kk, float* vv) {
    const size_t off = ((size_t)(s.kv_off + j) * p.Hkv + g) * D + lane * E;
    load_lane<T, E>(Kc + off, kk);
    load_lane<T, E>(Vc + off, vv);
  };
  auto key_new = [&](int j, float* kk, float* vv) {  // j: row of the sequence's new keys
    const size_t off = ((size_t)(s.k_off + j) * p.Hkv + g) * D + lane * E;
    load_lane<T, E>(Kn + off, kk);
    load_lane<T, E>(Vn + off, vv);
  };
  const bool fresh = i < s.new_len;
  const int n_fresh = fresh ? i + 1 : s.new_len;
  if (p.pre_o) {
    // the prompt part from the prompt pass: the state (m = lse, l = 1, acc = O)
    // continues the softmax exactly where that pass left it
    const bool any = s.cache_len + n_fresh > 0;
#pragma unroll
    for (int h = 0; h < GH; ++h) {
      if (h >= gh || !any) continue;
      const size_t r = (size_t)qr * p.Hq + h0 + h;
      st.m[h] = p.pre_lse[r];
      st.l[h] = 1.f;
#pragma unroll
      for (int e = 0; e < E; ++e) st.acc[h][e] = p.pre_o[r * D + lane * E + e];
    }
  } else {
    // prompt keys: the cache, then the fresh prompt rows (all of them for a mask
    // slot; up to the row itself for a fresh row), cut into kTreeWarps
    // contiguous ranges, one per warp; the partial softmax states are then merged
    const int n_prompt = s.cache_len + n_fresh;
    const int j_lo = (int)(((long long)n_prompt * wl) / kTreeWarps);
    const int j_hi = (int)(((long long)n_prompt * (wl + 1)) / kTreeWarps);
    auto key_prompt = [&](int j, float* kk, float* vv) {
      if (j < s.cache_len) key_cache(j, kk, vv);
      else key_new(j - s.cache_len, kk, vv);
    };
    int j = j_lo;
    for (; j + 4 <= j_hi; j += 4) {
      float kk[4][E], vv[4][E];
#pragma unroll
      for (int k = 0; k < 4; ++k) key_prompt(j + k, kk[k], vv[k]);
      add_keys4<E, GH>(st, q, kk, vv, gh);
    }
    for (; j < j_hi; ++j) {
      float kk[E], vv[E];
      key_prompt(j, kk, vv);
      add_key<E, GH>(st, q, kk, vv, gh);
    }
    if (lane == 0) {
#pragma unroll
      for (int h = 0; h < GH; ++h) {
        s_ml[wl][0][h] = st.m[h];
        s_ml[wl][1][h] = st.l[h];
      }
    }
#pragma unroll
    for (int h = 0; h < GH; ++h)
#pragma unroll
      for (int e = 0; e < E; ++e) s_acc[wl][h][lane * E + e] = st.acc[h][e];
    __syncthreads();
    // every warp forms the merged state (the ranges in order; empty ones have max -inf)
#pragma unroll
    for (int h = 0; h < GH; ++h) {
      float M = -INFINITY;
      for (int u = 0; u < kTreeWarps; ++u) M = fmaxf(M, s_ml[u][0][h]);
      float l = 0.f, acc[E];
#pragma unroll
      for (int e = 0; e < E; ++e) acc[e] = 0.f;
      if (M > -INFINITY) {
        for (int u = 0; u < kTreeWarps; ++u) {
          const float mu = s_ml[u][0][h];
          if (!(mu > -INFINITY)) continue;
          const float f = exp2f(mu - M);
          l = fmaf(s_ml[u][1][h], f, l);
#pragma unroll
          for (int e = 0; e < E; ++e) acc[e] = fmaf(s_acc[u][h][lane * E + e], f, acc[e]);
        }
      }
      st.m[h] = M;
      st.l[h] = l;
#pragma unroll
      for (int e = 0; e < E; ++e) st.acc[h][e] = acc[e];
    }
  }
  if (fresh) {
    if (wl == 0) store_row<OutT, E, GH>(st, O + (size_t)(s.o_off + i) * p.Hq * D, h0, gh, lane);
    return;
  }
  // a mask slot: each node where its position is undecided continues a copy of
  // the prompt state over the node's tail keys; nodes dealt to the warps in turn
  const int pp = i - s.new_len;  // position of this mask slot
  const unsigned long long full = (s.block >= 64) ? ~0ull : ((1ull << s.block) - 1ull);
  int* klist = s_keys[wl];
  for (int n = wl; n <= s.n_edges; n += kTreeWarps) {
    if ((cm[n] >> pp) & 1ull) continue;  // committed at n: no row
    // the node's tail keys (rows of the sequence's new keys): the data rows of
    // the path's edges, then the mask rows of the positions undecided at n
    int cnt = 0;
    if (lane == 0) {
      for (unsigned long long m = pm[n]; m; m &= m - 1) klist[cnt++] = s.new_len + __ffsll((long long)m) - 1;
      for (unsigned long long m = full & ~cm[n]; m; m &= m - 1)
        klist[cnt++] = s.new_len + s.n_edges + __ffsll((long long)m) - 1;
    }
    cnt = __shfl_sync(0xffffffffu, cnt, 0);
    __syncwarp();
    RunState<E, GH> t = st;
    int k = 0;
    for (; k + 4 <= cnt; k += 4) {  // four keys' loads in flight at once
      float kk[4][E], vv[4][E];
#pragma unroll
      for (int u = 0; u < 4; ++u) key_new(klist[k + u], kk[u], vv[u]);
      add_keys4<E, GH>(t, q, kk, vv, gh);
    }
    for (; k < cnt; ++k) {
      float kk[E], vv[E];
      key_new(klist[k], kk, vv);
      add_key<E, GH>(t, q, kk, vv, gh);
    }
    __syncwarp();  // the list is rewritten for the warp's next node
    store_row<OutT, E, GH>(t, O + (size_t)(s.o_off + s.new_len + n * s.block + pp) * p.Hq * D, h0, gh, lane);
  }
}

// The prompt pass's sequence table: the tree sequence's cache, fresh prompt
// rows and its B mask-slot query rows; its fresh keys start at k_off (carried
// in tau_off, which a prompt-only pass reads in place of a stage map).
__global__ void tree_prompt_seqs_kernel(const ssv_tree_seq* ts, ssv_seq* out, int batch) {
  const int b = blockIdx.x * blockDim.x + threadIdx.x;
  if (b >= batch) return;
  const ssv_tree_seq t = ts[b];
  ssv_seq o;
  o.cache_len = t.cache_len;
  o.new_len = t.new_len;
  o.block = t.block;
  o.q_off = t.q_off;
  o.kv_off = t.kv_off;
  o.tau_off = t.k_off;
  out[b] = o;
}

template <typename T, typename OutT, int D, int GH>
cudaError_t launch_tree_attn_gh(const TreeAttnParams& p, cudaStream_t st) {
  const int G = p.Hq / p.Hkv;
  const long long grid = (long long)p.total_q * p.Hkv * ((G + GH - 1) / GH);  // one CTA per task
  if (grid > 0x7fffffffLL) return cudaErrorInvalidValue;
  tree_attn_kernel<T, OutT, D, GH><<<(unsigned)grid, kTreeWarps * 32, 0, st>>>(p);
  return cudaGetLastError();
}

// heads served per warp: the group size rounded up to a power of two, at most kTreeHeads
template <typename T, typename OutT, int D>
cudaError_t launch_tree_attn_t(const TreeAttnParams& p, cudaStream_t st) {
  const int G = p.Hq / p.Hkv;
  if (G <= 1) return launch_tree_attn_gh<T, OutT, D, 1>(p, st);
  if (G <= 2) return launch_tree_attn_gh<T, OutT, D, 2>(p, st);
  if (G <= 4) return launch_tree_attn_gh<T, OutT, D, 4>(p, st);
  return launch_tree_attn_gh<T, OutT, D, kTreeHeads>(p, st);
}

// ---------------------------------------------------------------------------
// acceptance
// ---------------------------------------------------------------------------
struct TreeAccParams {
  int mode;
  float T, c2;
  int V, nchunks;
  const ssv_tree_seq* seqs;
  int batch;
  const void* logits;
  const int32_t* parent;
  const int32_t* pos;
  const int32_t* token;
  int total_edges, total_out;
  const float* noise;
  int n_noise_rows;
  const int32_t* noise_row;
  const int32_t* pos_off;
  int total_positions;
  int32_t* n_acc;
  int32_t* path;
  int32_t* emit_pos;
  int32_t* emit_tok;
  int32_t* dev_status;
  AccPartial* part;  // [total_out][nchunks]
  int vec;           // rows (logits and noise) allow 16-byte loads of 8-entry runs
  struct __align__(8) RowConf {
    float conf;      // log-probability of the decision under softmax(l)
    int dec;         // the decision token, -1 if none
  }* rowconf;        // [total_out]
};

constexpr int kTrThreads = 256;

template <int MODE, typename T>
__global__ void __launch_bounds__(kTrThreads) tree_reduce_kernel(const TreeAccParams p) {
  __shared__ float s_v[kTrThreads / 32], s_m[kTrThreads / 32], s_h[kTrThreads / 32], s_l[kTrThreads / 32];
  __shared__ int s_i[kTrThreads / 32];
  const int row = blockIdx.x / p.nchunks, chunk = blockIdx.x % p.nchunks;
  const int b = find_tree_seq(p.seqs, p.batch, row, [](const ssv_tree_seq& s) { return s.o_off; });
  if (b < 0) return;
  const ssv_tree_seq s = p.seqs[b];
  const int li = row - s.o_off - s.new_len;  // node-major (n, p) index
  if (s.block < 1 || s.block > kTreeMaxB || li < 0 || li >= (s.n_edges + 1) * s.block) return;
  const int pp = li % s.block;
  const float* nrow = nullptr;
  if (MODE == SSV_ACCEPT_GUMBEL) {
    const long long k = (long long)p.pos_off[b] + pp;
    const int nr = (k >= 0 && k < p.total_positions) ? p.noise_row[k] : -1;
    if (nr < 0 || nr >= p.n_noise_rows) {
      if (threadIdx.x == 0 && chunk == 0) report(p.dev_status, SSV_ERR_INVALID);
      return;
    }
    nrow = p.noise + (size_t)nr * p.V;
  }
  const T* lrow = static_cast<const T*>(p.logits) + (size_t)row * p.V;
  const int c0 = chunk * kAccChunk;
  const bool unit_t = p.T == 1.0f;  // l / 1 is exact
  float best = -INFINITY, mx = -INFINITY;
  int bi = INT_MAX;
  constexpr int kRuns = kAccChunk / kTrThreads / 8;  // runs of 8 consecutive entries per thread
  float xs[kRuns * 8];  // entries past V hold -inf
#pragma unroll
  for (int g = 0; g < kRuns; ++g) {
    const int e0 = c0 + 8 * (g * kTrThreads + (int)threadIdx.x);
    float x8[8], n8[8];
    if (p.vec && e0 + 8 <= p.V) {  // 16-byte loads
      if constexpr (sizeof(T) == 2) {
        const uint4 u = *reinterpret_cast<const uint4*>(lrow + e0);
        const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          x8[2 * j] = __uint_as_float(w[j] << 16);
          x8[2 * j + 1] = __uint_as_float(w[j] & 0xffff0000u);
        }
      } else {
        const float4 a = *reinterpret_cast<const float4*>(lrow + e0), c = *reinterpret_cast<const float4*>(lrow + e0 + 4);
        x8[0] = a.x; x8[1] = a.y; x8[2] = a.z; x8[3] = a.w; x8[4] = c.x; x8[5] = c.y; x8[6] = c.z; x8[7] = c.w;
      }
      if (MODE == SSV_ACCEPT_GUMBEL) {
        const float4 a = *reinterpret_cast<const float4*>(nrow + e0), c = *reinterpret_cast<const float4*>(nrow + e0 + 4);
        n8[0] = a.x; n8[1] = a.y; n8[2] = a.z; n8[3] = a.w; n8[4] = c.x; n8[5] = c.y; n8[6] = c.z; n8[7] = c.w;
      }
    } else {
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        x8[j] = (e0 + j < p.V) ? Elem<T>::to_f32(lrow[e0 + j]) : -INFINITY;
        n8[j] = (MODE == SSV_ACCEPT_GUMBEL && e0 + j < p.V) ? nrow[e0 + j] : 0.f;
      }
    }
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      xs[g * 8 + j] = x8[j];
      if (MODE == SSV_ACCEPT_GUMBEL && e0 + j < p.V) {
        const float sc = __fadd_rn(unit_t ? x8[j] : __fdiv_rn(x8[j], p.T), n8[j]);
        if (sc > best || bi == INT_MAX) { best = sc; bi = e0 + j; }
      }
    }
  }
  // chunk max (3-input max)
#pragma unroll
  for (int k = 0; k < kRuns * 8; k += 2) mx = ptx::max3(mx, xs[k], xs[k + 1]);
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  const float wm = warp_max(mx);
  if (MODE != SSV_ACCEPT_GUMBEL) {
    // greedy: the score is the logit, so the warp's best is its max; only
    // lanes holding it look for their first entry equal to it (entries in
    // increasing order; past V never)
    if (mx == wm) {
#pragma unroll
      for (int k = 0; k < kRuns * 8; ++k) {
        const int e = c0 + 8 * ((k >> 3) * kTrThreads + (int)threadIdx.x) + (k & 7);
        if (bi == INT_MAX && xs[k] == wm && e < p.V) bi = e;
      }
      best = wm;
    }
  }
  if (lane == 0) s_m[wid] = wm;
  __syncthreads();
  float cm = s_m[0];
#pragma unroll
  for (int w2 = 1; w2 < kTrThreads / 32; ++w2) cm = fmaxf(cm, s_m[w2]);
  // the sum of 2^((x - max) c2): packed f32x2 FMA and add, two chains per thread
  const float nm = (cm == -INFINITY) ? 0.f : -cm * p.c2;
  using namespace ptx;
  const uint64_t c22 = pack2(p.c2, p.c2), nm2 = pack2(nm, nm);
  uint64_t acc2 = pack2(0.f, 0.f);
#pragma unroll
  for (int k = 0; k < kRuns * 8; k += 2) {
    float y0, y1;
    unpack2(ffma2(pack2(xs[k], xs[k + 1]), c22, nm2), y0, y1);
    acc2 = fadd2(acc2, pack2(ex2f(y0), ex2f(y1)));
  }
  float sh, sl = 0.f, s1;
  unpack2(acc2, sh, s1);
  two_sum_acc(sh, sl, s1, 0.f);
  warp_sum2(sh, sl);
  warp_argmax(best, bi);
  if (lane == 0) { s_h[wid] = sh; s_l[wid] = sl; s_v[wid] = best; s_i[wid] = bi; }
  __syncthreads();
  if (threadIdx.x == 0) {
    for (int w2 = 1; w2 < kTrThreads / 32; ++w2) {
      two_sum_acc(sh, sl, s_h[w2], s_l[w2]);
      argmax_combine(best, bi, s_v[w2], s_i[w2]);
    }
    AccPartial r;
    r.m_a = cm; r.sa_hi = sh; r.sa_lo = sl;
    r.m_b = 0.f; r.sb_hi = r.sb_lo = 0.f;
    r.val = best; r.idx = bi;
    p.part[(size_t)row * p.nchunks + chunk] = r;
  }
}

// Every output row's decision and confidence from its chunk records, one
// warp per row (lanes over chunks), all rows at once (the walk then only
// compares them).  No fp64 (a narrow pipe on this part): the normaliser
// S = sum of s_c e^(m_c - M) in double-float, each scale factor an fp32 exp2
// of an argument formed from the exact difference m_c - M.
constexpr int kConfWarps = 4;

template <int MODE, typename T>
__global__ void __launch_bounds__(kConfWarps * 32) tree_rowconf_kernel(const TreeAccParams p) {
  pdl_wait();  // the chunk records
  pdl_trigger();
  const int lane = threadIdx.x & 31;
  const int row = blockIdx.x * kConfWarps + (threadIdx.x >> 5);
  if (row >= p.total_out) return;
  const int b = find_tree_seq(p.seqs, p.batch, row, [](const ssv_tree_seq& s) { return s.o_off; });
  if (b < 0) return;
  const ssv_tree_seq s = p.seqs[b];
  const int li = row - s.o_off - s.new_len;
  if (s.block < 1 || s.block > kTreeMaxB || li < 0 || li >= (s.n_edges + 1) * s.block) return;
  const AccPartial* pr = p.part + (size_t)row * p.nchunks;
  float v = -INFINITY, M = -INFINITY;
  int idx = INT_MAX;
  for (int c = lane; c < p.nchunks; c += 32) {
    argmax_combine(v, idx, __ldcg(&pr[c].val), __ldcg(&pr[c].idx));
    M = fmaxf(M, __ldcg(&pr[c].m_a));
  }
  warp_argmax(v, idx);
  M = warp_max(M);
  dfx S{0.f, 0.f};
  for (int c = lane; c < p.nchunks; c += 32) {
    const float cmx = __ldcg(&pr[c].m_a);
    if (cmx == -INFINITY) continue;
    const dfx cs{__ldcg(&pr[c].sa_hi), __ldcg(&pr[c].sa_lo)};
    const dfx dm = dfx_two_sum(cmx, -M);  // exact m_c - M <= 0
    const float f = (cmx == M) ? 1.f : exp2f(__fmaf_rn(dm.hi, p.c2, __fmul_rn(dm.lo, p.c2)));
    S = dfx_add(S, dfx_mul(cs, dfx{f, 0.f}));
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1)
    S = dfx_add(S, dfx{__shfl_xor_sync(0xffffffffu, S.hi, o), __shfl_xor_sync(0xffffffffu, S.lo, o)});
  if (lane != 0) return;
  TreeAccParams::RowConf rc;
  rc.dec = -1;
  rc.conf = -INFINITY;
  if (idx != INT_MAX) {
    const float ld = (MODE == SSV_ACCEPT_GUMBEL) ? Elem<T>::to_f32(static_cast<const T*>(p.logits)[(size_t)row * p.V + idx])
                                                 : v;
    // (l_d - M) - ln S, S = sum e^(l - M) >= 1; ln(hi + lo) = ln hi + lo / hi to first order
    rc.conf = __fsub_rn(__fsub_rn(ld, M), __fadd_rn(logf(S.hi), __fdiv_rn(S.lo, S.hi)));
    rc.dec = idx;
  }
  p.rowconf[row] = rc;
}

template <int MODE, typename T>
__global__ void __launch_bounds__(32) tree_walk_kernel(const TreeAccParams p) {
  __shared__ unsigned long long s_cm[kTreeMaxE + 1], s_pm[kTreeMaxE + 1];
  const int b = blockIdx.x, lane = threadIdx.x;
  pdl_wait();
  const ssv_tree_seq s = p.seqs[b];
  if (lane < 32) {
    for (int j = lane; j < kTreeMaxB; j += 32) p.path[(size_t)b * kTreeMaxB + j] = -1;
  }
  const bool ok = s.block >= 1 && s.block <= kTreeMaxB && s.n_edges >= 0 && s.n_edges <= kTreeMaxE &&
                  s.edge_off >= 0 && (long long)s.edge_off + s.n_edges <= p.total_edges && s.o_off >= 0 &&
                  (long long)s.o_off + s.new_len + (long long)(s.n_edges + 1) * s.block <= p.total_out &&
                  s.new_len >= 0;
  if (!ok || !build_tree_masks(s, p.parent, p.pos, s_cm, s_pm)) {
    if (lane == 0) {
      report(p.dev_status, SSV_ERR_INVALID);
      p.n_acc[b] = -1;
      p.emit_pos[b] = -1;
      p.emit_tok[b] = -1;
    }
    return;
  }
  const unsigned long long full = (s.block >= 64) ? ~0ull : ((1ull << s.block) - 1ull);
  int n = 0, acc = 0, epos = -1, etok = -1;
  while (true) {
    const unsigned long long und = full & ~s_cm[n];
    if (!und) break;
    // each lane: positions lane and lane + 32
    float best_c = -INFINITY;
    int best_p = INT_MAX, best_t = -1;
#pragma unroll
    for (int hpos = 0; hpos < 2; ++hpos) {
      const int pp = lane + 32 * hpos;
      if (pp >= s.block || !((und >> pp) & 1ull)) continue;
      const size_t row = (size_t)s.o_off + s.new_len + (size_t)n * s.block + pp;
      const int dec = __ldcg(&p.rowconf[row].dec);
      if (dec < 0) continue;
      const float conf = __ldcg(&p.rowconf[row].conf);  // log-probability of the decision under softmax(l)
      if (conf > best_c || (conf == best_c && pp < best_p)) { best_c = conf; best_p = pp; best_t = dec; }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float oc = __shfl_xor_sync(0xffffffffu, best_c, o);
      const int op = __shfl_xor_sync(0xffffffffu, best_p, o), ot = __shfl_xor_sync(0xffffffffu, best_t, o);
      if (oc > best_c || (oc == best_c && op < best_p)) { best_c = oc; best_p = op; best_t = ot; }
    }
    if (best_p == INT_MAX) break;  // no decision (V = 0 cannot happen; defensive)
    // the child edge carrying that transition (lowest edge id)
    unsigned found = 0;
    int echild = -1;
#pragma unroll
    for (int h2 = 0; h2 < 2; ++h2) {
      const int e = lane + 32 * h2;
      const bool hit = e < s.n_edges && p.parent[s.edge_off + e] + 1 == n && p.pos[s.edge_off + e] == best_p &&
                       p.token[s.edge_off + e] == best_t;
      const unsigned bl = __ballot_sync(0xffffffffu, hit);
      if (bl && echild < 0) { echild = 32 * h2 + __ffs(bl) - 1; found = 1; }
    }
    if (!found) { epos = best_p; etok = best_t; break; }
    if (lane == 0) p.path[(size_t)b * kTreeMaxB + acc] = echild;
    ++acc;
    n = echild + 1;
  }
  if (lane == 0) {
    p.n_acc[b] = acc;
    p.emit_pos[b] = epos;
    p.emit_tok[b] = etok;
  }
}

}  // namespace
}  // namespace ssv

using namespace ssv;

namespace {

ssv_status tree_attn_check(const ssv_tree_attn_args* a) {
  if (!a) return SSV_ERR_INVALID;
  if (a->batch < 0 || a->total_q < 0 || a->total_k < 0 || a->total_cache < 0 || a->total_edges < 0 ||
      a->total_out < 0)
    return SSV_ERR_INVALID;
  if (a->Hq <= 0 || a->Hkv <= 0 || a->Hq % a->Hkv != 0) return SSV_ERR_INVALID;
  if (a->d != 64 && a->d != 128) return SSV_ERR_UNSUPPORTED;
  if (a->in_dtype != SSV_F32 && a->in_dtype != SSV_BF16) return SSV_ERR_INVALID;
  if (a->out_dtype != SSV_F32 && a->out_dtype != SSV_BF16) return SSV_ERR_INVALID;
  if (a->in_dtype == SSV_F32 && a->out_dtype != SSV_F32) return SSV_ERR_UNSUPPORTED;
  if (!isfinite(a->scale) || a->scale < 0.f || a->max_cache < 0) return SSV_ERR_INVALID;
  if (a->batch == 0 || a->total_q == 0) return SSV_OK;
  if (!a->q || !a->k_new || !a->v_new || !a->o || !a->seqs || (a->total_edges > 0 && (!a->parent || !a->pos)))
    return SSV_ERR_INVALID;
  if (a->total_cache > 0 && (!a->k_cache || !a->v_cache)) return SSV_ERR_INVALID;
  const uintptr_t al = (uintptr_t)a->q | (uintptr_t)a->k_cache | (uintptr_t)a->v_cache | (uintptr_t)a->k_new |
                       (uintptr_t)a->v_new | (uintptr_t)a->o;
  if (al & 15u) return SSV_ERR_INVALID;
  return SSV_OK;
}

float tree_scale(const ssv_tree_attn_args* a) {
  return a->scale > 0.f ? a->scale : (float)(1.0 / sqrt((double)a->d));
}

// The prompt pass as a prompt-only verify-attention pass on the tensor cores:
// its parameters (workspace pointers left for the caller), or false when the
// shapes are outside that schedule (fp32 inputs, d = 64, ...).
bool tree_prompt_params(const ssv_tree_attn_args* a, AttnParams& ap) {
  if (a->in_dtype != SSV_BF16 || a->d != 128) return false;
  memset(&ap, 0, sizeof(ap));
  ap.q = a->q;
  ap.k_cache = a->k_cache;
  ap.v_cache = a->v_cache;
  ap.k_new = a->k_new;
  ap.v_new = a->v_new;
  ap.in_dtype = SSV_BF16;
  ap.out_dtype = SSV_F32;
  ap.Hq = a->Hq;
  ap.Hkv = a->Hkv;
  ap.d = a->d;
  ap.scale = tree_scale(a);
  ap.batch = a->batch;
  ap.tau = nullptr;
  ap.total_rows = a->total_q;
  ap.total_cache = a->total_cache;
  ap.total_slots = 0;
  ap.max_cache = a->max_cache;
  ap.max_new = a->total_q;  // every N is below the query rows
  ap.max_block = kTreeMaxB;
  ap.dev_status = a->dev_status;
  ap.early = 0;
  ap.wait_budget = kDefaultWaitBudget;
  ap.fault_skip = -1;
  ap.prompt_only = 1;
  ap.total_krows = a->total_k;
  return tc::attn_tc_supported(ap);
}

struct TreeWs {
  size_t attn, o, lse, seqs, total;
};

TreeWs tree_ws_layout(const ssv_tree_attn_args* a, const AttnParams& ap) {
  TreeWs L;
  size_t off = 0;
  L.attn = off;
  off = align_up(off + tc::attn_tc_workspace(ap), 256);
  L.o = off;
  off = align_up(off + sizeof(float) * (size_t)a->total_q * a->Hq * a->d, 256);
  L.lse = off;
  off = align_up(off + sizeof(float) * (size_t)a->total_q * a->Hq, 256);
  L.seqs = off;
  off = align_up(off + sizeof(ssv_seq) * (size_t)a->batch, 256);
  L.total = off;
  return L;
}

}  // namespace

extern "C" ssv_status ssv_tree_verify_attn_workspace(const ssv_tree_attn_args* a, size_t* bytes) {
  if (!bytes) return SSV_ERR_INVALID;
  const ssv_status v = tree_attn_check(a);
  if (v != SSV_OK) return v;
  *bytes = 0;
  AttnParams ap;
  if (a->batch > 0 && a->total_q > 0 && tree_prompt_params(a, ap)) *bytes = tree_ws_layout(a, ap).total;
  return SSV_OK;
}

extern "C" ssv_status ssv_tree_verify_attn(const ssv_tree_attn_args* a, void* ws, size_t ws_bytes, void* stream) {
  const ssv_status v = tree_attn_check(a);
  if (v != SSV_OK) return v;
  if (a->batch == 0 || a->total_q == 0) return SSV_OK;
  TreeAttnParams p;
  p.q = a->q; p.k_cache = a->k_cache; p.v_cache = a->v_cache; p.k_new = a->k_new; p.v_new = a->v_new; p.o = a->o;
  p.Hq = a->Hq; p.Hkv = a->Hkv; p.d = a->d;
  p.scale = tree_scale(a);
  p.seqs = a->seqs; p.batch = a->batch; p.parent = a->parent; p.pos = a->pos;
  p.total_q = a->total_q; p.total_k = a->total_k; p.total_cache = a->total_cache;
  p.total_edges = a->total_edges; p.total_out = a->total_out; p.max_cache = a->max_cache;
  p.dev_status = a->dev_status;
  p.pre_o = nullptr;
  p.pre_lse = nullptr;
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaSuccess;
  AttnParams ap;
  if (tree_prompt_params(a, ap)) {
    // the prompt part of every query row on the tensor cores, then the nodes
    const TreeWs L = tree_ws_layout(a, ap);
    if (!ws || ((uintptr_t)ws & 255u) || ws_bytes < L.total) return SSV_ERR_WORKSPACE;
    char* w = static_cast<char*>(ws);
    ssv_seq* pseqs = reinterpret_cast<ssv_seq*>(w + L.seqs);
    tree_prompt_seqs_kernel<<<(a->batch + 127) / 128, 128, 0, st>>>(a->seqs, pseqs, a->batch);
    e = cudaGetLastError();
    ap.seqs = pseqs;
    ap.o = w + L.o;
    ap.lse = reinterpret_cast<float*>(w + L.lse);
    if (e == cudaSuccess) e = tc::launch_attn_tc(ap, w + L.attn, st);
    p.pre_o = reinterpret_cast<const float*>(w + L.o);
    p.pre_lse = reinterpret_cast<const float*>(w + L.lse);
  }
  if (e != cudaSuccess) return SSV_ERR_CUDA;
  const bool bf = a->in_dtype == SSV_BF16, obf = a->out_dtype == SSV_BF16;
  if (a->d == 128) {
    e = !bf ? launch_tree_attn_t<float, float, 128>(p, st)
            : (obf ? launch_tree_attn_t<__nv_bfloat16, __nv_bfloat16, 128>(p, st)
                   : launch_tree_attn_t<__nv_bfloat16, float, 128>(p, st));
  } else {
    e = !bf ? launch_tree_attn_t<float, float, 64>(p, st)
            : (obf ? launch_tree_attn_t<__nv_bfloat16, __nv_bfloat16, 64>(p, st)
                   : launch_tree_attn_t<__nv_bfloat16, float, 64>(p, st));
  }
  return e == cudaSuccess ? SSV_OK : SSV_ERR_CUDA;
}

static ssv_status tree_accept_check(const ssv_tree_accept_args* a, int* nchunks) {
  if (!a) return SSV_ERR_INVALID;
  if (a->mode != SSV_ACCEPT_ARGMAX && a->mode != SSV_ACCEPT_GUMBEL) return SSV_ERR_INVALID;
  if (!isfinite(a->T) || a->T < 0.f) return SSV_ERR_NOT_FINITE;
  if (a->V < 1 || a->batch < 0 || a->total_out < 0 || a->total_edges < 0) return SSV_ERR_INVALID;
  if (a->logits_dtype != SSV_F32 && a->logits_dtype != SSV_BF16) return SSV_ERR_INVALID;
  *nchunks = (a->V + kAccChunk - 1) / kAccChunk;
  if (a->batch == 0) return SSV_OK;
  if (!a->seqs || !a->logits || !a->n_acc || !a->path || !a->emit_pos || !a->emit_tok) return SSV_ERR_INVALID;
  if (a->total_edges > 0 && (!a->parent || !a->pos || !a->token)) return SSV_ERR_INVALID;
  if (a->mode == SSV_ACCEPT_GUMBEL && a->T > 0.f &&
      (!a->noise || !a->noise_row || !a->pos_off || a->n_noise_rows < 1 || a->total_positions < 1))
    return SSV_ERR_INVALID;
  return SSV_OK;
}

extern "C" ssv_status ssv_tree_accept_workspace(const ssv_tree_accept_args* a, size_t* bytes) {
  if (!bytes) return SSV_ERR_INVALID;
  int nchunks = 0;
  const ssv_status st = tree_accept_check(a, &nchunks);
  if (st != SSV_OK) return st;
  *bytes = align_up(sizeof(AccPartial) * (size_t)a->total_out * nchunks, 256) +
           align_up(sizeof(TreeAccParams::RowConf) * (size_t)a->total_out + 256, 256);
  return SSV_OK;
}

extern "C" ssv_status ssv_tree_accept(const ssv_tree_accept_args* a, void* ws, size_t ws_bytes, void* stream) {
  int nchunks = 0;
  ssv_status st = tree_accept_check(a, &nchunks);
  if (st != SSV_OK) return st;
  if (a->batch == 0) return SSV_OK;
  size_t need = 0;
  ssv_tree_accept_workspace(a, &need);
  if (!ws || ((uintptr_t)ws & 255u) || ws_bytes < need) return SSV_ERR_WORKSPACE;
  TreeAccParams p;
  int mode = a->mode;
  if (mode == SSV_ACCEPT_GUMBEL && a->T == 0.f) mode = SSV_ACCEPT_ARGMAX;
  p.mode = mode;
  p.T = a->T;                     // the coupled-noise decision divides by T
  p.c2 = 1.4426950408889634f;     // confidences use softmax(l): weights 2^((l - max) log2 e) = e^(l - max)
  p.V = a->V;
  p.nchunks = nchunks;
  p.seqs = a->seqs; p.batch = a->batch; p.logits = a->logits;
  p.parent = a->parent; p.pos = a->pos; p.token = a->token;
  p.total_edges = a->total_edges; p.total_out = a->total_out;
  p.noise = a->noise; p.n_noise_rows = a->n_noise_rows; p.noise_row = a->noise_row; p.pos_off = a->pos_off;
  p.total_positions = a->total_positions;
  p.n_acc = a->n_acc; p.path = a->path; p.emit_pos = a->emit_pos; p.emit_tok = a->emit_tok;
  p.dev_status = a->dev_status;
  p.part = static_cast<AccPartial*>(ws);
  p.rowconf = reinterpret_cast<TreeAccParams::RowConf*>(static_cast<char*>(ws) +
                                                        align_up(sizeof(AccPartial) * (size_t)a->total_out * nchunks, 256));
  {
    const size_t es = a->logits_dtype == SSV_BF16 ? 2 : 4;
    bool v = ((size_t)a->V * es) % 16 == 0 && ((uintptr_t)a->logits & 15u) == 0;
    if (mode == SSV_ACCEPT_GUMBEL) v = v && ((size_t)a->V * 4) % 16 == 0 && ((uintptr_t)a->noise & 15u) == 0;
    p.vec = v ? 1 : 0;
  }
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  const long long g1 = (long long)a->total_out * nchunks;
  if (g1 > 0x7fffffffLL) return SSV_ERR_INVALID;
  const bool bf = a->logits_dtype == SSV_BF16;
  cudaError_t e = cudaSuccess;
  const TreeAccParams& pr = p;
  if (g1 > 0) {
    if (mode == SSV_ACCEPT_GUMBEL) {
      if (bf) tree_reduce_kernel<SSV_ACCEPT_GUMBEL, __nv_bfloat16><<<(unsigned)g1, kTrThreads, 0, s>>>(pr);
      else tree_reduce_kernel<SSV_ACCEPT_GUMBEL, float><<<(unsigned)g1, kTrThreads, 0, s>>>(pr);
    } else {
      if (bf) tree_reduce_kernel<SSV_ACCEPT_ARGMAX, __nv_bfloat16><<<(unsigned)g1, kTrThreads, 0, s>>>(pr);
      else tree_reduce_kernel<SSV_ACCEPT_ARGMAX, float><<<(unsigned)g1, kTrThreads, 0, s>>>(pr);
    }
    e = cudaGetLastError();
  }
  if (e == cudaSuccess && a->total_out > 0) {
    const dim3 gr((unsigned)((a->total_out + kConfWarps - 1) / kConfWarps)), bl(kConfWarps * 32);
    if (mode == SSV_ACCEPT_GUMBEL)
      e = bf ? launch_pdl(tree_rowconf_kernel<SSV_ACCEPT_GUMBEL, __nv_bfloat16>, gr, bl, 0, s, p)
             : launch_pdl(tree_rowconf_kernel<SSV_ACCEPT_GUMBEL, float>, gr, bl, 0, s, p);
    else
      e = bf ? launch_pdl(tree_rowconf_kernel<SSV_ACCEPT_ARGMAX, __nv_bfloat16>, gr, bl, 0, s, p)
             : launch_pdl(tree_rowconf_kernel<SSV_ACCEPT_ARGMAX, float>, gr, bl, 0, s, p);
  }
  if (e == cudaSuccess) {
    if (mode == SSV_ACCEPT_GUMBEL)
      e = bf ? launch_pdl(tree_walk_kernel<SSV_ACCEPT_GUMBEL, __nv_bfloat16>, dim3(a->batch), dim3(32), 0, s, p)
             : launch_pdl(tree_walk_kernel<SSV_ACCEPT_GUMBEL, float>, dim3(a->batch), dim3(32), 0, s, p);
    else
      e = bf ? launch_pdl(tree_walk_kernel<SSV_ACCEPT_ARGMAX, __nv_bfloat16>, dim3(a->batch), dim3(32), 0, s, p)
             : launch_pdl(tree_walk_kernel<SSV_ACCEPT_ARGMAX, float>, dim3(a->batch), dim3(32), 0, s, p);
  }
  return e == cudaSuccess ? SSV_OK : SSV_ERR_CUDA;
}
