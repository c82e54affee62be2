// SIMT verify attention: one warp per (query row, query head), fp32 FMA
// throughout.  This is the exact path for fp32 inputs (no tensor cores:
// tf32 would miss a 1e-5 tolerance) and the fallback schedule for shapes the
// tensor-core kernels do not cover.
//
// SimSD summary, section 2: the temporal mask is evaluated on the fly from
// tau for the 2B tail keys; prompt keys are causal for fresh prompt rows and
// fully visible to tail rows.  Online softmax in the log2 domain.
#include "ssv_internal.cuh"
#include "attn.cuh"

namespace ssv {

constexpr int kSimtWarps = 4;

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

template <typename T, typename OutT, int D>
__global__ void __launch_bounds__(kSimtWarps * 32)
attn_simt_kernel(const AttnParams p) {
  constexpr int E = D / 32;
  const int lane = threadIdx.x & 31;
  const long long w = (long long)blockIdx.x * kSimtWarps + (threadIdx.x >> 5);
  if (w >= (long long)p.total_rows * p.Hq) return;
  const int row = (int)(w / p.Hq);
  const int h = (int)(w % p.Hq);
  const int b = find_seq_by_row(p.seqs, p.batch, row);
  if (b < 0) return;
  const ssv_seq s = p.seqs[b];
  const int i = row - s.q_off;
  const int B = s.block;
  if (!seq_extents_ok(s, p.total_rows, p.total_cache, p.total_slots) || s.cache_len > p.max_cache ||
      s.new_len > p.max_new || s.block > p.max_block) {
    if (lane == 0) report(p.dev_status, SSV_ERR_INVALID);  // sequence outside the buffers: skipped
    return;
  }
  if (i >= s.new_len + 2 * B) return;
  const int kvh = h / (p.Hq / p.Hkv);
  const int32_t* tau = p.tau + s.tau_off;
  if (!warp_tau_is_permutation(tau, B)) {
    if (lane == 0) report(p.dev_status, SSV_ERR_BAD_TAU);
    return;
  }

  const T* Q = static_cast<const T*>(p.q);
  const T* Kc = static_cast<const T*>(p.k_cache);
  const T* Vc = static_cast<const T*>(p.v_cache);
  const T* Kn = static_cast<const T*>(p.k_new);
  const T* Vn = static_cast<const T*>(p.v_new);

  float q[E];
  load_lane<T, E>(Q + ((size_t)row * p.Hq + h) * D + lane * E, q);
  const float qs = p.scale * 1.4426950408889634f;  // fold log2(e)
#pragma unroll
  for (int e = 0; e < E; ++e) q[e] *= qs;

  float m = -INFINITY, l = 0.f, acc[E];
#pragma unroll
  for (int e = 0; e < E; ++e) acc[e] = 0.f;

  const bool tail_row = i >= s.new_len;
  const int r = i - s.new_len;                    // tail row index when tail_row
  const int tau_r = tail_row ? tau[r % B] : 0;
  const int n_new = tail_row ? s.new_len + 2 * B : i + 1;   // new-segment keys to scan
  const int total_keys = s.cache_len + n_new;

  constexpr int U = 4;
  for (int j0 = 0; j0 < total_keys; j0 += U) {
    float sc[U];
    float vv[U][E];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int j = j0 + u;
      bool ok = j < total_keys;
      const T* kp = nullptr;
      const T* vp = nullptr;
      if (ok) {
        if (j < s.cache_len) {
          const size_t off = ((size_t)(s.kv_off + j) * p.Hkv + kvh) * D + lane * E;
          kp = Kc + off; vp = Vc + off;
        } else {
          const int jn = j - s.cache_len;
          if (tail_row && jn >= s.new_len) {
            const int t = jn - s.new_len;
            ok = tail_allowed(r, t, B, tau_r, tau[t % B]);
          }
          const size_t off = ((size_t)(s.q_off + jn) * p.Hkv + kvh) * D + lane * E;
          kp = Kn + off; vp = Vn + off;
        }
      }
      float part = 0.f;
      if (ok) {
        float kk[E];
        load_lane<T, E>(kp, kk);
        load_lane<T, E>(vp, vv[u]);
#pragma unroll
        for (int e = 0; e < E; ++e) part = fmaf(q[e], kk[e], part);
      } else {
#pragma unroll
        for (int e = 0; e < E; ++e) vv[u][e] = 0.f;
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) part += __shfl_xor_sync(0xffffffffu, part, o);
      sc[u] = ok ? part : -INFINITY;
    }
    float mx = m;
#pragma unroll
    for (int u = 0; u < U; ++u) mx = fmaxf(mx, sc[u]);
    if (mx == -INFINITY) continue;
    const float corr = exp2f(m - mx);
    l *= corr;
#pragma unroll
    for (int e = 0; e < E; ++e) acc[e] *= corr;
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const float pk = exp2f(sc[u] - mx);
      l += pk;
#pragma unroll
      for (int e = 0; e < E; ++e) acc[e] = fmaf(pk, vv[u][e], acc[e]);
    }
    m = mx;
  }
  const float inv = 1.f / l;
  OutT* O = static_cast<OutT*>(p.o) + ((size_t)row * p.Hq + h) * D + lane * E;
#pragma unroll
  for (int e = 0; e < E; ++e) O[e] = Elem<OutT>::from_f32(acc[e] * inv);
}

template <typename T, typename OutT, int D>
static cudaError_t launch_simt_t(const AttnParams& p, cudaStream_t st) {
  const long long warps = (long long)p.total_rows * p.Hq;
  const long long grid = (warps + kSimtWarps - 1) / kSimtWarps;
  if (grid > 0x7fffffffLL) return cudaErrorInvalidValue;
  attn_simt_kernel<T, OutT, D><<<(unsigned)grid, kSimtWarps * 32, 0, st>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_attn_simt(const AttnParams& p, cudaStream_t st) {
  if (p.in_dtype == SSV_F32) {
    if (p.out_dtype != SSV_F32) return cudaErrorInvalidValue;
    return p.d == 128 ? launch_simt_t<float, float, 128>(p, st) : launch_simt_t<float, float, 64>(p, st);
  }
  if (p.out_dtype == SSV_F32)
    return p.d == 128 ? launch_simt_t<__nv_bfloat16, float, 128>(p, st)
                      : launch_simt_t<__nv_bfloat16, float, 64>(p, st);
  return p.d == 128 ? launch_simt_t<__nv_bfloat16, __nv_bfloat16, 128>(p, st)
                    : launch_simt_t<__nv_bfloat16, __nv_bfloat16, 64>(p, st);
}

}  // namespace ssv
