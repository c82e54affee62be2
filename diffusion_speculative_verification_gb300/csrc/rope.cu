// ssv_rope_copy: rotary embedding of Q and K_new with the RoPE-copy index.
//
// SimSD summary, section 3 "Position Encoding Alignment": mask slot D~_k
// reuses the RoPE index of data token D_k.  Fresh prompt row i sits at
// position C + i, tail row r at P + (r mod B).
//
// One CTA handles ROWS consecutive rows.  The (cos, sin) pair of each
// (row, frequency) is computed once into shared memory -- angle formed and
// reduced modulo 2*pi in fp64, since positions reach 10^4 radians and fp32
// would lose ~1e-3 rad -- then every head of Q and K of those rows is
// rotated with 16-byte vector accesses.  HBM-bound: each element is read
// and written once.
#include "ssv_internal.cuh"

#include <math.h>

namespace ssv {

struct RopeTheta {
  double theta[64];  // theta_i = base^(-2i/d), i < d/2
};

constexpr int kRopeRows = 4;
constexpr int kRopeThreads = 256;

template <typename T> struct Vec16;
template <> struct Vec16<float> { static constexpr int N = 4; };
template <> struct Vec16<__nv_bfloat16> { static constexpr int N = 8; };

template <typename T>
__device__ __forceinline__ void load16(const T* p, float* out) {
  const uint4 raw = *reinterpret_cast<const uint4*>(p);
  if constexpr (sizeof(T) == 4) {
    out[0] = __uint_as_float(raw.x); out[1] = __uint_as_float(raw.y);
    out[2] = __uint_as_float(raw.z); out[3] = __uint_as_float(raw.w);
  } else {
    const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      out[2 * i] = __uint_as_float(w[i] << 16);
      out[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
    }
  }
}

template <typename T>
__device__ __forceinline__ void store16(T* p, const float* v) {
  uint4 raw;
  if constexpr (sizeof(T) == 4) {
    raw.x = __float_as_uint(v[0]); raw.y = __float_as_uint(v[1]);
    raw.z = __float_as_uint(v[2]); raw.w = __float_as_uint(v[3]);
  } else {
    uint32_t w[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint32_t lo = __bfloat16_as_ushort(__float2bfloat16_rn(v[2 * i]));
      const uint32_t hi = __bfloat16_as_ushort(__float2bfloat16_rn(v[2 * i + 1]));
      w[i] = lo | (hi << 16);
    }
    raw.x = w[0]; raw.y = w[1]; raw.z = w[2]; raw.w = w[3];
  }
  *reinterpret_cast<uint4*>(p) = raw;
}

template <typename T, int D>
__global__ void __launch_bounds__(kRopeThreads)
rope_copy_kernel(const T* __restrict__ q_in, const T* __restrict__ k_in, T* q_out, T* k_out,
                 int Hq, int Hkv, const ssv_seq* __restrict__ seqs, int batch, int total_rows,
                 const __grid_constant__ RopeTheta th) {
  constexpr int HALF = D / 2;
  constexpr int VEC = Vec16<T>::N;
  constexpr int CHUNKS = HALF / VEC;
  __shared__ float s_cos[kRopeRows][HALF];
  __shared__ float s_sin[kRopeRows][HALF];
  __shared__ int s_pos[kRopeRows];

  const int row0 = blockIdx.x * kRopeRows;
  if (threadIdx.x < kRopeRows) {
    const int row = row0 + threadIdx.x;
    int pos = -1;
    if (row < total_rows) {
      const int b = find_seq_by_row(seqs, batch, row);
      if (b >= 0) {
        const ssv_seq s = seqs[b];
        const int i = row - s.q_off;
        if (i < s.new_len) pos = s.cache_len + i;
        else if (i < s.new_len + 2 * s.block) pos = s.cache_len + s.new_len + (i - s.new_len) % s.block;
      }
    }
    s_pos[threadIdx.x] = pos;
  }
  __syncthreads();
  for (int t = threadIdx.x; t < kRopeRows * HALF; t += blockDim.x) {
    const int lr = t / HALF, i = t % HALF;
    const int pos = s_pos[lr];
    float c = 1.f, s = 0.f;
    if (pos > 0) {
      // a = pos * theta_i, reduced to [-pi, pi] with a two-part 2*pi (fp64).
      const double a = (double)pos * th.theta[i];
      const double kq = rint(a * 0.15915494309189535);   // 1 / (2 pi)
      double r = fma(-kq, 6.283185307179586, a);          // 2 pi, high part
      r = fma(-kq, 2.4492935982947064e-16, r);            // 2 pi, low part
      sincosf((float)r, &s, &c);
    }
    s_cos[lr][i] = c;
    s_sin[lr][i] = s;
  }
  __syncthreads();

  const int heads = Hq + Hkv;
  const int items = kRopeRows * heads * CHUNKS;
  for (int it = threadIdx.x; it < items; it += blockDim.x) {
    const int ch = it % CHUNKS;
    const int hh = (it / CHUNKS) % heads;
    const int lr = it / (CHUNKS * heads);
    const int row = row0 + lr;
    if (s_pos[lr] < 0) continue;
    const T* src;
    T* dst;
    if (hh < Hq) {
      src = q_in + ((size_t)row * Hq + hh) * D;
      dst = q_out + ((size_t)row * Hq + hh) * D;
    } else {
      src = k_in + ((size_t)row * Hkv + (hh - Hq)) * D;
      dst = k_out + ((size_t)row * Hkv + (hh - Hq)) * D;
    }
    float x1[VEC], x2[VEC], y1[VEC], y2[VEC];
    load16<T>(src + ch * VEC, x1);
    load16<T>(src + HALF + ch * VEC, x2);
#pragma unroll
    for (int v = 0; v < VEC; ++v) {
      const float c = s_cos[lr][ch * VEC + v], s = s_sin[lr][ch * VEC + v];
      y1[v] = x1[v] * c - x2[v] * s;
      y2[v] = x2[v] * c + x1[v] * s;
    }
    store16<T>(dst + ch * VEC, y1);
    store16<T>(dst + HALF + ch * VEC, y2);
  }
}

template <typename T, int D>
static cudaError_t launch_rope(const ssv_rope_args* a, const RopeTheta& th, cudaStream_t st) {
  const int grid = (a->total_rows + kRopeRows - 1) / kRopeRows;
  rope_copy_kernel<T, D><<<grid, kRopeThreads, 0, st>>>(
      static_cast<const T*>(a->q_in), static_cast<const T*>(a->k_in), static_cast<T*>(a->q_out),
      static_cast<T*>(a->k_out), a->Hq, a->Hkv, a->seqs, a->batch, a->total_rows, th);
  return cudaGetLastError();
}

}  // namespace ssv

extern "C" ssv_status ssv_rope_copy(const ssv_rope_args* a, void* stream) {
  using namespace ssv;
  if (!a) return SSV_ERR_INVALID;
  if (a->total_rows < 0 || a->batch < 0 || a->Hq <= 0 || a->Hkv <= 0) return SSV_ERR_INVALID;
  if (a->total_rows == 0 || a->batch == 0) return SSV_OK;
  if (!a->q_in || !a->k_in || !a->q_out || !a->k_out || !a->seqs) return SSV_ERR_INVALID;
  if (a->d != 64 && a->d != 128) return SSV_ERR_UNSUPPORTED;
  if (a->dtype != SSV_F32 && a->dtype != SSV_BF16) return SSV_ERR_INVALID;
  if (!(a->base > 1.0) || !isfinite(a->base)) return SSV_ERR_INVALID;
  const uintptr_t al = (uintptr_t)a->q_in | (uintptr_t)a->k_in | (uintptr_t)a->q_out | (uintptr_t)a->k_out;
  if (al & 15u) return SSV_ERR_INVALID;
  RopeTheta th;
  for (int i = 0; i < 64; ++i) th.theta[i] = (i < a->d / 2) ? pow(a->base, -2.0 * i / a->d) : 0.0;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e;
  if (a->dtype == SSV_BF16) {
    e = (a->d == 128) ? launch_rope<__nv_bfloat16, 128>(a, th, st) : launch_rope<__nv_bfloat16, 64>(a, th, st);
  } else {
    e = (a->d == 128) ? launch_rope<float, 128>(a, th, st) : launch_rope<float, 64>(a, th, st);
  }
  return e == cudaSuccess ? SSV_OK : SSV_ERR_CUDA;
}
