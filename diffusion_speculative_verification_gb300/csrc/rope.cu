// ssv_rope_copy: rotary embedding of Q and K_new with the RoPE-copy index.
//
// SimSD summary, section 3 "Position Encoding Alignment": mask slot D~_k
// reuses the RoPE index of data token D_k.  Fresh prompt row i sits at
// position C + i, tail row r at P + (r mod B); or, with a position table,
// each fresh row and each data row D_k at its table entry and D~_k at D_k's.
//
// One CTA handles ROWS consecutive rows.  Their first elements are loaded
// at entry, together with the sequence table, so that the one DRAM round
// trip covers both.  The (cos, sin) pair of each (row, frequency) is then
// computed once into shared memory -- angle formed and reduced modulo 2*pi
// in fp64, since positions reach 10^4 radians and fp32 would lose ~1e-3
// rad -- and every head of Q and K of those rows is rotated with 16-byte
// vector accesses.  HBM-bound: each element is read and written once.
#include "ssv_internal.cuh"

#include <math.h>

namespace ssv {

struct RopeTheta {
  double theta[64];  // theta_i = base^(-2i/d), i < d/2
};

constexpr int kRopeRows = 4;  // rows per CTA (one when that leaves most SMs idle)
constexpr int kRopeThreads = 256;

template <typename T> struct Vec16;
template <> struct Vec16<float> { static constexpr int N = 4; };
template <> struct Vec16<__nv_bfloat16> { static constexpr int N = 8; };

template <typename T>
__device__ __forceinline__ void unpack16(const uint4 raw, float* out) {
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
__device__ __forceinline__ void load16(const T* p, float* out) {
  unpack16<T>(*reinterpret_cast<const uint4*>(p), out);
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

template <typename T, int D, int ROWS>
__global__ void __launch_bounds__(kRopeThreads, 4)  // four CTAs per SM: a whole decode batch in one wave
rope_copy_kernel(const T* __restrict__ q_in, const T* __restrict__ k_in, T* q_out, T* k_out,
                 int Hq, int Hkv, const ssv_seq* __restrict__ seqs, int batch, int total_rows,
                 const int32_t* __restrict__ positions, int32_t* dev_status,
                 const __grid_constant__ RopeTheta th) {
  constexpr int HALF = D / 2;
  constexpr int VEC = Vec16<T>::N;
  constexpr int CHUNKS = HALF / VEC;
  constexpr int PRE = 5;  // items per thread loaded before the positions are known (all of them up to 40 heads)
  __shared__ float s_cos[ROWS][HALF];
  __shared__ float s_sin[ROWS][HALF];
  __shared__ int s_pos[ROWS];
  __shared__ ssv_seq s_seq[kRopeThreads];

  pdl_wait();  // Q and K come from the preceding kernel
  pdl_trigger();  // dependents start only once every kernel before this one is complete
  const int row0 = blockIdx.x * ROWS;
  const int heads = Hq + Hkv;
  const int items = ROWS * heads * CHUNKS;
  auto item_ptrs = [&](int it, const T*& src, T*& dst, int& lr, int& ch) -> bool {
    ch = it % CHUNKS;
    const int hh = (it / CHUNKS) % heads;
    lr = it / (CHUNKS * heads);
    const int row = row0 + lr;
    if (row >= total_rows) return false;
    if (hh < Hq) {
      src = q_in + ((size_t)row * Hq + hh) * D;
      dst = q_out + ((size_t)row * Hq + hh) * D;
    } else {
      src = k_in + ((size_t)row * Hkv + (hh - Hq)) * D;
      dst = k_out + ((size_t)row * Hkv + (hh - Hq)) * D;
    }
    return true;
  };
  // The rows' data does not depend on the positions: issue those loads first,
  // together with the sequence table (one round trip for both).
  uint4 pr1[PRE], pr2[PRE];  // kept packed until the angles are known
#pragma unroll
  for (int k = 0; k < PRE; ++k) {
    const int it = threadIdx.x + k * kRopeThreads;
    const T* src;
    T* dst;
    int lr, ch;
    if (it < items && item_ptrs(it, src, dst, lr, ch)) {
      pr1[k] = *reinterpret_cast<const uint4*>(src + ch * VEC);
      pr2[k] = *reinterpret_cast<const uint4*>(src + HALF + ch * VEC);
    }
  }
  const bool table = batch <= kRopeThreads;
  if (table && threadIdx.x < batch) s_seq[threadIdx.x] = seqs[threadIdx.x];
  __syncthreads();
  if (threadIdx.x < ROWS) {
    const int row = row0 + threadIdx.x;
    int pos = -1;
    if (row < total_rows) {
      int b = -1;
      if (table) {
        int lo = 0, hi = batch - 1;
        while (lo <= hi) {
          const int mid = (lo + hi) >> 1;
          if (s_seq[mid].q_off <= row) { b = mid; lo = mid + 1; } else { hi = mid - 1; }
        }
      } else {
        b = find_seq_by_row(seqs, batch, row);
      }
      if (b >= 0) {
        const ssv_seq sq = table ? s_seq[b] : seqs[b];
        // a sequence outside the rows (or whose positions leave int range) is
        // skipped: its rows are left as they are
        const bool ok = sq.cache_len >= 0 && sq.new_len >= 0 && sq.block >= 1 && sq.block <= 64 &&
                        sq.q_off >= 0 && (long long)sq.q_off + sq.new_len + 2LL * sq.block <= total_rows &&
                        (long long)sq.cache_len + sq.new_len + sq.block <= 0x7fffffffLL;
        const int i = row - sq.q_off;
        if (!ok) {
          report(dev_status, SSV_ERR_INVALID);
        } else if (i < sq.new_len + 2 * sq.block) {
          // the row whose position applies: itself, or for a tail row its data row
          const int k = (i - sq.new_len) % sq.block;
          const int src = (i < sq.new_len) ? row : sq.q_off + sq.new_len + k;
          pos = (i < sq.new_len) ? sq.cache_len + i : sq.cache_len + sq.new_len + k;
          if (positions) {
            pos = positions[src];
            if (pos < 0) {
              report(dev_status, SSV_ERR_INVALID);
              pos = -1;
            }
          }
        }
      }
    }
    s_pos[threadIdx.x] = pos;
  }
  __syncthreads();
  for (int t = threadIdx.x; t < ROWS * HALF; t += blockDim.x) {
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

  auto rotate = [&](int lr, int ch, const float* x1, const float* x2, T* dst) {
    float y1[VEC], y2[VEC];
#pragma unroll
    for (int v = 0; v < VEC; ++v) {
      const float c = s_cos[lr][ch * VEC + v], s = s_sin[lr][ch * VEC + v];
      y1[v] = x1[v] * c - x2[v] * s;
      y2[v] = x2[v] * c + x1[v] * s;
    }
    store16<T>(dst + ch * VEC, y1);
    store16<T>(dst + HALF + ch * VEC, y2);
  };
#pragma unroll
  for (int k = 0; k < PRE; ++k) {
    const int it = threadIdx.x + k * kRopeThreads;
    const T* src;
    T* dst;
    int lr, ch;
    if (it < items && item_ptrs(it, src, dst, lr, ch) && s_pos[lr] >= 0) {
      float x1[VEC], x2[VEC];
      unpack16<T>(pr1[k], x1);
      unpack16<T>(pr2[k], x2);
      rotate(lr, ch, x1, x2, dst);
    }
  }
  for (int it = threadIdx.x + PRE * kRopeThreads; it < items; it += blockDim.x) {
    const T* src;
    T* dst;
    int lr, ch;
    if (!item_ptrs(it, src, dst, lr, ch) || s_pos[lr] < 0) continue;
    float x1[VEC], x2[VEC];
    load16<T>(src + ch * VEC, x1);
    load16<T>(src + HALF + ch * VEC, x2);
    rotate(lr, ch, x1, x2, dst);
  }
}

template <typename T, int D, int ROWS>
static cudaError_t launch_rope_rows(const ssv_rope_args* a, const RopeTheta& th, cudaStream_t st) {
  const int grid = (a->total_rows + ROWS - 1) / ROWS;
  return launch_pdl(rope_copy_kernel<T, D, ROWS>, dim3(grid), dim3(kRopeThreads), 0, st,
                    static_cast<const T*>(a->q_in), static_cast<const T*>(a->k_in), static_cast<T*>(a->q_out),
                    static_cast<T*>(a->k_out), a->Hq, a->Hkv, a->seqs, a->batch, a->total_rows, a->positions,
                    a->dev_status, th);
}

// A small batch (fewer than four rows per SM) gets one row per CTA, so that its
// loads and angles spread over the SMs; a larger one four rows per CTA.
template <typename T, int D>
static cudaError_t launch_rope(const ssv_rope_args* a, const RopeTheta& th, cudaStream_t st) {
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return cudaErrorInvalidDevice;
  if ((long long)a->total_rows < 4LL * sms) return launch_rope_rows<T, D, 1>(a, th, st);
  return launch_rope_rows<T, D, kRopeRows>(a, th, st);
}

}  // namespace ssv

namespace ssv {
ssv_status rope_validate(const ssv_rope_args* a) {
  if (!a) return SSV_ERR_INVALID;
  if (a->total_rows < 0 || a->batch < 0 || a->Hq <= 0 || a->Hkv <= 0) return SSV_ERR_INVALID;
  if (a->total_rows == 0 || a->batch == 0) return SSV_OK;
  if (!a->q_in || !a->k_in || !a->q_out || !a->k_out || !a->seqs) return SSV_ERR_INVALID;
  if (a->d != 64 && a->d != 128) return SSV_ERR_UNSUPPORTED;
  if (a->dtype != SSV_F32 && a->dtype != SSV_BF16) return SSV_ERR_INVALID;
  if (!(a->base > 1.0) || !isfinite(a->base)) return SSV_ERR_INVALID;
  const uintptr_t al = (uintptr_t)a->q_in | (uintptr_t)a->k_in | (uintptr_t)a->q_out | (uintptr_t)a->k_out;
  if (al & 15u) return SSV_ERR_INVALID;
  return SSV_OK;
}
}  // namespace ssv

extern "C" ssv_status ssv_rope_copy(const ssv_rope_args* a, void* stream) {
  using namespace ssv;
  const ssv_status v = rope_validate(a);
  if (v != SSV_OK) return v;
  if (a->total_rows == 0 || a->batch == 0) return SSV_OK;
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
