// Tensor-core verify attention (bf16 in, fp32 accumulate, head_dim 128).
//
// SimSD summary, section 2 "Temporal Attention Mask" and section 4
// "Verification": one pass of softmax(q K^T * scale) V under the temporal
// mask, which is evaluated per (row, key) from tau on the fly.
//
// Tile = (sequence b, kv head g, R consecutive query rows of b) x all G query
// heads of the group, M = R * G = 128 rows, so one K/V block feeds every
// head that shares it (grouped-query packing).  Row m of the tile is
// (query row row0 + m / G, head g * G + m % G); the Q box of the TMA tensor
// map (64 x G x R elements) lands in exactly that order.
//
// Per CTA (192 threads, one CTA per SM: 226 KB of shared memory):
//   warp 0      TMA producer (Q once, then K/V blocks into a 2-stage ring)
//               and TMEM allocator (512 columns: S double buffer + O)
//   warp 1      MMA issuer: S_j = Q K_j^T (M=128, N=128, K=128) into TMEM,
//               then O += P_{j-1} V_{j-1} (P from shared memory, V MN-major)
//   warps 2..5  softmax: tcgen05.ld of S rows (thread = row = TMEM lane),
//               mask, online max with lazy rescaling (only when the max
//               grows by more than 2^8), exp2, bf16 P into swizzled shared
//               memory; epilogue O / l from TMEM to global.
// Key blocks: the sequence's cache keys (all visible to every row), then its
// fresh keys (prompt rows causal, tail rows per tau).  Blocks whose 128 keys
// are visible to every valid row of the tile skip the mask.
#include "ssv_internal.cuh"
#include "attn.cuh"
#include "tc_ptx.cuh"

#include <cuda.h>
#include <cudaTypedefs.h>
#include <math.h>
#include <mutex>

namespace ssv {
namespace tc {

using namespace ptx;

constexpr int D = 128;
constexpr int BM = 128;        // query rows per tile (M)
constexpr int BN = 128;        // keys per block
constexpr int NST = 2;         // K/V pipeline stages
constexpr int kThreads = 192;
constexpr uint32_t TILE_BYTES = 128 * 128 * 2;  // one 128 x 128 bf16 operand
constexpr uint32_t HALF_BYTES = TILE_BYTES / 2;  // one 64-column swizzle atom column (16 KB)
constexpr uint32_t SM_Q = 0;
constexpr uint32_t SM_K = SM_Q + TILE_BYTES;
constexpr uint32_t SM_V = SM_K + NST * TILE_BYTES;
constexpr uint32_t SM_P = SM_V + NST * TILE_BYTES;
constexpr uint32_t SM_BAR = SM_P + 2 * TILE_BYTES;
constexpr uint32_t SM_TOTAL = SM_BAR + 256;
constexpr uint32_t SM_ALLOC = SM_TOTAL + 1024;  // base is rounded up to 1024 B
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t TM_S = 0;    // S double buffer: columns [0, 256)
constexpr uint32_t TM_O = 256;  // O: columns [256, 384)
constexpr float kRescaleThreshold = 8.0f;  // log2 units

// barrier slots (8 bytes each) inside SM_BAR
enum : uint32_t {
  B_Q = 0,
  B_KV_FULL = 1,   // +stage
  B_KV_EMPTY = 3,  // +stage
  B_S_FULL = 5,    // +buffer
  B_S_FREE = 7,    // +buffer
  B_P_FULL = 9,    // +buffer
  B_PV_DONE = 11,  // +buffer
  B_FINAL = 13,
  B_COUNT = 14
};

struct TcMaps {
  CUtensorMap q, kc, vc, kn, vn;
};

struct TileGeom {
  int C, N, B, q_off, kv_off, tau_off;
  int row0, rows;       // first local query row of the tile, rows of the sequence
  int cache_blocks, nblocks;
  int full_new;         // fresh keys [0, full_new) are visible to every valid row of the tile
};

__device__ __forceinline__ uint32_t bar_addr(uint32_t base, int i) { return base + SM_BAR + 8u * i; }

template <typename OutT>
__global__ void __launch_bounds__(kThreads, 1)
attn_tc_kernel(const __grid_constant__ TcMaps maps, const AttnParams p, int R, int G) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  volatile int* abort = reinterpret_cast<volatile int*>(smem + SM_BAR + 8 * B_COUNT + 4);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + SM_BAR + 8 * B_COUNT);
  __shared__ int s_ok;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int b = blockIdx.z, g = blockIdx.y, tile = blockIdx.x;
  const ssv_seq sq = p.seqs[b];
  TileGeom t;
  t.C = sq.cache_len; t.N = sq.new_len; t.B = sq.block;
  t.q_off = sq.q_off; t.kv_off = sq.kv_off; t.tau_off = sq.tau_off;
  t.rows = t.N + 2 * t.B;
  t.row0 = tile * R;
  if (t.row0 >= t.rows) return;  // uniform: this sequence has fewer tiles
  t.cache_blocks = (t.C + BN - 1) / BN;
  const int kmax = (t.row0 + R <= t.N) ? (t.row0 + R) : t.rows;
  t.nblocks = t.cache_blocks + (kmax + BN - 1) / BN;
  t.full_new = (t.row0 < t.N) ? (t.row0 + 1) : t.N;
  const int32_t* tau = p.tau + t.tau_off;

  if (warp == 0) {
    const bool ok = (t.B >= 1 && t.B <= 64) ? warp_tau_is_permutation(tau, t.B) : false;
    if (lane == 0) {
      s_ok = ok;
      *abort = 0;
      for (int i = 0; i < B_COUNT; ++i) {
        uint32_t cnt = 1;
        if (i == B_S_FREE || i == B_S_FREE + 1 || i == B_P_FULL || i == B_P_FULL + 1) cnt = 4;
        mbar_init(bar_addr(sbase, i), cnt);
      }
      fence_mbar_init();
      if (!ok) report(p.dev_status, SSV_ERR_BAD_TAU);
    }
    __syncwarp();
    tmem_alloc(smem_u32(tmem_slot), TMEM_COLS);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const bool ok = s_ok != 0;

  if (ok && warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      tma_prefetch(&maps.q); tma_prefetch(&maps.kc); tma_prefetch(&maps.vc);
      tma_prefetch(&maps.kn); tma_prefetch(&maps.vn);
      const uint32_t bq = bar_addr(sbase, B_Q);
      mbar_expect_tx(bq, TILE_BYTES);
      tma_load_3d(sbase + SM_Q, &maps.q, 0, g * G, t.q_off + t.row0, bq);
      tma_load_3d(sbase + SM_Q + HALF_BYTES, &maps.q, 64, g * G, t.q_off + t.row0, bq);
      int issued = 0;
      for (int j = 0; j < t.nblocks; ++j) {
        const int st = j % NST;
        if (j >= NST && !mbar_wait(bar_addr(sbase, B_KV_EMPTY + st), ((j - NST) / NST) & 1, abort)) break;
        const uint32_t bf = bar_addr(sbase, B_KV_FULL + st);
        mbar_expect_tx(bf, 2 * TILE_BYTES);
        const uint32_t dk = sbase + SM_K + st * TILE_BYTES, dv = sbase + SM_V + st * TILE_BYTES;
        if (j < t.cache_blocks) {
          const int z = t.kv_off + j * BN;
          tma_load_3d(dk, &maps.kc, 0, g, z, bf);
          tma_load_3d(dk + HALF_BYTES, &maps.kc, 64, g, z, bf);
          tma_load_3d(dv, &maps.vc, 0, g, z, bf);
          tma_load_3d(dv + HALF_BYTES, &maps.vc, 64, g, z, bf);
        } else {
          const int z = t.q_off + (j - t.cache_blocks) * BN;
          tma_load_3d(dk, &maps.kn, 0, g, z, bf);
          tma_load_3d(dk + HALF_BYTES, &maps.kn, 64, g, z, bf);
          tma_load_3d(dv, &maps.vn, 0, g, z, bf);
          tma_load_3d(dv + HALF_BYTES, &maps.vn, 64, g, z, bf);
        }
        issued = j + 1;
      }
      // drain: every issued copy must land before the CTA exits (bounded,
      // and regardless of the abort flag)
      {
        const long long t0 = clock64();
        while (!mbar_try_wait(bar_addr(sbase, B_Q), 0) && clock64() - t0 < kWaitBudget) {
        }
      }
      for (int j = (issued > NST ? issued - NST : 0); j < issued; ++j) {
        const int st = j % NST;
        const long long t0 = clock64();
        while (!mbar_try_wait(bar_addr(sbase, B_KV_FULL + st), (j / NST) & 1) && clock64() - t0 < kWaitBudget) {
        }
      }
    }
  } else if (ok && warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t id_s = idesc_bf16(128, 128, false);
      const uint32_t id_pv = idesc_bf16(128, 128, true);
      bool run = mbar_wait(bar_addr(sbase, B_Q), 0, abort);
      auto issue_pv = [&](int jj) -> bool {
        const int sb = jj & 1, st = jj % NST;
        if (!mbar_wait(bar_addr(sbase, B_P_FULL + sb), (jj >> 1) & 1, abort)) return false;
        tc_fence_after();
        const uint32_t pa = sbase + SM_P + sb * TILE_BYTES, va = sbase + SM_V + st * TILE_BYTES;
#pragma unroll
        for (int k = 0; k < BN / 16; ++k) {
          const uint64_t ad = smem_desc_sw128(pa + (k >> 2) * HALF_BYTES + (k & 3) * 32, 16, 1024);
          const uint64_t bd = smem_desc_sw128(va + k * 2048, HALF_BYTES, 1024);
          mma_f16(tmem + TM_O, ad, bd, id_pv, (jj > 0 || k > 0) ? 1u : 0u);
        }
        mma_commit(bar_addr(sbase, B_PV_DONE + sb));
        mma_commit(bar_addr(sbase, B_KV_EMPTY + st));
        return true;
      };
      for (int j = 0; run && j < t.nblocks; ++j) {
        const int st = j % NST, sb = j & 1;
        if (!mbar_wait(bar_addr(sbase, B_KV_FULL + st), (j / NST) & 1, abort)) { run = false; break; }
        if (j >= 2 && !mbar_wait(bar_addr(sbase, B_S_FREE + sb), ((j - 2) >> 1) & 1, abort)) { run = false; break; }
        tc_fence_after();
        const uint32_t ka = sbase + SM_K + st * TILE_BYTES;
#pragma unroll
        for (int k = 0; k < D / 16; ++k) {
          const uint32_t off = (k >> 2) * HALF_BYTES + (k & 3) * 32;
          const uint64_t ad = smem_desc_sw128(sbase + SM_Q + off, 16, 1024);
          const uint64_t bd = smem_desc_sw128(ka + off, 16, 1024);
          mma_f16(tmem + TM_S + sb * 128, ad, bd, id_s, k > 0 ? 1u : 0u);
        }
        mma_commit(bar_addr(sbase, B_S_FULL + sb));
        if (j >= 1 && !issue_pv(j - 1)) { run = false; break; }
      }
      if (run) issue_pv(t.nblocks - 1);
      // all MMAs issued by this thread complete before TMEM is released
      mma_commit(bar_addr(sbase, B_FINAL));
      const long long t0 = clock64();
      while (!mbar_try_wait(bar_addr(sbase, B_FINAL), 0) && clock64() - t0 < kWaitBudget) {
      }
    }
  } else if (ok) {
    // ------------------------------------------------------------ softmax
    const int q4 = warp & 3;                 // TMEM lane quadrant of this warp
    const int m = q4 * 32 + lane;            // tile row = TMEM lane
    const int r_local = m / G, hj = m % G;
    const int i = t.row0 + r_local;          // local query row
    const bool valid = i < t.rows;
    const bool prompt = i < t.N;
    const int r = i - t.N;                   // tail row index
    // allowed tail keys of this row: bit tk of (tm0 | tm1 << 32 | ...), 2B <= 128
    uint32_t tm0 = 0u, tm1 = 0u, tm2 = 0u, tm3 = 0u;
    if (valid && !prompt) {
      const int tr = tau[r % t.B];
      for (int tk = 0; tk < 2 * t.B; ++tk) {
        if (!tail_allowed(r, tk, t.B, tr, tau[tk % t.B])) continue;
        const uint32_t bit = 1u << (tk & 31);
        if (tk < 32) tm0 |= bit; else if (tk < 64) tm1 |= bit; else if (tk < 96) tm2 |= bit; else tm3 |= bit;
      }
    }
    const float qk_scale = p.scale * 1.4426950408889634f;
    const uint32_t lane_base = static_cast<uint32_t>(q4 * 32) << 16;
    float m_used = -INFINITY, l_sum = 0.f;
    bool run = true;
    // every thread waits (bounded); the warp proceeds only if all succeeded,
    // so the warp-collective tcgen05.ld / st below are never split
    auto warp_wait = [&](uint32_t bar, uint32_t parity) -> bool {
      const bool w = mbar_wait(bar, parity, abort);
      return __all_sync(0xffffffffu, w);
    };
    for (int j = 0; j < t.nblocks; ++j) {
      const int sb = j & 1;
      if (!warp_wait(bar_addr(sbase, B_S_FULL + sb), (j >> 1) & 1)) { run = false; break; }
      tc_fence_after();
      float s[BN];
      {
        uint32_t sr[BN];
#pragma unroll
        for (int c = 0; c < BN / 32; ++c) tmem_ld32(tmem + lane_base + TM_S + sb * 128 + c * 32, sr + c * 32);
        tmem_wait_ld();
#pragma unroll
        for (int c = 0; c < BN; ++c) s[c] = __uint_as_float(sr[c]);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_addr(sbase, B_S_FREE + sb));
      // ---- mask + scale
      const bool is_cache = j < t.cache_blocks;
      const int kbase = is_cache ? j * BN : (j - t.cache_blocks) * BN;
      const bool full = is_cache ? (kbase + BN <= t.C) : (kbase + BN <= t.full_new);
      float mx = -INFINITY;
      if (full && valid) {
#pragma unroll
        for (int c = 0; c < BN; ++c) { s[c] *= qk_scale; mx = fmaxf(mx, s[c]); }
      } else {
#pragma unroll
        for (int c = 0; c < BN; ++c) {
          const int kk = kbase + c;
          bool al;
          if (!valid) al = false;
          else if (is_cache) al = kk < t.C;
          else if (kk >= t.rows) al = false;
          else if (prompt) al = kk <= i;
          else if (kk < t.N) al = true;
          else {
            const int tk = kk - t.N;
            const uint32_t wsel = tk < 64 ? (tk < 32 ? tm0 : tm1) : (tk < 96 ? tm2 : tm3);
            al = (wsel >> (tk & 31)) & 1u;
          }
          s[c] = al ? s[c] * qk_scale : -INFINITY;
          mx = fmaxf(mx, s[c]);
        }
      }
      // ---- online max with lazy rescale of O (warp-uniform: tcgen05.ld/st are collective)
      const bool need = mx > m_used + kRescaleThreshold || (m_used == -INFINITY && mx > -INFINITY);
      if (j > 0 && __any_sync(0xffffffffu, need)) {
        // O holds PV of blocks < j; it must be complete before rescaling
        if (!warp_wait(bar_addr(sbase, B_PV_DONE + ((j - 1) & 1)), ((j - 1) >> 1) & 1)) { run = false; break; }
        tc_fence_after();
        const float f = need ? exp2f(m_used - mx) : 1.f;
        uint32_t raw[32];
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
          tmem_ld32(tmem + lane_base + TM_O + c * 32, raw);
          tmem_wait_ld();
#pragma unroll
          for (int e = 0; e < 32; ++e) raw[e] = __float_as_uint(__uint_as_float(raw[e]) * f);
          tmem_st32(tmem + lane_base + TM_O + c * 32, raw);
        }
        tmem_wait_st();
        l_sum *= f;
      }
      if (need) m_used = mx;
      // ---- P = exp2(s - m), bf16, into the swizzled P buffer
      if (j >= 2 && !warp_wait(bar_addr(sbase, B_PV_DONE + sb), ((j - 2) >> 1) & 1)) { run = false; break; }
      const float mref = (m_used == -INFINITY) ? 0.f : m_used;
      uint8_t* pbuf = smem + SM_P + sb * TILE_BYTES;
#pragma unroll
      for (int c8 = 0; c8 < BN / 8; ++c8) {
        uint32_t w[4];
#pragma unroll
        for (int h = 0; h < 4; ++h) {
          const float p0 = exp2f(s[c8 * 8 + 2 * h] - mref);
          const float p1 = exp2f(s[c8 * 8 + 2 * h + 1] - mref);
          const __nv_bfloat16 b0 = __float2bfloat16_rn(p0), b1 = __float2bfloat16_rn(p1);
          l_sum += __bfloat162float(b0) + __bfloat162float(b1);
          w[h] = static_cast<uint32_t>(__bfloat16_as_ushort(b0)) | (static_cast<uint32_t>(__bfloat16_as_ushort(b1)) << 16);
        }
        const int atom = c8 >> 3, chunk = c8 & 7;
        uint8_t* dst = pbuf + atom * HALF_BYTES + (m >> 3) * 1024 + (m & 7) * 128 + ((chunk ^ (m & 7)) << 4);
        *reinterpret_cast<uint4*>(dst) = make_uint4(w[0], w[1], w[2], w[3]);
      }
      fence_proxy_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_addr(sbase, B_P_FULL + sb));
    }
    // ---- epilogue
    if (run && warp_wait(bar_addr(sbase, B_PV_DONE + ((t.nblocks - 1) & 1)), ((t.nblocks - 1) >> 1) & 1)) {
      tc_fence_after();
      const float inv = (l_sum > 0.f) ? 1.f / l_sum : 0.f;
      OutT* orow = static_cast<OutT*>(p.o) + ((size_t)(t.q_off + i) * p.Hq + g * G + hj) * D;
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        uint32_t raw[32];
        tmem_ld32(tmem + lane_base + TM_O + c * 32, raw);
        tmem_wait_ld();
        if (valid) {
          if constexpr (sizeof(OutT) == 4) {
#pragma unroll
            for (int e = 0; e < 32; e += 4)
              *reinterpret_cast<float4*>(orow + c * 32 + e) =
                  make_float4(__uint_as_float(raw[e]) * inv, __uint_as_float(raw[e + 1]) * inv,
                              __uint_as_float(raw[e + 2]) * inv, __uint_as_float(raw[e + 3]) * inv);
          } else {
#pragma unroll
            for (int e = 0; e < 32; e += 8) {
              uint32_t w[4];
#pragma unroll
              for (int h = 0; h < 4; ++h) {
                const __nv_bfloat16 b0 = __float2bfloat16_rn(__uint_as_float(raw[e + 2 * h]) * inv);
                const __nv_bfloat16 b1 = __float2bfloat16_rn(__uint_as_float(raw[e + 2 * h + 1]) * inv);
                w[h] = static_cast<uint32_t>(__bfloat16_as_ushort(b0)) |
                       (static_cast<uint32_t>(__bfloat16_as_ushort(b1)) << 16);
              }
              *reinterpret_cast<uint4*>(orow + c * 32 + e) = make_uint4(w[0], w[1], w[2], w[3]);
            }
          }
        }
      }
    }
  }
  // ---------------------------------------------------------------- teardown
  tc_fence_before();
  __syncthreads();
  if (ok && *abort && threadIdx.x == 0) report(p.dev_status, SSV_ERR_TIMEOUT);
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, TMEM_COLS);
  }
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------
static PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  });
  return fn;
}

// 3-D map over a [rows, heads, 128] bf16 tensor: dims (128, heads, rows),
// box (64, box_heads, box_rows), 128-byte swizzle.
static bool encode_3d(CUtensorMap* m, const void* base, int heads, long long rows, int box_heads, int box_rows) {
  auto fn = encode_fn();
  if (!fn || rows <= 0) return false;
  cuuint64_t dims[3] = {128, (cuuint64_t)heads, (cuuint64_t)rows};
  cuuint64_t strides[2] = {128 * 2, (cuuint64_t)heads * 128 * 2};
  cuuint32_t box[3] = {64, (cuuint32_t)box_heads, (cuuint32_t)box_rows};
  cuuint32_t es[3] = {1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool attn_tc_supported(const AttnParams& p) {
  if (p.in_dtype != SSV_BF16 || p.d != D) return false;
  const int G = p.Hq / p.Hkv;
  if (G < 1 || G > 128 || (128 % G) != 0) return false;
  if (p.max_block > 64) return false;
  return encode_fn() != nullptr;
}

template <typename OutT>
static cudaError_t launch_t(const AttnParams& p, const TcMaps& maps, int R, int G, dim3 grid, cudaStream_t st) {
  static std::once_flag once;
  static cudaError_t attr_err = cudaSuccess;
  std::call_once(once, [] {
    attr_err = cudaFuncSetAttribute(attn_tc_kernel<OutT>, cudaFuncAttributeMaxDynamicSharedMemorySize, SM_ALLOC);
  });
  if (attr_err != cudaSuccess) return attr_err;
  attn_tc_kernel<OutT><<<grid, kThreads, SM_ALLOC, st>>>(maps, p, R, G);
  return cudaGetLastError();
}

cudaError_t launch_attn_tc(const AttnParams& p, cudaStream_t st) {
  const int G = p.Hq / p.Hkv;
  const int R = BM / G;
  TcMaps maps;
  if (!encode_3d(&maps.q, p.q, p.Hq, p.total_rows, G, R)) return cudaErrorInvalidValue;
  if (!encode_3d(&maps.kn, p.k_new, p.Hkv, p.total_rows, 1, BN)) return cudaErrorInvalidValue;
  if (!encode_3d(&maps.vn, p.v_new, p.Hkv, p.total_rows, 1, BN)) return cudaErrorInvalidValue;
  if (p.total_cache > 0) {
    if (!encode_3d(&maps.kc, p.k_cache, p.Hkv, p.total_cache, 1, BN)) return cudaErrorInvalidValue;
    if (!encode_3d(&maps.vc, p.v_cache, p.Hkv, p.total_cache, 1, BN)) return cudaErrorInvalidValue;
  } else {
    maps.kc = maps.kn;  // never read: every sequence has C = 0
    maps.vc = maps.vn;
  }
  const int max_rows = p.max_new + 2 * p.max_block;
  dim3 grid((max_rows + R - 1) / R, p.Hkv, p.batch);
  if (p.out_dtype == SSV_F32) return launch_t<float>(p, maps, R, G, grid, st);
  return launch_t<__nv_bfloat16>(p, maps, R, G, grid, st);
}

}  // namespace tc
}  // namespace ssv
