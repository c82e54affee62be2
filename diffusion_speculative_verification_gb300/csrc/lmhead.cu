// LM head over the mask slots fused with acceptance (ssv_lmhead_accept).
//
// SimSD summary, section 4 "Speculative decoding pipeline": the target scores
// every drafted position in one pass and acceptance walks the stages in the
// temporal order the draft induces.  SPOT review, section "How it is used":
// state equality (greedy) and the coupled-noise match argmax(l/T + G[pos]).
// Reading: the logits of mask slot k are l_k = W h_k (W the LM head).  This
// kernel forms l = H W^T on the tensor cores and takes the decision of every
// verified row in the epilogue, so no logits row ever reaches memory.
//
// Rows.  A gather kernel first lists the slots whose rows the acceptance
// reads (stage <= min(gamma + 1, B)) in slot order and, unless that is every
// slot, copies their hidden states into the workspace, so no tensor-core work
// is spent on unverified stages.  The GEMM kernel counts the same rows
// itself; it waits for the gather only when the rows were compacted.
//
// Work split.  The n verified rows form Mt = ceil(n / 128) M-tiles; the
// vocabulary is cut into 256-column pieces (the last one narrower when 256
// does not divide V) and the pieces into G contiguous ranges, G = min(SMs /
// Mt, pieces).  CTA c = g * Mt + m computes tile m over range g.  The Mt CTAs
// of a range are adjacent in launch order and stream the same LM-head tiles
// side by side, so each tile is read from HBM once and from L2 by the others.
// Roles (192 threads, one CTA per SM):
//   warp 0      TMA producer: per (piece, 64-wide K chunk) the A chunk (128
//               hidden-state rows) and the B chunk (the piece's LM-head rows)
//               into a 4-stage ring, 128-byte swizzle;
//   warp 1      TMEM owner (two 256-column fp32 accumulators) and MMA issuer
//               (M = 128, N = piece width, K = 16 per instruction);
//   warps 2-5   epilogue, thread = row = TMEM lane: decision score per column
//               (l, or fl(fl(l / T) + G[row][v]); the noise of the next piece is
//               prefetched into L2 and that of the next 32 columns into
//               registers), running first-argmax over
//               the CTA's range, folded at the end into the row's best key
//               with one 64-bit atomic maximum (key: the score's order-
//               preserving bits above the complemented index, so equal scores
//               go to the lowest index).
// Completion: an arrival counter per M-tile; the CTA that brings the tile's
// last range reads each row's key (thread per row), writes the row results,
// counts verified rows per sequence, and the warp holding a sequence's last
// row walks its stages (the walk ssv_accept uses).  No CTA waits for another; every mbarrier wait is bounded
// and an expired wait ends the CTA with SSV_ERR_TIMEOUT after draining its
// own copies and MMAs.
#include "accept.cuh"
#include "tc_ptx.cuh"

#include <cuda.h>
#include <cudaTypedefs.h>
#include <math.h>
#include <algorithm>
#include <mutex>

namespace ssv {
namespace {

using namespace ptx;

constexpr int kLmThreads = 192;
constexpr int kLmStages = 4;
constexpr int kLmMaxSlots = 2048;
constexpr int kGatherThreads = 256;
constexpr int kGatherPer = kLmMaxSlots / kGatherThreads;  // slots per thread in the listing
constexpr int kLmMaxBatch = 2048;
constexpr uint32_t kLmABytes = 128u * 128u;  // 128 rows x 64 bf16
constexpr uint32_t kLmBBytes = 256u * 128u;  // 256 rows x 64 bf16
constexpr uint32_t kLmTmemCols = 512;        // two 256-column accumulators

enum : int {
  LB_FULL = 0,
  LB_EMPTY = LB_FULL + kLmStages,
  LB_ACCF = LB_EMPTY + kLmStages,  // accumulator buffer ready for the epilogue
  LB_ACCE = LB_ACCF + 2,           // accumulator buffer drained by the 4 epilogue warps
  LB_FIN = LB_ACCE + 2,            // every MMA issued has completed
  LB_COUNT = LB_FIN + 1
};

constexpr uint32_t SM_A = 0;
constexpr uint32_t SM_B = SM_A + kLmStages * kLmABytes;
constexpr uint32_t SM_BAR = SM_B + kLmStages * kLmBBytes;
constexpr uint32_t SM_MISC = SM_BAR + 8u * LB_COUNT;  // tmem slot, abort flag, tile-complete flag
constexpr uint32_t SM_WALK = (SM_MISC + 16u + 15u) & ~15u;
constexpr uint32_t SM_SEQOF = SM_WALK + 4u * sizeof(WalkSmem);  // u16 per slot: its sequence
constexpr uint32_t SM_NEED = SM_SEQOF + 2u * kLmMaxSlots;         // u8 per sequence: rows it needs
constexpr uint32_t SM_WCNT = SM_NEED + kLmMaxBatch;               // per-warp counts
constexpr uint32_t SM_TOTAL = SM_WCNT + 64u;
constexpr size_t kLmSmem = SM_TOTAL + 1024;  // + alignment slack of the dynamic base
static_assert(kLmSmem <= 227u * 1024u, "shared memory");

struct LmMaps {
  CUtensorMap h;    // compacted hidden states of the verified rows [S, hidden], box 64 x 128
  CUtensorMap h0;   // the caller's hidden states [S, hidden], box 64 x 128 (every slot verified)
  CUtensorMap w;    // LM head [V, hidden], box 64 x 256
  CUtensorMap w64;  // LM head, box 64 x 64 (narrower pieces)
  CUtensorMap w16;  // LM head, box 64 x 16
};

struct LmParams {
  AcceptParams acc;  // metadata, outputs, row results and sequence counters (walk)
  int hidden, nk;    // nk = hidden / 64
  int Mt, V16, NP;     // Mt: M-tiles of the slot count (an upper bound); NP: 256-column pieces
  int use_noise, vec;
  float T;
  const float* noise;
  int n_noise_rows;
  const int32_t* noise_row;
  const __nv_bfloat16* h_src;   // hidden states [S, hidden] (gather input)
  __nv_bfloat16* h_rows;        // [S, hidden]: hidden states of the verified rows, compacted
  int32_t* n_rows;              // [2]: verified rows, 1 if they are every slot (written by the gather)
  int32_t* row_slot;            // [S]: slot of each compacted row
  int32_t* cnt_tile;            // [Mt]
  unsigned long long* rowkey;   // [Mt * 128]: best (score, index) key of each row, 0 = none
  // bounded waits give up after wait_budget SM cycles; fault_skip >= 0 makes
  // CTA 0 leave out that operand stage's copies (test support,
  // ssv_set_fault_injection)
  long long wait_budget;
  int fault_skip;
};

// Order-preserving 32-bit image of a non-NaN float (-0 taken as +0), above
// the complemented index: a larger key is a larger score, or the same score
// at a lower index.
__device__ __forceinline__ unsigned long long score_key(float s, int idx) {
  uint32_t b = __float_as_uint(s == 0.f ? 0.f : s);
  b = (b & 0x80000000u) ? ~b : (b | 0x80000000u);
  return ((unsigned long long)b << 32) | (unsigned long long)(0xFFFFFFFFu - (uint32_t)idx);
}

__device__ __forceinline__ int key_index(unsigned long long k) { return (int)(0xFFFFFFFFu - (uint32_t)k); }

// Vocabulary piece j: first column and width (256, or less for the last
// piece; a multiple of 16 either way).
__device__ __forceinline__ void piece_of(int V16, int j, int& v0, int& w) {
  v0 = 256 * j;
  w = min(256, 16 * V16 - v0);
}

// The noise of columns [v, v + 256) of a row into L2 (eight 128-byte lines).
__device__ __forceinline__ void prefetch_noise_l2(const float* nrow, int v, int V) {
#pragma unroll
  for (int j = 0; j < 256; j += 32)
    if (v + j < V) asm volatile("prefetch.global.L2 [%0];" ::"l"(nrow + v + j));
}

__device__ __forceinline__ void epi_sync() { asm volatile("bar.sync 1, 128;" ::: "memory"); }

// Bounded wait that ignores the abort flag: used to drain a role's own
// asynchronous work before the CTA exits.
__device__ __forceinline__ bool drain_wait(uint32_t bar, uint32_t parity, long long budget) {
  const long long t0 = clock64();
  while (!mbar_try_wait(bar, parity))
    if (clock64() - t0 > budget) return false;
  return true;
}

template <int N>
__device__ __forceinline__ void load_noise(const LmParams& p, const float* nrow, int v, float* gn) {
#pragma unroll
  for (int j = 0; j < N; ++j) gn[j] = 0.f;
  if (!nrow) return;
  if (p.vec) {
#pragma unroll
    for (int j = 0; j < N; j += 4) {
      if (v + j < p.acc.V) {  // V % 4 == 0: a group lies wholly inside or outside
        const float4 t = __ldg(reinterpret_cast<const float4*>(nrow + v + j));
        gn[j] = t.x; gn[j + 1] = t.y; gn[j + 2] = t.z; gn[j + 3] = t.w;
      }
    }
  } else {
#pragma unroll
    for (int j = 0; j < N; ++j)
      if (v + j < p.acc.V) gn[j] = __ldg(nrow + v + j);
  }
}

// Decision scores of N columns (N = 32 or 16) starting at vocabulary index v
// (a multiple of 16), folded into the running first-argmax (best, bi); gn
// holds their noise (coupled noise only).  The TMEM load is warp-wide; rows
// that need no decision (padding, unverified stages) skip the arithmetic.
template <int MODE, int N>
__device__ __forceinline__ void lm_columns(const LmParams& p, uint32_t taddr, int v, const float* gn, bool live,
                                           float& best, int& bi) {
  uint32_t x[N];
  if (N == 32) tmem_ld32(taddr, x); else tmem_ld16(taddr, x);
  tmem_wait_ld();
  if (!live) return;
#pragma unroll
  for (int j = 0; j < N; ++j) {
    float s = __uint_as_float(x[j]);
    if (MODE == SSV_ACCEPT_GUMBEL) s = __fadd_rn(__fdiv_rn(s, p.T), gn[j]);
    if (v + j < p.acc.V && s > best) {
      best = s;
      bi = v + j;
    }
  }
}

// Sequence of every slot (0xFFFF: none) and rows each sequence needs (0: sizes
// rejected), for the listing below.  Called by every thread of the CTA.
__device__ __forceinline__ void seq_tables(const AcceptParams& a, unsigned short* seq_of, unsigned char* need_s) {
  for (int i = threadIdx.x; i < kLmMaxSlots; i += blockDim.x) seq_of[i] = 0xFFFFu;
  __syncthreads();
  for (int b = threadIdx.x; b < a.batch; b += blockDim.x) {
    const int off = a.slot_off[b], B = a.block[b], g = a.gamma[b];
    const bool ok = off >= 0 && B >= 1 && B <= 64 && g >= 0 && g <= B && off + B <= a.total_slots;
    need_s[b] = ok ? (unsigned char)min(g + 1, B) : 0;
    if (ok)
      for (int j = 0; j < B; ++j) seq_of[off + j] = (unsigned short)b;
  }
  __syncthreads();
}

// Whether slot is listed: inside its sequence's sane extent, stage in 1..need.
__device__ __forceinline__ int listed(const AcceptParams& a, const unsigned short* seq_of,
                                      const unsigned char* need_s, int slot) {
  if (slot >= a.total_slots || seq_of[slot] == 0xFFFFu) return 0;
  const int st = a.tau[slot];
  return (st >= 1 && st <= need_s[seq_of[slot]]) ? 1 : 0;
}

// Lists the verified slots in slot order (every CTA builds the same list;
// CTA 0 publishes it) and copies their hidden-state rows, one warp per row,
// rows dealt to CTAs in turn.  A slot is listed when it lies inside its
// sequence's sane extent and its stage is in 1..min(gamma + 1, B); the GEMM
// epilogue still checks the whole sequence before using a row (and reports
// the sequences it rejects).
__global__ void __launch_bounds__(kGatherThreads) lmhead_gather_kernel(const LmParams p) {
  __shared__ int32_t list[kLmMaxSlots];
  __shared__ unsigned short seq_of[kLmMaxSlots];
  __shared__ unsigned char need_s[kLmMaxBatch];
  __shared__ int32_t wsum[kGatherThreads / 32];
  pdl_wait();  // hidden states and metadata may come from the kernels before this one
  pdl_trigger();  // the GEMM may set up; it reads nothing of ours before its own wait
  const AcceptParams& a = p.acc;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  seq_tables(a, seq_of, need_s);
  int flag[kGatherPer];
  int cnt = 0;
#pragma unroll
  for (int i = 0; i < kGatherPer; ++i) {
    flag[i] = listed(a, seq_of, need_s, tid * kGatherPer + i);
    cnt += flag[i];
  }
  // exclusive scan of the per-thread counts (slot order = thread order)
  int incl = cnt;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) wsum[warp] = incl;
  __syncthreads();
  int before = 0, total = 0;
#pragma unroll
  for (int w = 0; w < kGatherThreads / 32; ++w) {
    before += (w < warp) ? wsum[w] : 0;
    total += wsum[w];
  }
  int pos = before + incl - cnt;
#pragma unroll
  for (int i = 0; i < kGatherPer; ++i)
    if (flag[i]) list[pos++] = tid * kGatherPer + i;
  __syncthreads();
  const bool identity = total == a.total_slots;  // then list[i] == i
  if (blockIdx.x == 0) {
    if (!identity)
      for (int i = tid; i < total; i += kGatherThreads) p.row_slot[i] = list[i];
    if (tid == 0) {
      p.n_rows[0] = total;
      p.n_rows[1] = identity ? 1 : 0;
    }
  }
  if (identity) return;  // the GEMM reads the caller's rows directly
  // copy: row i by CTA i mod gridDim, warp (i / gridDim) mod 8, 16-byte vectors,
  // eight loads in flight per lane before their stores
  const size_t row_vec = (size_t)p.hidden / 8;  // 16-byte vectors per row
  const int nw = kGatherThreads / 32;
  for (int i = blockIdx.x + gridDim.x * warp; i < total; i += gridDim.x * nw) {
    const uint4* src = reinterpret_cast<const uint4*>(p.h_src) + (size_t)list[i] * row_vec;
    uint4* dst = reinterpret_cast<uint4*>(p.h_rows) + (size_t)i * row_vec;
    for (size_t e0 = lane; e0 < row_vec; e0 += 32 * 8) {
      uint4 v[8];
#pragma unroll
      for (int t = 0; t < 8; ++t)
        if (e0 + 32 * t < row_vec) v[t] = __ldg(src + e0 + 32 * t);
#pragma unroll
      for (int t = 0; t < 8; ++t)
        if (e0 + 32 * t < row_vec) dst[e0 + 32 * t] = v[t];
    }
  }
}

template <int MODE>
__global__ void __launch_bounds__(kLmThreads, 1)
lmhead_accept_kernel(const __grid_constant__ LmMaps maps, const LmParams p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  auto bar = [&](int i) -> uint32_t { return sbase + SM_BAR + 8u * (uint32_t)i; };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + SM_MISC);
  volatile int* abort = reinterpret_cast<volatile int*>(smem + SM_MISC + 4);
  volatile int* tile_done = reinterpret_cast<volatile int*>(smem + SM_MISC + 8);
  WalkSmem* walk = reinterpret_cast<WalkSmem*>(smem + SM_WALK);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    *abort = 0;
    *tile_done = 0;
    for (int i = 0; i < LB_COUNT; ++i) mbar_init(bar(i), (i == LB_ACCE || i == LB_ACCE + 1) ? 4u : 1u);
    fence_mbar_init();
    tma_prefetch(&maps.h);
    tma_prefetch(&maps.h0);
    tma_prefetch(&maps.w);
    tma_prefetch(&maps.w64);
    tma_prefetch(&maps.w16);
  }
  if (warp == 1) tmem_alloc(smem_u32(tmem_slot), kLmTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // Count the verified rows here (the gather kernel reaches the same count):
  // as the second kernel of the call this one may read the call's inputs
  // before its wait, since the gather lets it start only after its own wait.
  // When every slot is verified the rows are read from the caller's hidden
  // states and nothing of the gather's is needed: the wait moves to the end.
  int n_rows;
  {
    unsigned short* seq_of = reinterpret_cast<unsigned short*>(smem + SM_SEQOF);
    unsigned char* need_s = smem + SM_NEED;
    int* wcnt = reinterpret_cast<int*>(smem + SM_WCNT);
    seq_tables(p.acc, seq_of, need_s);
    int c = 0;
    for (int slot = threadIdx.x; slot < p.acc.total_slots; slot += blockDim.x) c += listed(p.acc, seq_of, need_s, slot);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) c += __shfl_xor_sync(0xffffffffu, c, o);
    if (lane == 0) wcnt[warp] = c;
    __syncthreads();
    n_rows = 0;
    for (int w = 0; w < kLmThreads / 32; ++w) n_rows += wcnt[w];
  }
  const bool identity = n_rows == p.acc.total_slots;
  if (!identity) {
    pdl_wait();  // the compacted rows (and, through the gather, every kernel before)
    pdl_trigger();
  }
  // tiles of the verified rows and this CTA's (tile, range); CTAs past the
  // last (tile, range) pair have no work
  const CUtensorMap* hmap = identity ? &maps.h0 : &maps.h;
  const int Mt = (n_rows + 127) / 128;
  const int G = Mt > 0 ? min((int)gridDim.x / Mt, p.NP) : 0;
  const bool active = (int)blockIdx.x < G * Mt;
  const int m = active ? (int)blockIdx.x % Mt : 0, g = active ? (int)blockIdx.x / Mt : 0;
  const int j_begin = active ? (int)(((long long)p.NP * g) / G) : 0;
  const int npieces = active ? (int)(((long long)p.NP * (g + 1)) / G) - j_begin : 0;  // pieces of this range

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      int it = 0;
      bool ok = true;
      for (int pc = 0; pc < npieces && ok; ++pc) {
        int v0, w;
        piece_of(p.V16, j_begin + pc, v0, w);
        for (int kc = 0; kc < p.nk; ++kc) {
          const int s = it % kLmStages;
          if (it >= kLmStages && !mbar_wait(bar(LB_EMPTY + s), ((it / kLmStages) - 1) & 1, abort, p.wait_budget)) {
            ok = false;
            break;
          }
          const uint32_t fb = bar(LB_FULL + s);
          if (blockIdx.x == 0 && it == p.fault_skip) {  // test support: this stage's copies are left out
            ++it;
            continue;
          }
          mbar_expect_tx(fb, kLmABytes + (uint32_t)w * 128u);
          tma_load_2d(sbase + SM_A + s * kLmABytes, hmap, kc * 64, m * 128, fb);
          const uint32_t bdst = sbase + SM_B + s * kLmBBytes;
          if (w == 256) {
            tma_load_2d(bdst, &maps.w, kc * 64, v0, fb);
          } else {  // 64-row boxes, then 16-row boxes (each lands 1024-byte aligned)
            int j = 0;
            for (; j + 64 <= w; j += 64) tma_load_2d(bdst + (uint32_t)j * 128u, &maps.w64, kc * 64, v0 + j, fb);
            for (; j < w; j += 16) tma_load_2d(bdst + (uint32_t)j * 128u, &maps.w16, kc * 64, v0 + j, fb);
          }
          ++it;
        }
      }
      // every copy issued lands before the CTA exits (the older ones were
      // consumed before their stage was reused)
      for (int j = max(0, it - kLmStages); j < it; ++j) drain_wait(bar(LB_FULL + j % kLmStages), (j / kLmStages) & 1, p.wait_budget);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      int it = 0;
      bool ok = true;
      for (int pc = 0; pc < npieces && ok; ++pc) {
        int v0, w;
        piece_of(p.V16, j_begin + pc, v0, w);
        const int buf = pc & 1;
        if (pc >= 2 && !mbar_wait_poll(bar(LB_ACCE + buf), ((pc >> 1) - 1) & 1, abort, p.wait_budget)) break;
        tc_fence_after();
        const uint32_t d = tmem + (uint32_t)buf * 256u;
        const uint32_t idesc = idesc_bf16(128, (uint32_t)w, false);
        for (int kc = 0; kc < p.nk; ++kc) {
          const int s = it % kLmStages;
          if (!mbar_wait_poll(bar(LB_FULL + s), (it / kLmStages) & 1, abort, p.wait_budget)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t ad = smem_desc_sw128(sbase + SM_A + s * kLmABytes, 16, 1024);
          const uint64_t bd = smem_desc_sw128(sbase + SM_B + s * kLmBBytes, 16, 1024);
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) mma_bf16_ss(d, ad + 2 * kk, bd + 2 * kk, idesc, (kc | kk) != 0);
          mma_commit(bar(LB_EMPTY + s));
          ++it;
        }
        if (ok) mma_commit(bar(LB_ACCF + buf));
      }
      // every MMA issued completes before TMEM is released
      mma_commit(bar(LB_FIN));
      drain_wait(bar(LB_FIN), 0, p.wait_budget);
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;           // TMEM lane quarter of this warp
    const int r = 32 * q + lane;      // row of the tile
    const int et = threadIdx.x - 64;  // 0..127
    const AcceptParams& a = p.acc;
    const int ci = m * 128 + r;  // compacted row
    const int slot = (active && ci < n_rows) ? (identity ? ci : p.row_slot[ci]) : a.total_slots;
    // this row: sequence, stage, and whether it is verified / tested.  A
    // sequence is usable when its sizes are sane, its stage map permutes
    // 1..B and (coupled noise) every verified slot has a table row; every row
    // of the sequence reaches the same answer, whichever CTA holds it.
    int b = -1, off = 0, B = 0, gm = 0;
    bool verified = false, tested = false;
    const float* nrow = nullptr;
    if (slot < a.total_slots) {
      b = find_seq_by_slot(a.slot_off, a.batch, slot);
      if (b >= 0) {
        off = a.slot_off[b];
        B = a.block[b];
        gm = a.gamma[b];
      }
      if (b >= 0 && off >= 0 && B >= 1 && B <= 64 && gm >= 0 && gm <= B && off + B <= a.total_slots &&
          slot < off + B) {
        const int need = min(gm + 1, B);
        unsigned long long seen = 0ull;
        bool perm = true, noise_ok = true;
#pragma unroll 8
        for (int j = 0; j < B; ++j) {
          const int t = a.tau[off + j];
          if (t < 1 || t > B) perm = false; else seen |= 1ull << (t - 1);
          if (p.use_noise && t >= 1 && t <= need) {
            const int nr = p.noise_row[off + j];
            if (nr < 0 || nr >= p.n_noise_rows) noise_ok = false;
          }
        }
        perm = perm && seen == ((B >= 64) ? ~0ull : ((1ull << B) - 1ull));
        const int st = a.tau[slot];
        verified = perm && noise_ok && st <= need;
        tested = st <= gm;
        if (verified && p.use_noise) nrow = p.noise + (size_t)p.noise_row[slot] * (size_t)a.V;
      } else {
        b = -1;
      }
    }
    // rejected sequences, reported once: sequence b by CTA b mod gridDim, epilogue
    // warp (b / gridDim) mod 4 (runs while the first piece is multiplied)
    for (int sb = blockIdx.x + gridDim.x * q; sb < a.batch; sb += gridDim.x * 4) {
      const int soff = a.slot_off[sb], sB = a.block[sb], sg = a.gamma[sb];
      if (!(soff >= 0 && sB >= 1 && sB <= 64 && sg >= 0 && sg <= sB && soff + sB <= a.total_slots)) {
        if (lane == 0) report(a.dev_status, SSV_ERR_BAD_TAU);
        continue;
      }
      if (!warp_tau_is_permutation(a.tau + soff, sB)) {
        if (lane == 0) report(a.dev_status, SSV_ERR_BAD_TAU);
        continue;
      }
      bool bad_row = false;
      if (p.use_noise)
        for (int j = lane; j < sB; j += 32)
          if (a.tau[soff + j] <= min(sg + 1, sB)) {
            const int nr = p.noise_row[soff + j];
            bad_row = bad_row || nr < 0 || nr >= p.n_noise_rows;
          }
      if (__any_sync(0xffffffffu, bad_row) && lane == 0) report(a.dev_status, SSV_ERR_INVALID);
    }
    // running first-argmax over the pieces of this CTA's range
    float best = -INFINITY;
    int bi = INT_MAX;
    bool ok = true;
    if (MODE == SSV_ACCEPT_GUMBEL && nrow && npieces > 0) prefetch_noise_l2(nrow, 256 * j_begin, a.V);
    for (int pc = 0; pc < npieces; ++pc) {
      int v0, w;
      piece_of(p.V16, j_begin + pc, v0, w);
      const int buf = pc & 1;
      float gn[2][32];
      if (MODE == SSV_ACCEPT_GUMBEL) {
        if (nrow && pc + 1 < npieces) prefetch_noise_l2(nrow, v0 + 256, a.V);
        load_noise<32>(p, nrow, v0, gn[0]);
      }
      // warp-uniform: a lane that saw the phase complete while another gave up
      // must not go on to the warp-collective TMEM loads alone
      if (!__all_sync(0xffffffffu, mbar_wait(bar(LB_ACCF + buf), (pc >> 1) & 1, abort, p.wait_budget))) {
        ok = false;
        break;
      }
      tc_fence_after();
      const uint32_t ta = tmem + ((uint32_t)(32 * q) << 16) + (uint32_t)buf * 256u;
      int c0 = 0;
#pragma unroll
      for (int k = 0; k < 8; ++k, c0 += 32) {  // 32-column chunks, noise one chunk ahead
        if (c0 + 32 > w) break;
        if (MODE == SSV_ACCEPT_GUMBEL && k < 7 && c0 + 64 <= w) load_noise<32>(p, nrow, v0 + c0 + 32, gn[(k + 1) & 1]);
        lm_columns<MODE, 32>(p, ta + c0, v0 + c0, gn[k & 1], verified, best, bi);
      }
      for (; c0 < w; c0 += 16) {  // a last piece narrower than a multiple of 32
        float g16[16];
        if (MODE == SSV_ACCEPT_GUMBEL) load_noise<16>(p, nrow, v0 + c0, g16);
        lm_columns<MODE, 16>(p, ta + c0, v0 + c0, g16, verified, best, bi);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(LB_ACCE + buf));
    }
    // fold this range's best into the row's key; the CTA that completes the
    // tile reads the keys
    if (active && ok && bi != INT_MAX) atomicMax(p.rowkey + (size_t)m * 128 + r, score_key(best, bi));
    __threadfence();
    epi_sync();
    if (et == 0 && active && ok && !*abort) {
      int prev;
      asm volatile("atom.acq_rel.gpu.global.add.s32 %0, [%1], 1;" : "=r"(prev) : "l"(p.cnt_tile + m) : "memory");
      *tile_done = (prev + 1 == G) ? 1 : 0;
    }
    epi_sync();
    if (*tile_done) {
      asm volatile("fence.acq_rel.gpu;" ::: "memory");
      if (et == 0) p.cnt_tile[m] = 0;
      unsigned long long* kp = p.rowkey + (size_t)m * 128 + r;
      const unsigned long long key = __ldcg(kp);
      *kp = 0ull;  // left zero for the next call
      const int i = key ? key_index(key) : -1;
      bool done = false;
      if (verified) {
        RowResult res;
        res.dec = i;
        res.ok = tested && a.draft_tokens[slot] == i;
        a.rowres[slot] = res;
        const int need = min(gm + 1, B);
        int prev;
        asm volatile("atom.acq_rel.gpu.global.add.s32 %0, [%1], 1;" : "=r"(prev) : "l"(a.cnt_seq + b) : "memory");
        done = prev + 1 == need;
        if (done) a.cnt_seq[b] = 0;  // every row of the sequence has arrived
      }
      unsigned dm = __ballot_sync(0xffffffffu, done);
      while (dm) {
        const int src = __ffs(dm) - 1;
        dm &= dm - 1;
        const int bb = __shfl_sync(0xffffffffu, b, src), oo = __shfl_sync(0xffffffffu, off, src);
        const int BB = __shfl_sync(0xffffffffu, B, src), g2 = __shfl_sync(0xffffffffu, gm, src);
        asm volatile("fence.acq_rel.gpu;" ::: "memory");
        warp_seq_walk<MODE>(a, bb, oo, BB, g2, walk[q], nullptr);
      }
    }
  }
  // ------------------------------------------------------------ teardown
  tc_fence_before();
  __syncthreads();
  if (identity && threadIdx.x == 0) {  // never complete before the gather
    pdl_wait();
    pdl_trigger();
  }
  if (*abort && threadIdx.x == 0) report(p.acc.dev_status, SSV_ERR_TIMEOUT);
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kLmTmemCols);
  }
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------
PFN_cuTensorMapEncodeTiled_v12000 lm_encode_fn() {
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

// 2-D map over a row-major [rows, cols] bf16 matrix: box (64, box_rows),
// 128-byte swizzle, zero fill outside the matrix.
bool encode_rows(CUtensorMap* m, const void* base, long long rows, int cols, int box_rows) {
  auto fn = lm_encode_fn();
  if (!fn || rows <= 0) return false;
  cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)cols * 2};
  cuuint32_t box[2] = {64, (cuuint32_t)box_rows};
  cuuint32_t es[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int lm_sm_count() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  return n;
}

struct LmLayout {
  size_t cnt_tile, cnt_seq, n_rows, row_slot, h_rows, rowkey, rowres, total;
  int Mt, V16, NP;
};

LmLayout lm_layout(const ssv_lmhead_accept_args* a, int nsm) {
  LmLayout L;
  L.Mt = (a->total_slots + 127) / 128;
  L.V16 = (a->V + 15) / 16;
  L.NP = (L.V16 + 15) / 16;
  (void)nsm;
  size_t o = 0;
  L.cnt_tile = o;  o += sizeof(int32_t) * (size_t)L.Mt;  // counters first, contiguous
  L.cnt_seq = o;   o = align_up(o + sizeof(int32_t) * (size_t)a->batch, 256);
  L.n_rows = o;    o = align_up(o + 2 * sizeof(int32_t), 256);                               // written every call
  L.row_slot = o;  o = align_up(o + sizeof(int32_t) * (size_t)a->total_slots, 256);
  L.h_rows = o;    o = align_up(o + 2u * (size_t)a->total_slots * (size_t)a->hidden, 256);
  L.rowkey = o;    o = align_up(o + sizeof(unsigned long long) * (size_t)L.Mt * 128, 256);  // zero between calls
  L.rowres = o;    o = align_up(o + sizeof(RowResult) * (size_t)a->total_slots, 256);
  L.total = o;
  return L;
}

ssv_status lm_check(const ssv_lmhead_accept_args* a) {
  if (!a) return SSV_ERR_INVALID;
  if (a->mode != SSV_ACCEPT_ARGMAX && a->mode != SSV_ACCEPT_GUMBEL) return SSV_ERR_INVALID;
  if (!isfinite(a->T) || a->T < 0.f) return SSV_ERR_NOT_FINITE;
  if (a->V < 1 || a->hidden < 64 || (a->hidden % 64) != 0 || a->batch < 0 || a->total_slots < 0)
    return SSV_ERR_INVALID;
  if (a->total_slots > kLmMaxSlots || a->batch > kLmMaxBatch) return SSV_ERR_UNSUPPORTED;
  if (a->batch == 0 || a->total_slots == 0) return SSV_OK;
  if (!a->hidden_states || !a->lm_head || !a->draft_tokens || !a->tau || !a->block || !a->gamma ||
      !a->slot_off || !a->n_acc || !a->n_out || !a->tokens)
    return SSV_ERR_INVALID;
  if (((uintptr_t)a->hidden_states | (uintptr_t)a->lm_head) & 15u) return SSV_ERR_INVALID;
  if (a->mode == SSV_ACCEPT_GUMBEL && a->T > 0.f) {
    if (!a->noise || !a->noise_row || a->n_noise_rows < 1) return SSV_ERR_INVALID;
    if ((uintptr_t)a->noise & 3u) return SSV_ERR_INVALID;
  }
  return SSV_OK;
}

template <int MODE>
cudaError_t lm_launch(const LmMaps& maps, const LmParams& p, int grid, cudaStream_t st) {
  static std::once_flag once;
  static cudaError_t attr = cudaSuccess;
  std::call_once(once, [] {
    attr = cudaFuncSetAttribute(lmhead_accept_kernel<MODE>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                (int)kLmSmem);
  });
  if (attr != cudaSuccess) return attr;
  return launch_pdl(lmhead_accept_kernel<MODE>, dim3(grid), dim3(kLmThreads), kLmSmem, st, maps, p);
}

}  // namespace
}  // namespace ssv

extern "C" ssv_status ssv_lmhead_accept_workspace(const ssv_lmhead_accept_args* a, size_t* bytes) {
  using namespace ssv;
  if (!bytes) return SSV_ERR_INVALID;
  const ssv_status st = lm_check(a);
  if (st != SSV_OK) return st;
  if (a->batch == 0 || a->total_slots == 0) {
    *bytes = 0;
    return SSV_OK;
  }
  const int nsm = lm_sm_count();
  if (nsm < 1) return SSV_ERR_CUDA;
  *bytes = lm_layout(a, nsm).total;
  return SSV_OK;
}

extern "C" ssv_status ssv_lmhead_accept(const ssv_lmhead_accept_args* a, void* ws, size_t ws_bytes, void* stream) {
  using namespace ssv;
  const ssv_status st = lm_check(a);
  if (st != SSV_OK) return st;
  if (a->batch == 0 || a->total_slots == 0) return SSV_OK;
  const int nsm = lm_sm_count();
  if (nsm < 1) return SSV_ERR_CUDA;
  const LmLayout L = lm_layout(a, nsm);
  if (!ws || ((uintptr_t)ws & 255u) || ws_bytes < L.total) return SSV_ERR_WORKSPACE;
  LmMaps maps;
  char* w = static_cast<char*>(ws);
  if (!encode_rows(&maps.h, w + L.h_rows, a->total_slots, a->hidden, 128) ||
      !encode_rows(&maps.h0, a->hidden_states, a->total_slots, a->hidden, 128) ||
      !encode_rows(&maps.w, a->lm_head, a->V, a->hidden, 256) ||
      !encode_rows(&maps.w64, a->lm_head, a->V, a->hidden, 64) ||
      !encode_rows(&maps.w16, a->lm_head, a->V, a->hidden, 16))
    return SSV_ERR_INVALID;
  LmParams p;
  memset(&p, 0, sizeof(p));
  const bool noise = a->mode == SSV_ACCEPT_GUMBEL && a->T > 0.f;
  AcceptParams& c = p.acc;
  c.mode = noise ? SSV_ACCEPT_GUMBEL : SSV_ACCEPT_ARGMAX;
  c.T = a->T;
  c.V = a->V;
  c.batch = a->batch;
  c.total_slots = a->total_slots;
  c.draft_tokens = a->draft_tokens;
  c.tau = a->tau;
  c.block = a->block;
  c.gamma = a->gamma;
  c.slot_off = a->slot_off;
  c.n_acc = a->n_acc;
  c.n_out = a->n_out;
  c.tokens = a->tokens;
  c.dev_status = a->dev_status;
  c.cnt_seq = reinterpret_cast<int32_t*>(w + L.cnt_seq);
  c.rowres = reinterpret_cast<RowResult*>(w + L.rowres);
  p.hidden = a->hidden;
  p.nk = a->hidden / 64;
  p.Mt = L.Mt;
  p.V16 = L.V16;
  p.NP = L.NP;
  p.use_noise = noise ? 1 : 0;
  p.vec = ((a->V % 4) == 0 && ((uintptr_t)a->noise & 15u) == 0) ? 1 : 0;
  p.T = a->T;
  p.noise = a->noise;
  p.n_noise_rows = a->n_noise_rows;
  p.noise_row = a->noise_row;
  p.cnt_tile = reinterpret_cast<int32_t*>(w + L.cnt_tile);
  p.h_src = static_cast<const __nv_bfloat16*>(a->hidden_states);
  p.h_rows = reinterpret_cast<__nv_bfloat16*>(w + L.h_rows);
  p.n_rows = reinterpret_cast<int32_t*>(w + L.n_rows);
  p.row_slot = reinterpret_cast<int32_t*>(w + L.row_slot);
  p.rowkey = reinterpret_cast<unsigned long long*>(w + L.rowkey);
  const FaultSetting f = fault_for(SSV_FAULT_LMHEAD);
  p.wait_budget = f.budget;
  p.fault_skip = f.skip;
  c.wait_budget = f.budget;
  c.fault_skip = -1;
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int gather_grid = std::min(nsm, std::max(1, (a->total_slots + 15) / 16));
  cudaError_t e = launch_pdl(lmhead_gather_kernel, dim3(gather_grid), dim3(kGatherThreads), 0, s, p);
  if (e == cudaSuccess)
    e = noise ? lm_launch<SSV_ACCEPT_GUMBEL>(maps, p, nsm, s) : lm_launch<SSV_ACCEPT_ARGMAX>(maps, p, nsm, s);
  return e == cudaSuccess ? SSV_OK : SSV_ERR_CUDA;
}
