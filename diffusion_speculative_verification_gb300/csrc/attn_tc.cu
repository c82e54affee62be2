// Tensor-core verify attention (bf16 in, fp32 accumulate, head_dim 128).
//
// SimSD summary, section 2 "Temporal Attention Mask" and section 4
// "Verification": one pass of softmax(q K^T * scale) V under the temporal
// mask, evaluated per (row, key) from tau on the fly (never stored).
//
// Work unit = (sequence b, kv head g, UR consecutive query rows of b) x all G
// query heads of the group.  It is split into MT M-tiles of 128 packed rows
// (R = 128 / G query rows x G heads each); tile row m is (query row
// row0 + mt * R + m / G, head g * G + m % G), which is exactly the order in
// which the 3-D TMA box (64 x G x R) lands in shared memory.  Every K/V block
// loaded for a unit feeds all of its tiles (grouped-query packing).
//
// Keys of a unit: the sequence's cache keys (visible to every row), then its
// fresh keys up to the last row that needs them (prompt rows are causal,
// tail rows follow tau).  Blocks of 128 keys visible to every valid row skip
// the mask.
//
// Scheduling is persistent stream-K: one CTA per SM; the concatenated key
// blocks of all units are cut into equal contiguous ranges, one per CTA (when
// there are no more units than SMs, each unit gets the same whole number of
// CTAs, so the kv heads of a sequence are read in lockstep).  A
// unit split across CTAs leaves fp32 partials (unnormalised O, running max,
// sum) in the workspace; for each 32-row group the warp that arrives last
// (per-group arrival counter, no waiting on other CTAs) merges the partials
// and writes the output.  The plan is derived on the device from seqs.
//
// Roles per CTA (4 * MT + 2 warps):
//   warp 0  TMA producer (Q tiles per segment, K/V blocks into a 2-stage
//           ring) and TMEM owner (512 columns)
//   warp 1  MMA issuer: S_mt = Q_mt K^T into TMEM, then O_mt += P_mt V with P
//           read from TMEM (it overwrites S_mt's first 64 columns) and V as
//           an MN-major shared-memory operand; with two active tiles they
//           alternate so one softmax warpgroup computes while the tensor core
//           serves the other; a unit with one active tile double-buffers its S
//           over both tiles' S columns instead, so S(n + 1) overlaps softmax(n)
//   warps 2.. softmax, 4 per tile (one TMEM lane quadrant each): S row from
//           TMEM, mask, running max with lazy rescaling of O (only when the
//           max grows by more than 2^8), exp2, bf16 P back into TMEM;
//           epilogue O / l, or partial + merge.
// Every wait is bounded; an expired wait raises a CTA abort flag, in-flight
// copies and MMAs are drained, TMEM is freed and SSV_ERR_TIMEOUT reported.
#include "ssv_internal.cuh"
#include "attn.cuh"
#include "tc_ptx.cuh"

#include <cuda.h>
#include <cudaTypedefs.h>
#include <math.h>
#include <mutex>
#include <type_traits>

namespace ssv {
namespace tc {

using namespace ptx;

constexpr int D = 128;
constexpr int BN = 128;   // keys per block
constexpr int NSK = 3;    // K pipeline stages (keys are needed first, so they run further ahead)
constexpr int NSV = 2;    // V pipeline stages
constexpr uint32_t TILE_BYTES = 128 * 128 * 2;  // one 128 x 128 bf16 operand
constexpr uint32_t HALF_BYTES = TILE_BYTES / 2;  // one 64-column swizzle atom column
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t TM_O = 256;                   // O_mt at columns 256 + 128 mt; S_mt / P_mt at 128 mt
constexpr float kRescaleThreshold = 8.0f;        // log2 units
constexpr int kMergeBlocks = 8;                  // key blocks a partial merge costs, roughly
// Work estimate of the plan, in cost units of about 0.3 us, fitted to the
// per-CTA times of a mixed decode batch (prompt lengths 256..8192, blocks of
// 4..32 slots): a key block multiplied into one tile costs 4 (1.2 us: the
// K/V fetch and one S / PV pair), into two tiles 7 (2.2 us: the tensor
// work doubles, the fetch does not); a segment's fixed work (Q load, the
// first block's two-pass softmax, the masked last block, the epilogue) 22.
constexpr int kSegCost = 22;
constexpr int kMaxBlockCost = 7;

enum : uint32_t {
  B_Q_FULL = 0,
  B_Q_EMPTY = 1,
  B_K_FULL = 2,                  // + stage
  B_K_EMPTY = B_K_FULL + NSK,    // + stage
  B_V_FULL = B_K_EMPTY + NSK,    // + stage
  B_V_EMPTY = B_V_FULL + NSV,    // + stage
  B_S_FULL = B_V_EMPTY + NSV,    // + tile (units with two active tiles)
  B_P_FULL = B_S_FULL + 2,       // + tile
  B_PV_DONE = B_P_FULL + 2,      // one active tile: each PV complete
  B_O_FREE = B_PV_DONE + 1,      // + tile
  B_SDB = B_O_FREE + 2,          // + S buffer (units with one active tile)
  B_PDB = B_SDB + 2,             // + S buffer
  B_SEG_DONE = B_PDB + 2,        // every PV of the segment complete (one phase per segment)
  B_FINAL = B_SEG_DONE + 1,
  B_COUNT = B_FINAL + 1
};

template <int MT>
struct Cfg {
  static constexpr int kSoftWarps = 4 * MT;
  static constexpr int kThreads = 64 + 32 * kSoftWarps;
  static constexpr uint32_t SM_Q = 0;
  static constexpr uint32_t SM_K = SM_Q + MT * TILE_BYTES;
  static constexpr uint32_t SM_V = SM_K + NSK * TILE_BYTES;
  static constexpr uint32_t SM_BAR = SM_V + NSV * TILE_BYTES;
  static constexpr uint32_t SM_TOTAL = SM_BAR + 256;
  static constexpr uint32_t SM_ALLOC = SM_TOTAL + 1024;
};
constexpr size_t kMaxSmemPerCta = 227 * 1024;  // opt-in limit per CTA on sm_100-family parts
static_assert(Cfg<2>::SM_ALLOC <= kMaxSmemPerCta, "pipeline buffers exceed shared memory");

struct TcMaps {
  CUtensorMap q, kc, vc, kn, vn;
};

struct TcWork {
  int32_t* plan;   // [grid][4][batch + 1] per-CTA planning tables
  int32_t* cnt;    // [units][MT][4] arrival counters (zero between calls)
  float* part_ml;  // [2 * grid][MT][128][2]  running max (log2 domain), sum
  float* part_o;   // [2 * grid][MT][D / 4][128][4] unnormalised O (see part_o_at)
};

// Release increment (no return value, so no round trip) and a bounded
// acquire poll for the per-(unit, tile, row group) arrival counters.
__device__ __forceinline__ void red_release_add(int32_t* p, int v) {
  asm volatile("red.release.gpu.global.add.s32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ int ld_acquire(const int32_t* p) {
  int v;
  asm volatile("ld.acquire.gpu.global.s32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
// Waits (bounded) until *p reaches `target`; false on timeout (raising *abort)
// or when another role has raised *abort.
__device__ __forceinline__ bool wait_count(const int32_t* p, int target, volatile int* abort, long long budget) {
  const long long t0 = clock64();
  while (ld_acquire(p) < target) {
    if (*abort) return false;
    if (clock64() - t0 > budget) {
      *abort = 1;
      return false;
    }
  }
  return true;
}

// Float4 group c4 (columns 4 c4 .. 4 c4 + 3) of partial row `slot_row` (= tile
// slot * 128 + row).  Column groups are outermost within a tile, so the 32
// lanes of a warp (consecutive rows) touch 512 contiguous bytes per access.
__device__ __forceinline__ float4* part_o_at(float* part_o, size_t slot_row, int c4) {
  return reinterpret_cast<float4*>(part_o + (slot_row >> 7) * (128 * D)) + (size_t)c4 * 128 + (slot_row & 127);
}

// Per head: W key blocks, U units, Pe owning CTAs and Wc cost units; this
// CTA's head g and its range [begin, end) of the head's blocks, which starts
// at block k0 of unit u0.
struct PlanHdr {
  long long Wc;
  int W, U, Pe, g, begin, end, u0, k0;
};
static_assert(8 * B_COUNT + 8 + sizeof(PlanHdr) <= 256, "barrier area overflow");

struct Unit {
  int b, g;
  int C, N, B, rows, q_off, k_off, kv_off, tau_off;  // k_off: first fresh key row
  int row0, nvalid, mc, cache_blocks, nblocks, full_new;
};

__device__ __forceinline__ int cdiv(int a, int b) { return (a + b - 1) / b; }

__device__ __forceinline__ int unit_weight(int rows, int row0, int UR, int R, int MT) {
  return (MT == 2 && min(UR, rows - row0) > R) ? 7 : 4;  // cost of a key block of the unit
}

// Key blocks of the unit whose rows start at row0: the cache, then the fresh
// keys up to its last prompt row (causal), or through the tail rows' keys when
// it holds tail rows (in a prompt-only pass tail rows see the prompt alone).
__device__ __forceinline__ int unit_nblocks(int C, int N, int rows, int row0, int UR, bool tail_keys) {
  const int kmax = (row0 + UR <= N) ? (row0 + UR) : (tail_keys ? rows : N);
  return cdiv(C, BN) + cdiv(kmax, BN);
}

// Query rows of a sequence: N prompt rows, then 2B tail rows (B data, B mask)
// or, in a prompt-only pass, B rows.
__device__ __forceinline__ int seq_rows(const ssv_seq& s, bool prompt_only) {
  return s.new_len + (prompt_only ? 1 : 2) * s.block;
}

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ uint32_t pick4(uint32_t a, uint32_t b, uint32_t c, uint32_t d, int w) {
  return w == 0 ? a : (w == 1 ? b : (w == 2 ? c : (w == 3 ? d : 0u)));
}

// bits [0, n) set, n clamped to [0, 32]
__device__ __forceinline__ uint32_t prefix32(int n) {
  return n >= 32 ? 0xffffffffu : (n <= 0 ? 0u : ((1u << n) - 1u));
}

// 32-bit window [t0, t0 + 32) of the 128-bit mask (w0 | w1 << 32 | ...), zero outside [0, 128)
__device__ __forceinline__ uint32_t window32(uint32_t w0, uint32_t w1, uint32_t w2, uint32_t w3, int t0) {
  if (t0 <= -32 || t0 >= 128) return 0u;
  const int w = t0 >> 5;  // floor division (arithmetic shift)
  const int sh = t0 & 31;
  const uint32_t lo = pick4(w0, w1, w2, w3, w);
  const uint32_t hi = pick4(w0, w1, w2, w3, w + 1);
  return sh == 0 ? lo : __funnelshift_r(lo, hi, sh);
}

template <int MT, typename OutT>
__global__ void __launch_bounds__(Cfg<MT>::kThreads, 1)
attn_tc_kernel(const __grid_constant__ TcMaps maps, const AttnParams p, const TcWork work, int G, int plan_smem) {
  using C_ = Cfg<MT>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C_::SM_BAR + 8 * B_COUNT);
  volatile int* abort = reinterpret_cast<volatile int*>(smem + C_::SM_BAR + 8 * B_COUNT + 4);
  PlanHdr* plan = reinterpret_cast<PlanHdr*>(smem + C_::SM_BAR + 8 * B_COUNT + 8);
  // planning tables of this CTA: shared memory when they fit, else the global
  // workspace (visible to the CTA after __syncthreads)
  int* s_prefU = plan_smem ? reinterpret_cast<int*>(smem + C_::SM_TOTAL)
                           : work.plan + (size_t)blockIdx.x * 4 * (p.batch + 1);
  int* s_prefB = s_prefU + (p.batch + 1);
  int* s_prefC = s_prefB + (p.batch + 1);
  int* s_ntile = s_prefC + (p.batch + 1);
  auto bar = [&](uint32_t i) -> uint32_t { return sbase + C_::SM_BAR + 8u * i; };

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const long long wb = p.wait_budget;  // cycles a bounded wait may take (kWaitBudget unless a test shortens it)
  const int R = 128 / G;
  const int UR = MT * R;
  const int P = gridDim.x;   // CTAs launched; only the first Pe own key blocks
  const int cta = blockIdx.x;
  const bool po = p.prompt_only != 0;

  // ------------------------------------------------------------------ plan
  // Work is partitioned per kv head: CTA c serves head g = c % Hkv as rank r = c / Hkv of
  // the Ph CTAs of that head, over the head's units in (sequence, row tile) order.  Every
  // head has identical work, so CTAs of different heads stay at the same token offsets and
  // read the heads of a token (adjacent in memory) together.  Tables are per head.
  if (warp == 0) {
    // Before the preceding kernel completes, only an early launch (its outputs
    // do not overlap seqs, tau or the KV cache) with the plan in shared memory
    // may read inputs; otherwise wait here (the barrier below orders the rest).
    if (!(p.early && plan_smem)) pdl_wait();
    int carryU = 0, carryB = 0, carryC = 0;
    for (int b0 = 0; b0 < p.batch; b0 += 32) {
      const int b = b0 + lane;
      int units = 0, blocks = 0, cost = 0;
      if (b < p.batch) {
        const ssv_seq s = p.seqs[b];
        const int rows = seq_rows(s, po);
        // a sequence outside the call's buffers (or above the stated maxima)
        // gets no units: its rows are neither read nor written
        const bool ext = po ? (s.cache_len >= 0 && s.new_len >= 0 && s.block >= 1 && s.block <= 64 && s.q_off >= 0 &&
                               (long long)s.q_off + rows <= p.total_rows && s.tau_off >= 0 &&
                               (long long)s.tau_off + s.new_len <= p.total_krows && s.kv_off >= 0 &&
                               (long long)s.kv_off + s.cache_len <= p.total_cache)
                            : seq_extents_ok(s, p.total_rows, p.total_cache, p.total_slots);
        const bool ok = ext && s.cache_len <= p.max_cache && s.new_len <= p.max_new && s.block <= p.max_block;
        if (!ok && cta == 0) report(p.dev_status, SSV_ERR_INVALID);
        // (a prompt-only sequence without prompt keys has nothing to attend to: no units)
        const int nt = (ok && (!po || s.cache_len + s.new_len > 0)) ? cdiv(rows, UR) : 0;
        for (int t = 0; t < nt; ++t) {
          const int nb = unit_nblocks(s.cache_len, s.new_len, rows, t * UR, UR, !po);
          blocks += nb;
          cost += kSegCost + unit_weight(rows, t * UR, UR, R, MT) * nb;
        }
        s_ntile[b] = nt;
        units = nt;
      }
      int iu = units, ib = blocks, ic = cost;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int yu = __shfl_up_sync(0xffffffffu, iu, o), yb = __shfl_up_sync(0xffffffffu, ib, o);
        const int yc = __shfl_up_sync(0xffffffffu, ic, o);
        if (lane >= o) { iu += yu; ib += yb; ic += yc; }
      }
      if (b < p.batch) { s_prefU[b + 1] = carryU + iu; s_prefB[b + 1] = carryB + ib; s_prefC[b + 1] = carryC + ic; }
      carryU += __shfl_sync(0xffffffffu, iu, 31);
      carryB += __shfl_sync(0xffffffffu, ib, 31);
      carryC += __shfl_sync(0xffffffffu, ic, 31);
    }
    __syncwarp();  // table entries written by every lane are read by lane 0 below
    if (lane == 0) {
      s_prefU[0] = 0;
      s_prefB[0] = 0;
      s_prefC[0] = 0;
      PlanHdr h;
      h.W = carryB;  // key blocks per head
      h.U = carryU;  // units per head
      // CTAs per head: all of them, unless there are no more units than CTAs and one CTA
      // per unit finishes sooner than spreading the head's blocks over all of them, which
      // splits units and costs a merge (about kMergeBlocks key blocks of time).
      const int cap = max(P / p.Hkv, 1);
      int ph = cap;
      if (carryU > 0 && carryU <= cap) {
        const long long per_unit = (long long)carryB * cap;             // (blocks per unit) * U * cap
        const long long per_cta = ((long long)carryB + (long long)kMergeBlocks * cap) * carryU;  // (...) * U * cap
        ph = per_cta < per_unit ? cap : carryU;
      }
      ph = min(ph, max(carryB, 1));
      // every range at least one block's weight wide: no range falls between two
      // block starts of a unit, so the ranks holding a unit's blocks are consecutive
      ph = min(ph, max(carryC / kMaxBlockCost, 1));
      h.Pe = ph;
      h.g = cta % p.Hkv;
      // The head's units are cut into Pe contiguous ranges of equal estimated cost.
      // Unit u occupies the costs [c_u, c_u + kSegCost + w_u n_u) (its fixed work
      // first), its i-th block sits at cost coordinate c_u + kSegCost + w_u i, and
      // rank r owns the blocks whose coordinate lies in [r Wc / Pe, (r + 1) Wc / Pe).
      const long long Wc = carryC;
      h.Wc = Wc;
      // first block at or after cost coordinate C, as (block, unit, offset in the unit)
      auto locate = [&](long long C, int& u_out, int& k_out) -> int {
        int lo = 0, hi = p.batch - 1, b = 0;
        while (lo <= hi) {  // last sequence whose cost range starts at or before C
          const int mid = (lo + hi) >> 1;
          if (s_prefC[mid] <= C) { b = mid; lo = mid + 1; } else { hi = mid - 1; }
        }
        const ssv_seq s = p.seqs[b];
        const int rows = seq_rows(s, po);
        int xs = s_prefB[b], uu = s_prefU[b];
        long long cu = s_prefC[b];
        for (int t = 0;; ++t, ++uu) {
          const int nb = unit_nblocks(s.cache_len, s.new_len, rows, t * UR, UR, !po);
          const int w = unit_weight(rows, t * UR, UR, R, MT);
          if (t == s_ntile[b] - 1 || cu + kSegCost + (long long)w * nb > C) {
            const long long d = C - cu - kSegCost;
            const int i = d <= 0 ? 0 : (int)min((d + w - 1) / w, (long long)nb);
            u_out = (i == nb) ? uu + 1 : uu;
            k_out = (i == nb) ? 0 : i;
            return xs + i;
          }
          xs += nb;
          cu += kSegCost + (long long)w * nb;
        }
      };
      const int r = cta / p.Hkv;
      h.begin = h.end = h.u0 = h.k0 = 0;
      if (cta < ph * p.Hkv && carryB > 0) {
        int u1, k1;
        h.begin = locate(((long long)r * Wc) / ph, h.u0, h.k0);
        h.end = (r + 1 == ph) ? carryB : locate(((long long)(r + 1) * Wc) / ph, u1, k1);
      }
      *plan = h;
      *abort = 0;
      for (uint32_t i = 0; i < B_COUNT; ++i) {
        uint32_t cnt = 1;
        if (i == B_P_FULL || i == B_P_FULL + 1 || i == B_PDB || i == B_PDB + 1 || i == B_O_FREE || i == B_O_FREE + 1)
          cnt = 4;
        mbar_init(bar(i), cnt);
      }
      fence_mbar_init();
    }
    __syncwarp();
    tmem_alloc(smem_u32(tmem_slot), TMEM_COLS);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  // Dependents may launch once every kernel before this one has completed,
  // or (early launch) once the step's rotation kernel, which waited for its
  // own predecessor before letting this one start, is the only one running.
  pdl_trigger();
  const uint32_t tmem = *tmem_slot;
  const int begin = plan->begin, end = plan->end, Ph = plan->Pe, Uh = plan->U;
  const long long Wc = plan->Wc;
  const int gh = plan->g;           // kv head served by this CTA
  const int rank = cta / p.Hkv;     // rank among the CTAs of head gh

  // decode head-local unit u (sequence, row tile) from the plan tables
  auto decode = [&](int u) -> Unit {
    Unit x;
    int lo = 0, hi = p.batch - 1, b = 0;
    while (lo <= hi) {
      const int mid = (lo + hi) >> 1;
      if (s_prefU[mid] <= u) { b = mid; lo = mid + 1; } else { hi = mid - 1; }
    }
    const int tile = u - s_prefU[b];
    x.b = b;
    x.g = gh;
    const ssv_seq s = p.seqs[b];
    x.C = s.cache_len; x.N = s.new_len; x.B = s.block;
    x.q_off = s.q_off; x.kv_off = s.kv_off; x.tau_off = s.tau_off;
    x.k_off = po ? s.tau_off : s.q_off;
    x.rows = seq_rows(s, po);
    x.row0 = tile * UR;
    x.nvalid = min(UR, x.rows - x.row0);
    x.mc = (MT == 2 && x.nvalid > R) ? 2 : 1;
    x.cache_blocks = cdiv(x.C, BN);
    x.nblocks = unit_nblocks(x.C, x.N, x.rows, x.row0, UR, !po);
    x.full_new = (x.row0 < x.N) ? (x.row0 + 1) : x.N;
    return x;
  };
  // rank r owns the head's blocks with cost coordinate in [cost_start(r), cost_start(r + 1))
  auto cost_start = [&](int r) -> long long { return ((long long)r * Wc) / Ph; };
  auto owner_at = [&](long long c) -> int {  // rank owning the block at cost coordinate c
    int r = (int)((c * Ph) / (Wc > 0 ? Wc : 1));
    r = min(max(r, 0), Ph - 1);
    while (r + 1 < Ph && cost_start(r + 1) <= c) ++r;
    while (r > 0 && cost_start(r) > c) --r;
    return r;
  };
  auto unit_cost = [&](int u) -> long long {  // cost coordinate where head-local unit u starts
    int lo = 0, hi = p.batch - 1, b = 0;
    while (lo <= hi) {
      const int mid = (lo + hi) >> 1;
      if (s_prefU[mid] <= u) { b = mid; lo = mid + 1; } else { hi = mid - 1; }
    }
    const ssv_seq s = p.seqs[b];
    const int rows = seq_rows(s, po);
    long long c = s_prefC[b];
    for (int t = 0; t < u - s_prefU[b]; ++t)
      c += kSegCost + (long long)unit_weight(rows, t * UR, UR, R, MT) *
                          unit_nblocks(s.cache_len, s.new_len, rows, t * UR, UR, !po);
    return c;
  };

  if (warp == 0) {
    // ============================================================ producer
    if (lane == 0 && begin < end) {
      tma_prefetch(&maps.q); tma_prefetch(&maps.kc); tma_prefetch(&maps.vc);
      tma_prefetch(&maps.kn); tma_prefetch(&maps.vn);
      int u = plan->u0, k = plan->k0, remaining = end - begin, seg = 0, kn = 0, vn = 0;
      bool run = true;
      auto load_k = [&](const Unit& x, int j) -> bool {
        const int st = kn % NSK;
        if (kn >= NSK && !mbar_wait(bar(B_K_EMPTY + st), ((kn / NSK) - 1) & 1, abort, wb)) return false;
        if (cta == 0 && kn == p.fault_skip) {  // test support: this key block's copy is left out
          ++kn;
          return true;
        }
        mbar_expect_tx(bar(B_K_FULL + st), TILE_BYTES);
        const bool cache = j < x.cache_blocks;
        const CUtensorMap* mk = cache ? &maps.kc : &maps.kn;
        const int z = cache ? (x.kv_off + j * BN) : (x.k_off + (j - x.cache_blocks) * BN);
        const uint32_t dk = sbase + C_::SM_K + st * TILE_BYTES;
        tma_load_3d(dk, mk, 0, x.g, z, bar(B_K_FULL + st));
        tma_load_3d(dk + HALF_BYTES, mk, 64, x.g, z, bar(B_K_FULL + st));
        ++kn;
        return true;
      };
      auto load_v = [&](const Unit& x, int j) -> bool {
        const int st = vn % NSV;
        if (vn >= NSV && !mbar_wait(bar(B_V_EMPTY + st), ((vn / NSV) - 1) & 1, abort, wb)) return false;
        mbar_expect_tx(bar(B_V_FULL + st), TILE_BYTES);
        const bool cache = j < x.cache_blocks;
        const CUtensorMap* mv = cache ? &maps.vc : &maps.vn;
        const int z = cache ? (x.kv_off + j * BN) : (x.k_off + (j - x.cache_blocks) * BN);
        const uint32_t dv = sbase + C_::SM_V + st * TILE_BYTES;
        tma_load_3d(dv, mv, 0, x.g, z, bar(B_V_FULL + st));
        tma_load_3d(dv + HALF_BYTES, mv, 64, x.g, z, bar(B_V_FULL + st));
        ++vn;
        return true;
      };
      // Q, K_new and V_new may come from the preceding kernel (the rotation):
      // they are loaded only after pdl_wait().  On an early launch KV-cache
      // blocks are not.
      bool waited = !(p.early && plan_smem);
      auto dep_wait = [&]() {
        if (!waited) {
          pdl_wait();
          waited = true;
        }
      };
      while (run && remaining > 0) {
        const Unit x = decode(u);
        const int len = min(x.nblocks - k, remaining);
        int jk = k, jv = k;  // next key / value block of the segment to load
        if (!waited) {
          // first segment: fill the rings with cache blocks while the preceding kernel runs
          while (jk < k + len && jk < x.cache_blocks && jk - k < NSK) {
            if (!load_k(x, jk++)) { run = false; break; }
          }
          while (run && jv + 1 < jk && jv - k < NSV) {
            if (!load_v(x, jv++)) { run = false; break; }
          }
          if (!run) break;
        }
        dep_wait();
        // the first key block does not depend on Q: start it before waiting for the Q buffer
        if (jk == k && !load_k(x, jk++)) break;
        if (seg > 0 && !mbar_wait(bar(B_Q_EMPTY), (seg - 1) & 1, abort, wb)) break;
        mbar_expect_tx(bar(B_Q_FULL), x.mc * TILE_BYTES);
        for (int mt = 0; mt < x.mc; ++mt) {
          const int z = x.q_off + x.row0 + mt * R;
          tma_load_3d(sbase + C_::SM_Q + mt * TILE_BYTES, &maps.q, 0, x.g * G, z, bar(B_Q_FULL));
          tma_load_3d(sbase + C_::SM_Q + mt * TILE_BYTES + HALF_BYTES, &maps.q, 64, x.g * G, z, bar(B_Q_FULL));
        }
        ++seg;
        // keys run one block ahead of values
        while (jk < k + len || jv < k + len) {
          if (jk < k + len && !load_k(x, jk++)) { run = false; break; }
          if (jv < k + len && (jv + 1 < jk || jk == k + len) && !load_v(x, jv++)) { run = false; break; }
        }
        if (!run) break;
        remaining -= len;
        ++u;
        k = 0;
      }
      if (!waited) pdl_wait();
      // drain (bounded, regardless of abort): the last Q load and the last K / V loads
      if (seg > 0) {
        const long long t0 = clock64();
        while (!mbar_try_wait(bar(B_Q_FULL), (seg - 1) & 1) && clock64() - t0 < wb) {
        }
      }
      for (int n = (kn > NSK ? kn - NSK : 0); n < kn; ++n) {
        const long long t0 = clock64();
        while (!mbar_try_wait(bar(B_K_FULL + n % NSK), (n / NSK) & 1) && clock64() - t0 < wb) {
        }
      }
      for (int n = (vn > NSV ? vn - NSV : 0); n < vn; ++n) {
        const long long t0 = clock64();
        while (!mbar_try_wait(bar(B_V_FULL + n % NSV), (n / NSV) & 1) && clock64() - t0 < wb) {
        }
      }
    }
  } else if (warp == 1) {
    // ============================================================ MMA issuer
    if (lane == 0 && begin < end) {
      const uint32_t id_s = idesc_bf16(128, 128, false);
      const uint32_t id_pv = idesc_bf16(128, 128, true);
      int u = plan->u0, k = plan->k0, remaining = end - begin, seg = 0;
      int nseg0 = 0, nseg1 = 0;  // segments of tile 0 / tile 1 (their O_FREE phases)
      bool run = true;
      const uint64_t dq0 = smem_desc_sw128(sbase + C_::SM_Q, 16, 1024);
      const uint64_t dq1 = smem_desc_sw128(sbase + C_::SM_Q + (MT > 1 ? TILE_BYTES : 0), 16, 1024);
      // The issue of a GEMM returns only once the tensor pipe's queue (about one MMA
      // deep) has room, so whatever this thread does between GEMMs leaves the pipe
      // idle: ring positions live in registers as barrier addresses, descriptors and
      // parities advanced by additions, and the phases waited on next are tested
      // inside the issue of the GEMM before (gemm_*_probe).  `seen` holds one bit
      // per such phase already observed complete; a probe only ever targets the next
      // phase of its kind still to be consumed, so a set bit stays true until used.
      enum : uint32_t { SEEN_K = 1, SEEN_V = 2, SEEN_P0 = 4, SEEN_P1 = 8, SEEN_PD = 16 };
      uint32_t seen = 0;
      uint32_t kb = bar(B_K_FULL), kph = 0u;  // K ring: FULL barrier of the next key block's stage, parity
      uint64_t kd = smem_desc_sw128(sbase + C_::SM_K, 16, 1024);  // and that stage's descriptor
      int ks = 0;
      uint32_t vb = bar(B_V_FULL), vph = 0u, vbn = bar(B_V_FULL + 1), vphn = 0u;  // V ring: next block, the one after
      uint64_t vd = smem_desc_sw128(sbase + C_::SM_V, HALF_BYTES, 1024);
      uint64_t vdn = smem_desc_sw128(sbase + C_::SM_V + TILE_BYTES, HALF_BYTES, 1024);
      const uint32_t pb0 = bar(B_P_FULL), pb1 = bar(B_P_FULL + 1);
      uint32_t pph0 = 0u, pph1 = 0u;
      int dbs = 0, dbp = 0;  // one-tile segments: blocks whose S / PV have been issued (S buffer = count & 1)
      static_assert(NSV == 2, "the V ring below has two stages");
      auto wait_seen = [&](uint32_t bit, uint32_t b, uint32_t par) -> bool {
        if (seen & bit) {
          seen &= ~bit;
          return true;
        }
        return mbar_wait_poll(b, par, abort, wb);
      };
      auto note = [&](uint32_t r, uint32_t bit_a, uint32_t bit_b) {
        seen |= ((r & 1u) ? bit_a : 0u) | ((r & 2u) ? bit_b : 0u);
      };
      auto k_advance = [&]() {
        if (ks == NSK - 1) {
          ks = 0;
          kb -= 8u * (NSK - 1);
          kd -= (uint64_t)(NSK - 1) * (TILE_BYTES >> 4);
          kph ^= 1u;
        } else {
          ++ks;
          kb += 8u;
          kd += TILE_BYTES >> 4;
        }
      };
      auto v_advance = [&]() {  // two stages: the next becomes current; a stage's parity flips per use
        const uint32_t tb = vb, tp = vph;
        const uint64_t td = vd;
        vb = vbn; vph = vphn; vd = vdn;
        vbn = tb; vphn = tp ^ 1u; vdn = td;
      };
      auto pdb_bar = [&](int n) -> uint32_t { return bar(B_PDB + (n & 1)); };
      auto pdb_par = [&](int n) -> uint32_t { return (uint32_t)(n >> 1) & 1u; };
      // one-tile segment: S of the next key block into S buffer dbs & 1
      auto issue_s_db = [&](uint32_t b1, uint32_t p1, uint32_t bit1, uint32_t b2, uint32_t p2, uint32_t bit2) -> bool {
        if (!wait_seen(SEEN_K, kb, kph)) return false;
        tc_fence_after();
        const uint32_t sbuf = (uint32_t)dbs & 1u;
        note(gemm_ss_k128_probe(tmem + sbuf * 128, dq0, kd, id_s, 0u, b1, p1, b2, p2), bit1, bit2);
        mma_commit(bar(B_SDB + sbuf));
        mma_commit(kb + 8u * NSK);  // K_EMPTY of the stage
        k_advance();
        ++dbs;
        return true;
      };
      while (run && remaining > 0) {
        const Unit x = decode(u);
        const int len = min(x.nblocks - k, remaining);
        if (!mbar_wait_poll(bar(B_Q_FULL), seg & 1, abort, wb)) break;
        if (x.mc == 1) {
          // ---- one active tile: S double-buffered over both tiles' S columns, so
          // S(n + 1) runs while the softmax warps work on S(n).  Per block: PV(n)
          // (P(n) in buffer n & 1), then S(n + 2) into the same buffer (tensor-core
          // operations of this thread complete in issue order).
          if (!issue_s_db(vb, vph, SEEN_V, vb, vph, SEEN_V)) break;
          if (len > 1 && !issue_s_db(vb, vph, SEEN_V, pdb_bar(dbp), pdb_par(dbp), SEEN_PD)) break;
          for (int i = 0; i < len; ++i) {
            if (!wait_seen(SEEN_V, vb, vph) || !wait_seen(SEEN_PD, pdb_bar(dbp), pdb_par(dbp)) ||
                (i == 0 && nseg0 > 0 && !mbar_wait_poll(bar(B_O_FREE), (nseg0 - 1) & 1, abort, wb))) {
              run = false;
              break;
            }
            tc_fence_after();
            {
              const bool s_next = i + 2 < len;  // needed next: K for S(n + 2), else the next P
              const uint32_t b1 = s_next ? kb : pdb_bar(dbp + 1), p1 = s_next ? kph : pdb_par(dbp + 1);
              note(gemm_ts_k128_probe(tmem + TM_O, tmem + ((uint32_t)dbp & 1u) * 128, vd, id_pv, i > 0 ? 1u : 0u, b1,
                                      p1, vbn, vphn),
                   s_next ? SEEN_K : SEEN_PD, SEEN_V);
            }
            mma_commit(bar(B_PV_DONE));
            mma_commit(vb + 8u * NSV);  // V_EMPTY of the stage
            v_advance();
            ++dbp;
            if (i + 2 < len && !issue_s_db(pdb_bar(dbp), pdb_par(dbp), SEEN_PD, vb, vph, SEEN_V)) {
              run = false;
              break;
            }
          }
          if (!run) break;
        } else {
          // ---- two tiles: per block, PV_0(j) S_0(j + 1) PV_1(j) S_1(j + 1)
          if (!wait_seen(SEEN_K, kb, kph)) break;
          tc_fence_after();
          note(gemm_ss_k128_probe(tmem, dq0, kd, id_s, 0u, vb, vph, vb, vph), SEEN_V, SEEN_V);
          mma_commit(bar(B_S_FULL));
          note(gemm_ss_k128_probe(tmem + 128, dq1, kd, id_s, 0u, vb, vph, vb, vph), SEEN_V, SEEN_V);
          mma_commit(bar(B_S_FULL + 1));
          mma_commit(kb + 8u * NSK);
          k_advance();
          for (int i = 0; i < len; ++i) {
            const bool more = i + 1 < len;
            const uint32_t acc = i > 0 ? 1u : 0u;
            if (!wait_seen(SEEN_V, vb, vph)) { run = false; break; }
            // tile 0
            if (!wait_seen(SEEN_P0, pb0, pph0) ||
                (i == 0 && nseg0 > 0 && !mbar_wait_poll(bar(B_O_FREE), (nseg0 - 1) & 1, abort, wb))) {
              run = false;
              break;
            }
            tc_fence_after();
            {
              // needed next: the key block of S_0(j + 1) (else the next V), then tile 1's P
              const uint32_t b1 = more ? kb : vbn, p1 = more ? kph : vphn;
              note(gemm_ts_k128_probe(tmem + TM_O, tmem, vd, id_pv, acc, b1, p1, pb1, pph1), more ? SEEN_K : SEEN_V,
                   SEEN_P1);
            }
            pph0 ^= 1u;
            if (more) {
              if (!wait_seen(SEEN_K, kb, kph)) { run = false; break; }
              tc_fence_after();
              note(gemm_ss_k128_probe(tmem, dq0, kd, id_s, 0u, pb1, pph1, vbn, vphn), SEEN_P1, SEEN_V);
              mma_commit(bar(B_S_FULL));
            }
            // tile 1
            if (!wait_seen(SEEN_P1, pb1, pph1) ||
                (i == 0 && nseg1 > 0 && !mbar_wait_poll(bar(B_O_FREE + 1), (nseg1 - 1) & 1, abort, wb))) {
              run = false;
              break;
            }
            tc_fence_after();
            note(gemm_ts_k128_probe(tmem + TM_O + 128, tmem + 128, vd, id_pv, acc, pb0, pph0, vbn, vphn), SEEN_P0,
                 SEEN_V);
            pph1 ^= 1u;
            if (more) {
              note(gemm_ss_k128_probe(tmem + 128, dq1, kd, id_s, 0u, pb0, pph0, vbn, vphn), SEEN_P0, SEEN_V);
              mma_commit(bar(B_S_FULL + 1));
              mma_commit(kb + 8u * NSK);
              k_advance();
            }
            mma_commit(vb + 8u * NSV);
            v_advance();
          }
          if (!run) break;
          ++nseg1;
        }
        mma_commit(bar(B_SEG_DONE));
        mma_commit(bar(B_Q_EMPTY));
        ++nseg0;
        remaining -= len;
        ++seg;
        ++u;
        k = 0;
      }
    }
    if (lane == 0) {
      // every MMA issued by this thread completes before TMEM is released
      mma_commit(bar(B_FINAL));
      const long long t0 = clock64();
      while (!mbar_try_wait(bar(B_FINAL), 0) && clock64() - t0 < wb) {
      }
    }
  } else {
    // ============================================================ softmax
    const int mt = (warp - 2) >> 2;   // tile served by this warp
    const int q4 = warp & 3;          // TMEM lane quadrant
    const int m = q4 * 32 + lane;     // tile row = TMEM lane
    const uint32_t lane_base = static_cast<uint32_t>(q4 * 32) << 16;
    const uint32_t tO = tmem + lane_base + TM_O + mt * 128;
    const float cexp = p.scale * 1.4426950408889634f;
    int u = plan->u0, k = plan->k0, remaining = end - begin, seg = 0;
    int n2 = 0, ndb = 0;     // blocks in two-tile / one-tile units (their S / P barrier phases)
    bool run = true;
    auto warp_wait = [&](uint32_t b, uint32_t parity) -> bool {
      const bool w = mbar_wait(b, parity, abort, wb);
      return __all_sync(0xffffffffu, w);
    };
    while (run && remaining > 0) {
      const Unit x = decode(u);
      const int len = min(x.nblocks - k, remaining);
      const bool complete = (k == 0 && len == x.nblocks);
      if (mt < x.mc) {
        const int r_local = mt * R + m / G;
        const int hj = m % G;
        const int i = x.row0 + r_local;  // local query row in the sequence
        const bool valid = r_local < x.nvalid;
        const bool warp_active = (mt * R + (q4 * 32) / G) < x.nvalid;
        const bool db = x.mc == 1;  // one active tile: its S is double-buffered
        const bool prompt = i < x.N;
        const int r = i - x.N;
        uint32_t tm0 = 0u, tm1 = 0u, tm2 = 0u, tm3 = 0u;  // allowed tail keys of this row
        if (!po && warp_active && x.row0 + x.nvalid > x.N) {   // warp-uniform: the unit holds tail rows
          // stage map of the sequence in two registers per lane
          const int32_t* tau = p.tau + x.tau_off;
          const int ta = lane < x.B ? tau[lane] : 0;
          const int tb = lane + 32 < x.B ? tau[lane + 32] : 0;
          // the stage map must permute 1..B; a bad map cannot index out of range
          // (the shuffles below take lane indices mod 32): report only
          {
            unsigned long long seen = 0ull;
            bool ok = true;
            if (lane < x.B) { if (ta < 1 || ta > x.B) ok = false; else seen |= 1ull << (ta - 1); }
            if (lane + 32 < x.B) { if (tb < 1 || tb > x.B) ok = false; else seen |= 1ull << (tb - 1); }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) seen |= __shfl_xor_sync(0xffffffffu, seen, o);
            ok = __all_sync(0xffffffffu, ok);
            const unsigned long long full = (x.B >= 64) ? ~0ull : ((1ull << x.B) - 1ull);
            if (!(ok && seen == full) && lane == 0) report(p.dev_status, SSV_ERR_BAD_TAU);
          }
          const bool tail_row = valid && !prompt;  // other rows see no tail key (masks stay 0)
          const int slot_r = tail_row ? (r % x.B) : 0;  // the unit holds tail rows, so B > 0
          // the stage of this lane's own slot: fetch both halves from the holding lane and
          // choose here (a choice made inside the shuffle would use the source lane's slot)
          const int tra = __shfl_sync(0xffffffffu, ta, slot_r & 31), trb = __shfl_sync(0xffffffffu, tb, slot_r & 31);
          const int tr = slot_r < 32 ? tra : trb;
          // le / lt: the slots whose stage is <= tr / < tr, accumulated over the stages
          // v = 1..B in order (one ballot pair per stage: the slot holding stage v)
          unsigned long long acc = 0ull, le = 0ull, lt = 0ull;
          for (int v = 1; v <= x.B; ++v) {
            const uint32_t lo = __ballot_sync(0xffffffffu, ta == v), hi = __ballot_sync(0xffffffffu, tb == v);
            acc |= ((unsigned long long)hi << 32) | lo;
            if (v == tr - 1) lt = acc;
            if (v == tr) le = acc;
          }
          // tail key t < B is data slot t, t >= B mask slot t - B.  A data row sees the
          // data slots of stages <= its own; a mask row sees the data slots of earlier
          // stages and the mask slots of its own stage and later ones.
          // (every lane took part in the ballots; only tail rows keep masks)
          const unsigned long long bmask = (x.B >= 64) ? ~0ull : ((1ull << x.B) - 1ull);
          const bool data_row = r < x.B;
          const unsigned long long lo_part = !tail_row ? 0ull : (data_row ? le : lt);          // keys [0, B)
          const unsigned long long hi_part = (!tail_row || data_row) ? 0ull : (~lt & bmask);  // keys [B, 2B)
          const unsigned long long w01 = lo_part | (x.B < 64 ? (hi_part << x.B) : 0ull);
          const unsigned long long w23 = x.B == 0 ? 0ull : (x.B < 64 ? (hi_part >> (64 - x.B)) : hi_part);
          tm0 = (uint32_t)w01; tm1 = (uint32_t)(w01 >> 32);
          tm2 = (uint32_t)w23; tm3 = (uint32_t)(w23 >> 32);
        }
        float m_used = -INFINITY, l_sum = 0.f;
        for (int jj = 0; jj < len; ++jj) {
          const int j = k + jj;
          // one active tile: S alternates between two TMEM buffers (its n-th block in buffer n & 1)
          const int sb = db ? (ndb & 1) : mt;
          const uint32_t tS = tmem + lane_base + sb * 128;
          const uint32_t sparity = db ? ((ndb >> 1) & 1) : (n2 & 1);
          if (db) ++ndb; else ++n2;
          if (!warp_wait(db ? bar(B_SDB + sb) : bar(B_S_FULL + mt), sparity)) { run = false; break; }
          if (!warp_active) {
            __syncwarp();
            if (lane == 0) mbar_arrive(db ? bar(B_PDB + sb) : bar(B_P_FULL + mt));
            continue;
          }
          tc_fence_after();
          // ---- visibility of this block's 128 keys for this row, as 32-column bitmasks
          const bool is_cache = j < x.cache_blocks;
          const int kbase = is_cache ? j * BN : (j - x.cache_blocks) * BN;
          const bool full = is_cache ? (kbase + BN <= x.C) : (kbase + BN <= x.full_new);
          const bool all_vis = __all_sync(0xffffffffu, full && valid);
          int lim = BN, lim_rows = 0, toff = 0;  // prefix limit; tail bits for columns < lim_rows
          if (!valid) {
            lim = 0;
          } else if (!full) {
            if (is_cache) {
              lim = x.C - kbase;
            } else if (prompt) {
              lim = min(i + 1, x.rows) - kbase;
            } else {
              lim = x.N - kbase;
              lim_rows = x.rows - kbase;
              toff = kbase - x.N;  // tail index of column 0
            }
          }
          auto vis32 = [&](int q) -> uint32_t {  // visibility bits of columns [32q, 32q + 32)
            uint32_t v = prefix32(lim - 32 * q);
            if (lim_rows > 32 * q) v |= window32(tm0, tm1, tm2, tm3, toff + 32 * q) & prefix32(lim_rows - 32 * q);
            return v;
          };
          // ---- steady state (not the segment's first block): one pass with the running
          // max, P kept in registers until no row's max has grown past the rescale
          // threshold; otherwise fall through to the two-pass path (S intact).  Columns
          // a row may not see enter as -inf (their P is exactly 0).
          bool done = false;
          float l0 = 0.f, l1 = 0.f, l2 = 0.f, l3 = 0.f;
          auto one_pass = [&](auto masked_tag) {
            constexpr bool kMasked = decltype(masked_tag)::value;
            uint32_t b0[16], b1[16], pw[64];
            float a0 = -INFINITY, a1 = -INFINITY, a2 = -INFINITY, a3 = -INFINITY;
            uint64_t lp0 = 0ull, lp1 = 0ull;  // packed (even, odd) partial sums of P
            const uint64_t cc2 = pack2(cexp, cexp), nm2 = pack2(-m_used, -m_used);
            tmem_ld16(tS, b0);
            tmem_wait_ld();
#pragma unroll
            for (int q = 0; q < BN / 16; ++q) {
              uint32_t* cur = (q & 1) ? b1 : b0;
              uint32_t* nxt = (q & 1) ? b0 : b1;
              if (q + 1 < BN / 16) tmem_ld16(tS + (q + 1) * 16, nxt);
              uint32_t vq = ~0u;  // visibility of this chunk's 16 columns (bits 0..15)
              if constexpr (kMasked) vq = vis32(q >> 1) >> ((q & 1) * 16);
#pragma unroll
              for (int e = 0; e < 8; ++e) {
                float s0 = __uint_as_float(cur[2 * e]), s1 = __uint_as_float(cur[2 * e + 1]);
                if constexpr (kMasked) {
                  const uint32_t bits = vq >> (2 * e);
                  s0 = (bits & 1u) ? s0 : -INFINITY;
                  s1 = (bits & 2u) ? s1 : -INFINITY;
                }
                if ((e & 3) == 0) a0 = max3(a0, s0, s1);
                else if ((e & 3) == 1) a1 = max3(a1, s0, s1);
                else if ((e & 3) == 2) a2 = max3(a2, s0, s1);
                else a3 = max3(a3, s0, s1);
                float x0, x1;
                unpack2(ffma2(pack2(s0, s1), cc2, nm2), x0, x1);
                const float p0 = ex2(x0), p1 = ex2(x1);
                const __nv_bfloat162 pb = __floats2bfloat162_rn(p0, p1);
                pw[q * 8 + e] = *reinterpret_cast<const uint32_t*>(&pb);
                if (e & 1) lp1 = fadd2(lp1, pack2(p0, p1)); else lp0 = fadd2(lp0, pack2(p0, p1));
              }
              if (q + 1 < BN / 16) tmem_wait_ld();
            }
            const float mx1 = fmaxf(fmaxf(a0, a1), fmaxf(a2, a3));
            if (!__any_sync(0xffffffffu, mx1 * cexp > m_used + kRescaleThreshold)) {
#pragma unroll
              for (int q = 0; q < BN / 32; ++q) tmem_st16(tS + q * 16, pw + q * 16);
              unpack2(lp0, l0, l1);
              unpack2(lp1, l2, l3);
              done = true;
            }
          };
          if (jj > 0 && __all_sync(0xffffffffu, m_used > -INFINITY)) {
            if (all_vis) one_pass(std::false_type{});
            else one_pass(std::true_type{});
          }
          if (!done) {
            // ---- pass 1: row max of the raw scores (the scale is positive)
            float mx;
            {
              float a[8];
#pragma unroll
              for (int e = 0; e < 8; ++e) a[e] = -INFINITY;
#pragma unroll 1
              for (int h = 0; h < 2; ++h) {
                uint32_t sr[64];
                tmem_ld32(tS + h * 64, sr);
                tmem_ld32(tS + h * 64 + 32, sr + 32);
                tmem_wait_ld();
                if (all_vis) {
#pragma unroll
                  for (int e = 0; e < 64; ++e) a[e & 7] = fmaxf(a[e & 7], __uint_as_float(sr[e]));
                } else {
                  const uint32_t v0 = vis32(2 * h), v1 = vis32(2 * h + 1);
#pragma unroll
                  for (int e = 0; e < 64; ++e) {
                    const uint32_t vw = e < 32 ? v0 : v1;
                    const float f = ((vw >> (e & 31)) & 1u) ? __uint_as_float(sr[e]) : -INFINITY;
                    a[e & 7] = fmaxf(a[e & 7], f);
                  }
                }
              }
              mx = fmaxf(fmaxf(fmaxf(a[0], a[1]), fmaxf(a[2], a[3])), fmaxf(fmaxf(a[4], a[5]), fmaxf(a[6], a[7])));
            }
            const float mxs = mx * cexp;
            const bool need = (mx > -INFINITY) && (m_used == -INFINITY || mxs > m_used + kRescaleThreshold);
            if (jj > 0 && __any_sync(0xffffffffu, need)) {
              // O holds PV of the earlier blocks: it must be complete before rescaling.
              // Two active tiles: S(j) of a tile was issued after its PV(j - 1), so S(j)
              // being complete implies it.  One active tile: wait for the PV of the
              // previous block (phase ndb - 2 of the per-PV barrier, ndb counting this one).
              if (db && !warp_wait(bar(B_PV_DONE), ndb & 1)) { run = false; break; }
              tc_fence_after();
              const float f = need ? ex2(m_used - mxs) : 1.f;
              uint32_t raw[32];
#pragma unroll
              for (int c = 0; c < D / 32; ++c) {
                tmem_ld32(tO + c * 32, raw);
                tmem_wait_ld();
#pragma unroll
                for (int e = 0; e < 32; ++e) raw[e] = __float_as_uint(__uint_as_float(raw[e]) * f);
                tmem_st32(tO + c * 32, raw);
              }
              tmem_wait_st();
              l_sum *= f;
            }
            if (need) m_used = mxs;
            const float mref = (m_used == -INFINITY) ? 0.f : m_used;
            // ---- pass 2: P = exp2(s * c - m) as bf16 pairs into TMEM over S columns [0, 64).
            // Chunk q reads S columns [32q, 32q + 32) and writes P columns [16q, 16q + 16),
            // which lie in S columns already read.
#pragma unroll 1
            for (int q = 0; q < BN / 32; ++q) {
              uint32_t sr[32];
              tmem_ld32(tS + q * 32, sr);
              tmem_wait_ld();
              uint32_t pw[16];
              if (all_vis) {
#pragma unroll
                for (int e = 0; e < 16; ++e) {
                  const float p0 = ex2(fmaf(__uint_as_float(sr[2 * e]), cexp, -mref));
                  const float p1 = ex2(fmaf(__uint_as_float(sr[2 * e + 1]), cexp, -mref));
                  const __nv_bfloat162 pb = __floats2bfloat162_rn(p0, p1);
                  pw[e] = *reinterpret_cast<const uint32_t*>(&pb);
                  if (e & 1) { l2 += p0; l3 += p1; } else { l0 += p0; l1 += p1; }
                }
              } else {
                const uint32_t vw = vis32(q);
#pragma unroll
                for (int e = 0; e < 16; ++e) {
                  const float p0 = ((vw >> (2 * e)) & 1u) ? ex2(fmaf(__uint_as_float(sr[2 * e]), cexp, -mref)) : 0.f;
                  const float p1 =
                      ((vw >> (2 * e + 1)) & 1u) ? ex2(fmaf(__uint_as_float(sr[2 * e + 1]), cexp, -mref)) : 0.f;
                  const __nv_bfloat162 pb = __floats2bfloat162_rn(p0, p1);
                  pw[e] = *reinterpret_cast<const uint32_t*>(&pb);
                  if (e & 1) { l2 += p0; l3 += p1; } else { l0 += p0; l1 += p1; }
                }
              }
              tmem_st16(tS + q * 16, pw);
            }
          }
          tmem_wait_st();
          l_sum += (l0 + l1) + (l2 + l3);
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(db ? bar(B_PDB + sb) : bar(B_P_FULL + mt));
        }
        if (!run) break;
        // ---- segment epilogue: O stays in TMEM until O_FREE is signalled.
        // Every PV of the segment must be complete: the issuer commits the
        // segment-end barrier after the segment's last MMA.
        if (!warp_wait(bar(B_SEG_DONE), seg & 1)) {
          run = false;
          break;
        }
        if (warp_active) {
          tc_fence_after();
          OutT* orow = static_cast<OutT*>(p.o) + ((size_t)(x.q_off + i) * p.Hq + x.g * G + hj) * D;
          // log2-sum-exp2 of the row's scaled scores (m is that of the scores behind l)
          auto store_lse = [&](float m, float l) {
            if (p.lse && valid) p.lse[(size_t)(x.q_off + i) * p.Hq + x.g * G + hj] = l > 0.f ? m + log2f(l) : -INFINITY;
          };
          auto store_chunk = [&](int q, const float* v, float inv) {
            if (!valid) return;
            if constexpr (sizeof(OutT) == 4) {
#pragma unroll
              for (int c = 0; c < 32; c += 4)
                *reinterpret_cast<float4*>(orow + q * 32 + c) =
                    make_float4(v[c] * inv, v[c + 1] * inv, v[c + 2] * inv, v[c + 3] * inv);
            } else {
#pragma unroll
              for (int c = 0; c < 32; c += 8) {
                uint32_t w[4];
#pragma unroll
                for (int h = 0; h < 4; ++h) {
                  const __nv_bfloat162 bv = __floats2bfloat162_rn(v[c + 2 * h] * inv, v[c + 2 * h + 1] * inv);
                  w[h] = *reinterpret_cast<const uint32_t*>(&bv);
                }
                *reinterpret_cast<uint4*>(orow + q * 32 + c) = make_uint4(w[0], w[1], w[2], w[3]);
              }
            }
          };
          // (one-shot code: loops stay rolled, the instructions arrive cold)
          if (complete) {
            const float inv = (l_sum > 0.f) ? 1.f / l_sum : 0.f;
            store_lse(m_used, l_sum);
#pragma unroll 1
            for (int q = 0; q < D / 32; ++q) {
              uint32_t raw[32];
              tmem_ld32(tO + q * 32, raw);
              tmem_wait_ld();
              float v[32];
#pragma unroll
              for (int e = 0; e < 32; ++e) v[e] = __uint_as_float(raw[e]);
              store_chunk(q, v, inv);
            }
          } else {
            // ---- split unit: ranks c_a .. c_b of head gh hold its pieces.  Rank c_a holds
            // the head, which ends its range while every other piece starts its rank's
            // range, so as a rule c_a finishes last: it merges.  The others publish their
            // partial with a release increment and move on without waiting.
            const long long cu = unit_cost(u);
            const int c_a = owner_at(cu + kSegCost);                                   // ranks of head gh holding
            const int c_b = owner_at(cu + kSegCost + (long long)unit_weight(x.rows, x.row0, UR, R, MT) *
                                                          (x.nblocks - 1));                 // the first, last block
            int32_t* counter = work.cnt + (((size_t)gh * Uh + u) * MT + mt) * 4 + q4;
            // partial slot of rank rr (> c_a): its piece is the first segment of its range
            auto slot_of = [&](int rr) -> size_t { return ((size_t)((rr * p.Hkv + gh) * 2) * MT + mt) * 128 + m; };
            if (rank != c_a) {
              const size_t myslot = slot_of(rank);
              __stcg(reinterpret_cast<float2*>(work.part_ml + myslot * 2), make_float2(m_used, l_sum));
#pragma unroll 1
              for (int q = 0; q < D / 32; ++q) {
                uint32_t raw[32];
                tmem_ld32(tO + q * 32, raw);
                tmem_wait_ld();
#pragma unroll
                for (int c = 0; c < 32; c += 4)
                  __stcg(part_o_at(work.part_o, myslot, q * 8 + c / 4),
                         make_float4(__uint_as_float(raw[c]), __uint_as_float(raw[c + 1]),
                                     __uint_as_float(raw[c + 2]), __uint_as_float(raw[c + 3])));
              }
              __syncwarp();  // every lane's stores precede lane 0's release
              if (lane == 0) red_release_add(counter, 1);
            } else {
              int ok = 1;
              if (lane == 0) ok = wait_count(counter, c_b - c_a, abort, wb) ? 1 : 0;
              ok = __shfl_sync(0xffffffffu, ok, 0);
              __syncwarp();  // the other lanes' loads below follow lane 0's acquire
              if (!ok) run = false;
            }
            if (rank == c_a && run) {
              // combine in CTA order (not arrival order) so the result is deterministic
              const int nparts = c_b - c_a + 1;
              if (nparts <= 4) {
                // (m, l) of every partial in one round of loads, then O 64 columns at a
                // time with all of a partial's loads for those columns issued together
                float2 ml[4];
                size_t po[4];  // partial slot row of each part; ~0 for this CTA's own (in TMEM)
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                  const int cc = c_a + k;
                  po[k] = ~size_t(0);
                  ml[k] = make_float2(-INFINITY, 0.f);
                  if (k < nparts) {
                    if (cc == rank) {
                      ml[k] = make_float2(m_used, l_sum);
                    } else {
                      const size_t sl = slot_of(cc);
                      ml[k] = __ldcg(reinterpret_cast<const float2*>(work.part_ml + sl * 2));
                      po[k] = sl;
                    }
                  }
                }
                float M = -INFINITY;
#pragma unroll
                for (int k = 0; k < 4; ++k) M = fmaxf(M, ml[k].x);
                float L = 0.f, fo[4];
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                  fo[k] = (M == -INFINITY || k >= nparts) ? 0.f : ex2(ml[k].x - M);
                  L += ml[k].y * fo[k];
                }
                const float inv = (L > 0.f) ? 1.f / L : 0.f;
                store_lse(M, L);
#pragma unroll 1
                for (int q = 0; q < D / 32; ++q) {
                  float v[32];
#pragma unroll
                  for (int e = 0; e < 32; ++e) v[e] = 0.f;
#pragma unroll
                  for (int k = 0; k < 4; ++k) {
                    if (k >= nparts) break;
                    if (po[k] == ~size_t(0)) {
                      uint32_t raw[32];
                      tmem_ld32(tO + q * 32, raw);
                      tmem_wait_ld();
#pragma unroll
                      for (int e = 0; e < 32; ++e) v[e] += __uint_as_float(raw[e]) * fo[k];
                    } else {
                      float4 w4[8];
#pragma unroll
                      for (int c = 0; c < 8; ++c) w4[c] = __ldcg(part_o_at(work.part_o, po[k], q * 8 + c));
#pragma unroll
                      for (int c = 0; c < 8; ++c) {
                        v[4 * c] += w4[c].x * fo[k]; v[4 * c + 1] += w4[c].y * fo[k];
                        v[4 * c + 2] += w4[c].z * fo[k]; v[4 * c + 3] += w4[c].w * fo[k];
                      }
                    }
                  }
                  store_chunk(q, v, inv);
                }
              } else {
                float M = m_used;
                for (int cc = c_a; cc <= c_b; ++cc)
                  if (cc != rank) M = fmaxf(M, __ldcg(work.part_ml + slot_of(cc) * 2));
                float L = 0.f;
                for (int cc = c_a; cc <= c_b; ++cc) {
                  float mo = m_used, lo = l_sum;
                  if (cc != rank) {
                    const float2 mlc = __ldcg(reinterpret_cast<const float2*>(work.part_ml + slot_of(cc) * 2));
                    mo = mlc.x;
                    lo = mlc.y;
                  }
                  if (M > -INFINITY) L += lo * ex2(mo - M);
                }
                const float inv = (L > 0.f) ? 1.f / L : 0.f;
                store_lse(M, L);
#pragma unroll 1
                for (int q = 0; q < D / 32; ++q) {
                  float v[32];
#pragma unroll
                  for (int e = 0; e < 32; ++e) v[e] = 0.f;
                  for (int cc = c_a; cc <= c_b; ++cc) {
                    if (cc == rank) {
                      uint32_t raw[32];
                      tmem_ld32(tO + q * 32, raw);
                      tmem_wait_ld();
                      const float f = (M == -INFINITY) ? 0.f : ex2(m_used - M);
#pragma unroll
                      for (int e = 0; e < 32; ++e) v[e] += __uint_as_float(raw[e]) * f;
                    } else {
                      const size_t sl = slot_of(cc);
                      const float mo = __ldcg(work.part_ml + sl * 2);
                      const float f = (M == -INFINITY) ? 0.f : ex2(mo - M);
#pragma unroll
                      for (int c = 0; c < 32; c += 4) {
                        const float4 w4 = __ldcg(part_o_at(work.part_o, sl, q * 8 + c / 4));
                        v[c] += w4.x * f; v[c + 1] += w4.y * f; v[c + 2] += w4.z * f; v[c + 3] += w4.w * f;
                      }
                    }
                  }
                  store_chunk(q, v, inv);
                }
              }
              if (lane == 0) *counter = 0;  // ready for the next call
            }
          }
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(bar(B_O_FREE + mt));
        } else {
          __syncwarp();
          if (lane == 0) mbar_arrive(bar(B_O_FREE + mt));
        }
      }
      remaining -= len;
      ++seg;
      ++u;
      k = 0;
    }
  }
  // ------------------------------------------------------------------ teardown
  __syncwarp();  // the producer and issuer lanes rejoin their warps before the CTA barrier
  tc_fence_before();
  __syncthreads();
  if (*abort && threadIdx.x == 0) report(p.dev_status, SSV_ERR_TIMEOUT);
  if (threadIdx.x == 32) pdl_wait();  // this grid never completes before the one it follows
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
// box (64, box_heads, box_rows), 128-byte swizzle, zero fill out of bounds.
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

static int sm_count() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  return n;
}

static int choose_mt(const AttnParams& p) {
  const int G = p.Hq / p.Hkv;
  const long long max_rows = (long long)p.max_new + (p.prompt_only ? 1LL : 2LL) * p.max_block;
  return (max_rows * G > 128) ? 2 : 1;
}

struct WsLayout {
  size_t plan, cnt, ml, o, total;
  int grid, mt, units;
};

static WsLayout ws_layout(const AttnParams& p) {
  WsLayout L;
  const int G = p.Hq / p.Hkv;
  L.mt = choose_mt(p);
  const int UR = L.mt * (128 / G);
  const long long max_rows = (long long)p.max_new + (p.prompt_only ? 1LL : 2LL) * p.max_block;
  L.units = (int)((long long)p.batch * p.Hkv * ((max_rows + UR - 1) / UR));
  L.grid = sm_count();
  size_t off = 0;
  L.plan = off;
  off = align_up(off + sizeof(int32_t) * (size_t)L.grid * 4 * (p.batch + 1), 256);
  L.cnt = off;
  off = align_up(off + sizeof(int32_t) * (size_t)L.units * L.mt * 4, 256);
  L.ml = off;
  off = align_up(off + sizeof(float) * 2 * (size_t)(2 * L.grid) * L.mt * 128, 256);
  L.o = off;
  off = align_up(off + sizeof(float) * (size_t)(2 * L.grid) * L.mt * 128 * D, 256);
  L.total = off;
  return L;
}

bool attn_tc_supported(const AttnParams& p) {
  if (p.in_dtype != SSV_BF16 || p.d != D) return false;
  const int G = p.Hq / p.Hkv;
  if (G < 1 || G > 128 || (128 % G) != 0) return false;
  if (p.max_block > 64 || p.Hkv > sm_count()) return false;  // every kv head needs a CTA
  // total key blocks must fit comfortably in int32
  const long long max_rows = (long long)p.max_new + (p.prompt_only ? 1LL : 2LL) * p.max_block;
  const long long blocks = (long long)p.batch * p.Hkv * (max_rows / (128 / G) + 1) *
                           ((p.max_cache + BN - 1) / BN + (max_rows + BN - 1) / BN);
  if (blocks > (1LL << 26)) return false;  // plan costs (at most 29 units per block) stay in int32
  return encode_fn() != nullptr && sm_count() > 0;
}

size_t attn_tc_workspace(const AttnParams& p) { return ws_layout(p).total; }

// Shared memory of a launch: the pipeline buffers, plus the planning tables
// (4 x (batch + 1) ints) when they fit under the per-CTA limit.
static size_t plan_table_bytes(const AttnParams& p) { return sizeof(int32_t) * 4 * (size_t)(p.batch + 1); }

template <int MT>
static bool plan_in_smem(const AttnParams& p) {
  return Cfg<MT>::SM_ALLOC + plan_table_bytes(p) <= kMaxSmemPerCta;
}

template <int MT, typename OutT>
static cudaError_t launch_t(const AttnParams& p, const TcMaps& maps, const TcWork& w, int G, int grid,
                            cudaStream_t st) {
  static std::once_flag once;
  static cudaError_t attr_err = cudaSuccess;
  std::call_once(once, [] {
    attr_err = cudaFuncSetAttribute(attn_tc_kernel<MT, OutT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    (int)kMaxSmemPerCta);
  });
  if (attr_err != cudaSuccess) return attr_err;
  const int in_smem = plan_in_smem<MT>(p) ? 1 : 0;
  const size_t smem = Cfg<MT>::SM_ALLOC + (in_smem ? plan_table_bytes(p) : 0);
  // The merge of a split unit waits (bounded) on partials from other CTAs of
  // the grid, so every CTA must be able to be resident at once: one per SM,
  // checked here rather than discovered as a timeout.
  int per_sm = 0;
  const cudaError_t oe =
      cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, attn_tc_kernel<MT, OutT>, Cfg<MT>::kThreads, smem);
  if (oe != cudaSuccess) return oe;
  if ((long long)per_sm * sm_count() < grid) return cudaErrorCooperativeLaunchTooLarge;
  return launch_pdl(attn_tc_kernel<MT, OutT>, dim3(grid), dim3(Cfg<MT>::kThreads), smem, st, maps, p, w, G, in_smem);
}

cudaError_t launch_attn_tc(const AttnParams& p, void* ws, cudaStream_t st) {
  const int G = p.Hq / p.Hkv;
  const int R = 128 / G;
  const WsLayout L = ws_layout(p);
  TcMaps maps;
  if (!encode_3d(&maps.q, p.q, p.Hq, p.total_rows, G, R)) return cudaErrorInvalidValue;
  const int krows = p.prompt_only ? p.total_krows : p.total_rows;
  if (krows > 0) {
    if (!encode_3d(&maps.kn, p.k_new, p.Hkv, krows, 1, BN)) return cudaErrorInvalidValue;
    if (!encode_3d(&maps.vn, p.v_new, p.Hkv, krows, 1, BN)) return cudaErrorInvalidValue;
  } else {
    maps.kn = maps.q;  // never read: every sequence has N = 0
    maps.vn = maps.q;
  }
  if (p.total_cache > 0) {
    if (!encode_3d(&maps.kc, p.k_cache, p.Hkv, p.total_cache, 1, BN)) return cudaErrorInvalidValue;
    if (!encode_3d(&maps.vc, p.v_cache, p.Hkv, p.total_cache, 1, BN)) return cudaErrorInvalidValue;
  } else {
    maps.kc = maps.kn;  // never read: every sequence has C = 0
    maps.vc = maps.vn;
  }
  char* w = static_cast<char*>(ws);
  TcWork work;
  work.plan = reinterpret_cast<int32_t*>(w + L.plan);
  work.cnt = reinterpret_cast<int32_t*>(w + L.cnt);
  work.part_ml = reinterpret_cast<float*>(w + L.ml);
  work.part_o = reinterpret_cast<float*>(w + L.o);
  if (L.mt == 2) {
    if (p.out_dtype == SSV_F32) return launch_t<2, float>(p, maps, work, G, L.grid, st);
    return launch_t<2, __nv_bfloat16>(p, maps, work, G, L.grid, st);
  }
  if (p.out_dtype == SSV_F32) return launch_t<1, float>(p, maps, work, G, L.grid, st);
  return launch_t<1, __nv_bfloat16>(p, maps, work, G, L.grid, st);
}

}  // namespace tc
}  // namespace ssv
