// accept_stream: the acceptance reduce as one persistent CTA per SM.
//
// Each CTA lists the verified rows of the batch in slot order (the same list
// in every CTA), then takes the list's (row, chunk) units one at a time from
// a counter in the workspace (the last CTA to finish returns it to zero); a
// unit is kAccChunk vocabulary entries of the target logits row
// plus, where the rule needs one, the same entries of the draft logits
// (rejection sampling, tested stages) or of the noise row (coupled noise
// from a table; generated noise needs the logits alone).
// Warp roles:
//   warps 0..15  consumers: wait for a stage of the ring, reduce it with
//                warp shuffles (chunk max and compensated sums of
//                2^((x - max) log2(e) / T), or the first argmax of the
//                decision score), post one record per warp, release the
//                stage;
//   warp 16      producer (one lane): bulk-copies each unit's rows into the
//                next free stage (cp.async.bulk, completion on an mbarrier);
//   warp 17      publisher: merges the 16 warp records of a unit into its
//                AccPartial.  The row merges and sequence walks follow the
//                stream as programmatic dependents: accept_finish_kernel (one
//                CTA per sequence) for the decision modes; for rejection
//                sampling accept_rowmerge_kernel (a warp per slot, all rows
//                at once; the last row of a sequence walks it).
// The ring keeps 128 to 192 KB of loads in flight per SM; no CTA-wide
// barrier is taken once the list is built.  Every mbarrier wait is bounded:
// on timeout the CTA raises SSV_ERR_TIMEOUT, the producer still waits
// (bounded) for its own copies, and all roles return.
#include "accept.cuh"
#include "tc_ptx.cuh"

#include <mutex>
#include <type_traits>

namespace ssv {
namespace {

using namespace ptx;

constexpr int kStrConsumerWarps = 16;
constexpr int kStrConsumers = kStrConsumerWarps * 32;        // 512
constexpr int kStrThreads = kStrConsumers + 64;              // + producer warp + publisher warp
constexpr int kStrWarps = kStrThreads / 32;
constexpr int kStrProducerWarp = kStrConsumerWarps;
constexpr int kStrGroups = kAccChunk / (4 * kStrConsumers);  // 4-entry groups per consumer thread
constexpr int kStrRecRing = 8;
constexpr int kStrMaxStages = 8;
constexpr int kStrRingBytes = 192 * 1024;
constexpr int kStrMaxRows = 2048;
static_assert(kStrGroups * 4 * kStrConsumers == kAccChunk, "chunk split");

template <int MODE, typename T>
struct StrCfg {
  using TB = typename std::conditional<MODE == SSV_ACCEPT_GUMBEL, float, T>::type;  // second stream
  static constexpr uint32_t kRowB = kAccChunk * sizeof(T);                           // offset of the second row
  static constexpr bool kOneRow = MODE == SSV_ACCEPT_ARGMAX || MODE == SSV_ACCEPT_GUMBEL_GEN;  // logits only
  static constexpr uint32_t kStage = kAccChunk * (sizeof(T) + (kOneRow ? 0 : sizeof(TB)));
  static constexpr int kStages = (kStrRingBytes / kStage) < kStrMaxStages ? (kStrRingBytes / kStage) : kStrMaxStages;
  static constexpr int kSmem = kStages * kStage;
  static_assert(kStages >= 2, "ring depth");
};

constexpr int kStrPer = (kStrMaxRows + kStrThreads - 1) / kStrThreads;  // slots (sequences) per thread

struct StrShared {
  uint64_t full[kStrMaxStages];
  uint64_t empty[kStrMaxStages];
  uint64_t rec_full[kStrRecRing];
  uint64_t rec_empty[kStrRecRing];
  AccPartial rec[kStrRecRing][kStrConsumerWarps];
  int unit_of[kStrMaxStages];          // unit held by each ring stage (-1: no units left)
  int rec_unit[kStrRecRing];           // unit of each record-ring slot (-1: end)
  int32_t list[kStrMaxRows];           // verified slot | tested << 31
  int32_t off[kStrMaxRows];            // slot_off per sequence
  unsigned char blk[kStrMaxRows];      // block (0 when the sizes are invalid)
  unsigned char gam[kStrMaxRows];      // gamma
  unsigned char stage[kStrMaxRows];    // tau per slot (0 when outside 1..64)
  unsigned char seq_ok[kStrMaxRows];
  int wcount[kStrWarps];
  int abort;
};

// four consecutive entries of a staged row (e % 4 == 0)
template <typename T>
__device__ __forceinline__ void lds4(const unsigned char* row, int e, float* x) {
  if constexpr (sizeof(T) == 4) {
    const float4 v = *reinterpret_cast<const float4*>(row + (size_t)e * 4);
    x[0] = v.x; x[1] = v.y; x[2] = v.z; x[3] = v.w;
  } else {
    const uint2 v = *reinterpret_cast<const uint2*>(row + (size_t)e * 2);
    x[0] = __uint_as_float(v.x << 16); x[1] = __uint_as_float(v.x & 0xffff0000u);
    x[2] = __uint_as_float(v.y << 16); x[3] = __uint_as_float(v.y & 0xffff0000u);
  }
}

// Sequence holding `slot` (binary search over the shared slot offsets;
// sequences are packed in increasing slot order), or -1.
__device__ __forceinline__ int seq_of_slot(const StrShared& sh, int batch, int slot) {
  int lo = 0, hi = batch - 1, ans = -1;
  while (lo <= hi) {
    const int mid = (lo + hi) >> 1;
    if (sh.off[mid] <= slot) { ans = mid; lo = mid + 1; } else { hi = mid - 1; }
  }
  return ans;
}

// Is `slot` a verified row (stage <= min(gamma + 1, B)) of a valid sequence?
// b: its sequence; tested: its stage carries a draft token.
__device__ __forceinline__ bool verified_slot(const StrShared& sh, int batch, int slot, int& b, int& tested) {
  b = seq_of_slot(sh, batch, slot);
  if (b < 0 || !sh.seq_ok[b] || slot - sh.off[b] >= sh.blk[b]) return false;
  const int st = sh.stage[slot], g = sh.gam[b];
  tested = st <= g;
  return st >= 1 && st <= min(g + 1, (int)sh.blk[b]);
}

// Bounded wait that ignores the abort flag (used to drain copies in flight).
__device__ __forceinline__ void drain_wait(uint32_t bar, uint32_t parity, int32_t* dev_status, long long budget) {
  const long long t0 = clock64();
  while (!mbar_try_wait(bar, parity)) {
    if (clock64() - t0 > budget) {
      report(dev_status, SSV_ERR_TIMEOUT);
      return;
    }
  }
}

template <int MODE, typename T>
__global__ void __launch_bounds__(kStrThreads, 1) accept_stream_kernel(const AcceptParams p) {
  using C = StrCfg<MODE, T>;
  extern __shared__ __align__(128) unsigned char ring[];
  __shared__ StrShared sh;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (!p.early) pdl_wait();  // any input may come from the preceding kernel

  if (tid == 0) {
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(smem_u32(&sh.full[s]), 1);
      mbar_init(smem_u32(&sh.empty[s]), kStrConsumerWarps);
    }
    for (int r = 0; r < kStrRecRing; ++r) {
      mbar_init(smem_u32(&sh.rec_full[r]), kStrConsumerWarps);
      mbar_init(smem_u32(&sh.rec_empty[r]), 1);
    }
    sh.abort = 0;
    fence_mbar_init();
  }

  // ---- every metadata load at once (one round trip), kept in shared memory
  int nrow[kStrPer];
#pragma unroll
  for (int i = 0; i < kStrPer; ++i) {
    const int slot = tid + i * kStrThreads;
    nrow[i] = 0;
    if (slot < p.total_slots) {
      const int t = p.tau[slot];
      sh.stage[slot] = (t >= 1 && t <= 64) ? (unsigned char)t : 0;
      if (MODE == SSV_ACCEPT_GUMBEL) nrow[i] = p.noise_row[slot];
    }
    if (slot < p.batch) {
      const int off = p.slot_off[slot], B = p.block[slot], g = p.gamma[slot];
      const bool sizes = off >= 0 && B >= 1 && B <= 64 && g >= 0 && g <= B && off + B <= p.total_slots;
      sh.off[slot] = off;
      sh.blk[slot] = sizes ? (unsigned char)B : 0;
      sh.gam[slot] = sizes ? (unsigned char)g : 0;
    }
  }
  __syncthreads();
  // ---- sequence validity: sizes, and tau a permutation of 1..B (one warp per sequence)
  for (int b = warp; b < p.batch; b += kStrWarps) {
    const int B = sh.blk[b], off = sh.off[b];
    unsigned long long seen = 0ull;
    bool ok = B >= 1;
    if (ok) {
      for (int j = lane; j < B; j += 32) {
        const int t = sh.stage[off + j];
        if (t < 1 || t > B) ok = false; else seen |= 1ull << (t - 1);
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) seen |= __shfl_xor_sync(0xffffffffu, seen, o);
    }
    ok = __all_sync(0xffffffffu, ok) && seen == ((B >= 64) ? ~0ull : ((1ull << B) - 1ull));
    if (lane == 0) {
      sh.seq_ok[b] = ok;
      if (!ok && blockIdx.x == 0) report(p.dev_status, SSV_ERR_BAD_TAU);
    }
  }
  __syncthreads();
  if (MODE == SSV_ACCEPT_GUMBEL) {  // a verified row needs a noise row in range
#pragma unroll
    for (int i = 0; i < kStrPer; ++i) {
      const int slot = tid + i * kStrThreads;
      int b, tested;
      if (slot < p.total_slots && verified_slot(sh, p.batch, slot, b, tested) &&
          (nrow[i] < 0 || nrow[i] >= p.n_noise_rows)) {
        sh.seq_ok[b] = 0;
        if (blockIdx.x == 0) report(p.dev_status, SSV_ERR_INVALID);
      }
    }
    __syncthreads();
  }

  // ---- verified rows in slot order (ballot + warp counts per pass)
  int total = 0;
  for (int base = 0; base < p.total_slots; base += kStrThreads) {
    const int slot = base + tid;
    int b = -1, tested = 0;
    const bool v = slot < p.total_slots && verified_slot(sh, p.batch, slot, b, tested);
    const unsigned bal = __ballot_sync(0xffffffffu, v);
    if (lane == 0) sh.wcount[warp] = __popc(bal);
    __syncthreads();
    int before = total, sum = 0;
#pragma unroll
    for (int w = 0; w < kStrWarps; ++w) {
      const int c = sh.wcount[w];
      before += (w < warp) ? c : 0;
      sum += c;
    }
    if (v) {
      const int pos = before + __popc(bal & ((1u << lane) - 1u));
      sh.list[pos] = (int)((unsigned)slot | ((unsigned)tested << 31));
    }
    total += sum;
    __syncthreads();
  }

  // ---- the list's (row, chunk) units, U of them: each CTA's producer takes
  // the next one from a counter in the workspace whenever a ring stage frees,
  // so CTAs that stream faster take more units (a fixed split left the sweep's
  // CTAs finishing 30 us apart)
  const int U = total * p.nchunks;

  // Rows of unit u: the logits chunk and, where the rule needs it, the draft
  // logits or noise chunk (bytes multiples of 16 by construction).
  auto unit_rows = [&](int u, const void*& a, uint32_t& bytes_a, const void*& b, uint32_t& bytes_b) {
    const int e = sh.list[u / p.nchunks];
    const int slot = e & 0x7fffffff;
    const int c0 = (int)(u % p.nchunks) * kAccChunk;
    const int nvalid = min(kAccChunk, p.V - c0);
    a = static_cast<const T*>(p.logits) + (size_t)slot * p.V + c0;
    bytes_a = (uint32_t)nvalid * (uint32_t)sizeof(T);
    b = nullptr;
    bytes_b = 0;
    if (MODE == SSV_ACCEPT_REJECT && e < 0) {
      b = static_cast<const T*>(p.draft_logits) + (size_t)slot * p.V + c0;
      bytes_b = bytes_a;
    } else if (MODE == SSV_ACCEPT_GUMBEL) {
      b = p.noise + (size_t)p.noise_row[slot] * p.V + c0;
      bytes_b = (uint32_t)nvalid * 4u;
    }
  };
  // The list used only the batch metadata; logits, draft logits, noise and
  // the workspace are read only once the preceding kernel has completed.
  pdl_wait();
  pdl_trigger();
  if (MODE == SSV_ACCEPT_REJECT && blockIdx.x == 0) {
    // every emission record to "none"; the walks (after this grid) write the
    // valid sequences' own, so the emission passes can trust the records
    for (int b = tid; b < p.batch; b += kStrThreads) {
      p.emit[2 * b] = -1;
      p.emit[2 * b + 1] = 0;
    }
  }

  if (warp == kStrProducerWarp) {
    if (lane != 0) return;
    int issued = 0;
    int next = atomicAdd(p.unit_ctr, 1);  // one unit taken ahead, so the atomic's round trip overlaps the wait
    for (int k = 0;; ++k) {
      const int s = k % C::kStages;
      if (k >= C::kStages && !mbar_wait(smem_u32(&sh.empty[s]), ((k / C::kStages) - 1) & 1, &sh.abort, p.wait_budget)) break;
      const uint32_t fb = smem_u32(&sh.full[s]);
      const int u = next;
      if (u >= U) {  // no units left: this stage carries the end mark
        sh.unit_of[s] = -1;
        mbar_arrive(fb);
        issued = k + 1;
        break;
      }
      next = atomicAdd(p.unit_ctr, 1);
      sh.unit_of[s] = u;
      const void *src_a, *src_b;
      uint32_t bytes_a, bytes_b;
      unit_rows(u, src_a, bytes_a, src_b, bytes_b);
      const uint32_t dst = smem_u32(ring + (size_t)s * C::kStage);
      if (blockIdx.x == 0 && k == p.fault_skip) {  // test support: this chunk's copy is left out
        issued = k + 1;
        continue;
      }
      mbar_expect_tx(fb, bytes_a + bytes_b);
      bulk_load(dst, src_a, bytes_a, fb);
      if (bytes_b) bulk_load(dst + C::kRowB, src_b, bytes_b, fb);
      issued = k + 1;
    }
    // leave no copy in flight: the last fill of every stage has landed
    for (int s = 0; s < C::kStages && s < issued; ++s) {
      const int k_last = s + ((issued - 1 - s) / C::kStages) * C::kStages;
      drain_wait(smem_u32(&sh.full[s]), (k_last / C::kStages) & 1, p.dev_status, p.wait_budget);
    }
    // the last producer to finish taking units returns the counter to zero
    __threadfence();
    if (atomicAdd(p.unit_ctr + 1, 1) == (int)gridDim.x - 1) {
      p.unit_ctr[0] = 0;
      p.unit_ctr[1] = 0;
    }
    if (sh.abort) report(p.dev_status, SSV_ERR_TIMEOUT);
    return;
  }

  if (warp < kStrConsumerWarps) {
    const bool unit_t = p.T == 1.0f;  // l / 1 is exact
    for (int k = 0;; ++k) {
      const int s = k % C::kStages;
      const bool got = mbar_wait(smem_u32(&sh.full[s]), (k / C::kStages) & 1, &sh.abort, p.wait_budget);
      if (!__all_sync(0xffffffffu, got)) break;
      const int u = sh.unit_of[s];
      if (u < 0) {  // end mark: passed on to the publisher through the record ring
        const int rs = k % kStrRecRing;
        const bool room =
            k < kStrRecRing || mbar_wait(smem_u32(&sh.rec_empty[rs]), ((k / kStrRecRing) - 1) & 1, &sh.abort, p.wait_budget);
        if (!__all_sync(0xffffffffu, room)) break;
        if (lane == 0) {
          if (warp == 0) sh.rec_unit[rs] = -1;
          mbar_arrive(smem_u32(&sh.rec_full[rs]));
        }
        break;
      }
      const int chunk = u % p.nchunks;
      const bool tested = sh.list[u / p.nchunks] < 0;
      const int c0 = chunk * kAccChunk;
      const int nvalid = min(kAccChunk, p.V - c0);
      const unsigned char* ra = ring + (size_t)s * C::kStage;
      const unsigned char* rb = ra + C::kRowB;
      AccPartial r;
      if (MODE == SSV_ACCEPT_REJECT) {
        // chunk max (3-input max), then sum of 2^((x - max) c2) with packed
        // f32x2 FMA / add (two chains of 8 terms per thread), TwoSum across lanes
        float xa[4 * kStrGroups], xb[4 * kStrGroups];
#pragma unroll
        for (int j = 0; j < kStrGroups; ++j) {
          const int el = 4 * (j * kStrConsumers + tid);
          if (el < nvalid) {
            lds4<T>(ra, el, xa + 4 * j);
            if (tested) lds4<T>(rb, el, xb + 4 * j);
          } else {
#pragma unroll
            for (int q = 0; q < 4; ++q) xa[4 * j + q] = xb[4 * j + q] = -INFINITY;
          }
        }
        const uint64_t c22 = pack2(p.c2, p.c2);
        auto row_sum = [&](const float* x, float& m, float& hi, float& lo) {
          m = -INFINITY;
#pragma unroll
          for (int j = 0; j < 4 * kStrGroups; j += 2) m = max3(m, x[j], x[j + 1]);
          m = warp_max(m);
          const float nm = (m == -INFINITY) ? 0.f : -m * p.c2;
          const uint64_t nm2 = pack2(nm, nm);
          uint64_t acc = pack2(0.f, 0.f);
#pragma unroll
          for (int j = 0; j < 4 * kStrGroups; j += 2) {
            float y0, y1;
            unpack2(ffma2(pack2(x[j], x[j + 1]), c22, nm2), y0, y1);
            acc = fadd2(acc, pack2(ex2f(y0), ex2f(y1)));
          }
          float s0, s1;
          unpack2(acc, s0, s1);
          hi = s0;
          lo = 0.f;
          two_sum_acc(hi, lo, s1, 0.f);
          warp_sum2(hi, lo);
        };
        row_sum(xa, r.m_a, r.sa_hi, r.sa_lo);
        if (tested) {
          row_sum(xb, r.m_b, r.sb_hi, r.sb_lo);
        } else {
          r.m_b = -INFINITY;
          r.sb_hi = r.sb_lo = 0.f;
        }
        r.val = 0.f; r.idx = 0;
      } else if (MODE == SSV_ACCEPT_GUMBEL_GEN) {
        // Coupled noise generated here.  Every entry gets its generator word
        // and a cheap upper bound of its score (noise::gumbel_upper); the entry
        // with the largest bound in the warp is scored exactly, and only entries
        // whose bound reaches that score can beat it, so only those are scored
        // exactly (about 0.2% of entries): the warp's result is the exact first
        // argmax of the exact scores.
        const uint32_t pos = (uint32_t)p.noise_row[sh.list[u / p.nchunks] & 0x7fffffff];
        const uint32_t key0 = (uint32_t)p.noise_seed, key1 = (uint32_t)(p.noise_seed >> 32);
        const float inv_t = 1.f / p.T;
        float xv[4 * kStrGroups], ub[4 * kStrGroups];
        uint32_t wv[4 * kStrGroups];
        float umax = -INFINITY, xsel = 0.f;  // this lane's largest bound, and its entry's logit and word
        uint32_t wsel = 0u;
#pragma unroll
        for (int j = 0; j < kStrGroups; ++j) {
          const int el = 4 * (j * kStrConsumers + tid);
          if (el < nvalid) {
            lds4<T>(ra, el, xv + 4 * j);
            const uint4 w = noise::philox4x32_10(make_uint4((uint32_t)(c0 + el) >> 2, pos, 0u, 0u), key0, key1);
            wv[4 * j] = w.x; wv[4 * j + 1] = w.y; wv[4 * j + 2] = w.z; wv[4 * j + 3] = w.w;
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              const int jj = 4 * j + q;
              const float sa = unit_t ? xv[jj] : xv[jj] * inv_t;
              ub[jj] = (el + q < nvalid) ? __fmaf_rn(fabsf(sa), 1e-6f, sa + noise::gumbel_upper(wv[jj])) : -INFINITY;
              const bool up = ub[jj] > umax;
              umax = up ? ub[jj] : umax;
              xsel = up ? xv[jj] : xsel;
              wsel = up ? wv[jj] : wsel;
            }
          } else {
#pragma unroll
            for (int q = 0; q < 4; ++q) { ub[4 * j + q] = -INFINITY; xv[4 * j + q] = 0.f; wv[4 * j + q] = 0u; }
          }
        }
        // the warp's largest bound: its entry, scored exactly, bounds the warp's best from below
        const float wmax = warp_max(umax);
        const unsigned who = __ballot_sync(0xffffffffu, umax > -INFINITY && umax == wmax);
        const int src = who ? __ffs(who) - 1 : 0;
        float lb = -INFINITY;
        if (lane == src && who) lb = gen_score(xsel, wsel, p.T, unit_t);
        lb = __shfl_sync(0xffffffffu, lb, src);
        float best = -INFINITY;
        int bi = INT_MAX;
#pragma unroll
        for (int jj = 0; jj < 4 * kStrGroups; ++jj) {
          if (ub[jj] > -INFINITY && ub[jj] >= lb) {  // a token that can reach the warp's best: score it exactly
            const float sc = gen_score(xv[jj], wv[jj], p.T, unit_t);
            const int idx = c0 + 4 * ((jj >> 2) * kStrConsumers + tid) + (jj & 3);
            if (sc > best || bi == INT_MAX) { best = sc; bi = idx; }
          }
        }
        warp_argmax(best, bi);
        r.val = best; r.idx = bi;
        r.m_a = r.m_b = r.sa_hi = r.sa_lo = r.sb_hi = r.sb_lo = 0.f;
      } else {
        float best = -INFINITY;
        int bi = INT_MAX;
#pragma unroll
        for (int j = 0; j < kStrGroups; ++j) {
          const int el = 4 * (j * kStrConsumers + tid);
          if (el < nvalid) {
            float x[4];
            lds4<T>(ra, el, x);
            if (MODE == SSV_ACCEPT_GUMBEL) {
              float gn[4];
              lds4<float>(rb, el, gn);
#pragma unroll
              for (int q = 0; q < 4; ++q) x[q] = __fadd_rn(unit_t ? x[q] : __fdiv_rn(x[q], p.T), gn[q]);
            }
#pragma unroll
            for (int q = 0; q < 4; ++q)
              if (x[q] > best || bi == INT_MAX) { best = x[q]; bi = c0 + el + q; }
          }
        }
        warp_argmax(best, bi);
        r.val = best; r.idx = bi;
        r.m_a = r.m_b = r.sa_hi = r.sa_lo = r.sb_hi = r.sb_lo = 0.f;
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&sh.empty[s]));
      const int rs = k % kStrRecRing;
      const bool room =
          k < kStrRecRing || mbar_wait(smem_u32(&sh.rec_empty[rs]), ((k / kStrRecRing) - 1) & 1, &sh.abort, p.wait_budget);
      if (!__all_sync(0xffffffffu, room)) break;
      if (lane == 0) {
        sh.rec[rs][warp] = r;
        if (warp == 0) sh.rec_unit[rs] = u;
        mbar_arrive(smem_u32(&sh.rec_full[rs]));
      }
    }
    return;
  }

  // ---- publisher warp: the unit's record; the rows are merged and the
  // sequences walked by the completion kernels once every record is written.
  for (int k = 0;; ++k) {
    const int rs = k % kStrRecRing;
    const bool got = mbar_wait(smem_u32(&sh.rec_full[rs]), (k / kStrRecRing) & 1, &sh.abort, p.wait_budget);
    if (!__all_sync(0xffffffffu, got)) break;
    const int u = sh.rec_unit[rs];  // read before the slot is released
    if (u < 0) break;
    AccPartial x;
    if (lane < kStrConsumerWarps) {
      x = sh.rec[rs][lane];
    } else {
      x.m_a = x.m_b = -INFINITY;
      x.sa_hi = x.sa_lo = x.sb_hi = x.sb_lo = 0.f;
      x.val = -INFINITY;
      x.idx = INT_MAX;
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(smem_u32(&sh.rec_empty[rs]));
    if (MODE == SSV_ACCEPT_REJECT) {
      const float Ma = warp_max(x.m_a), Mb = warp_max(x.m_b);
      const float fa = (x.m_a == -INFINITY) ? 0.f : ex2f((x.m_a - Ma) * p.c2);
      const float fb = (x.m_b == -INFINITY) ? 0.f : ex2f((x.m_b - Mb) * p.c2);
      float ha = x.sa_hi * fa, la = x.sa_lo * fa, hb = x.sb_hi * fb, lb = x.sb_lo * fb;
      warp_sum2(ha, la);
      warp_sum2(hb, lb);
      x.m_a = Ma; x.m_b = Mb;
      x.sa_hi = ha; x.sa_lo = la; x.sb_hi = hb; x.sb_lo = lb;
    } else {
      warp_argmax(x.val, x.idx);
    }
    const int row = u / p.nchunks, chunk = u % p.nchunks;
    const int slot = sh.list[row] & 0x7fffffff;
    if (lane == 0) p.part[(size_t)slot * p.nchunks + chunk] = x;
  }
}

// Completion of the streaming pass for the decision modes (greedy, coupled
// noise), one CTA per sequence, launched as its programmatic dependent (every
// chunk record is written once the streaming grid has completed): each warp
// merges verified rows of the sequence (first argmax over the chunks), then
// warp 0 walks the stages.  A sequence the streaming pass rejected (sizes, stage
// map, coupled-noise rows) has no records: it is skipped here too.
constexpr int kFinWarps = 16;

template <int MODE, typename T>
__global__ void __launch_bounds__(kFinWarps * 32) accept_finish_kernel(const AcceptParams p) {
  __shared__ WalkSmem walk;
  __shared__ int s_ok;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int b = blockIdx.x;
  // Before the wait: the call's inputs (the streaming kernel writes none of
  // them, and it lets this kernel start only after its own wait) -- the
  // sequence's validity and the stages of the rows each warp merges.
  const int off = p.slot_off[b], B = p.block[b], g = p.gamma[b];
  const bool sizes = off >= 0 && B >= 1 && B <= 64 && g >= 0 && g <= B && off + B <= p.total_slots;
  const int need = sizes ? min(g + 1, B) : 0;
  int st[64 / kFinWarps];
#pragma unroll
  for (int k = 0; k < 64 / kFinWarps; ++k) {
    const int j = warp + k * kFinWarps;
    st[k] = (sizes && j < B) ? p.tau[off + j] : 0;
  }
  if (warp == 0) {
    bool ok = sizes && warp_seq_valid(p, b);
    if (ok && MODE == SSV_ACCEPT_GUMBEL) {
      bool bad = false;
      for (int j = lane; j < B; j += 32) {
        const int t = p.tau[off + j];
        if (t >= 1 && t <= need) {
          const int nr = p.noise_row[off + j];
          bad = bad || nr < 0 || nr >= p.n_noise_rows;
        }
      }
      ok = !__any_sync(0xffffffffu, bad);
    }
    if (lane == 0) s_ok = ok ? 1 : 0;
  }
  __syncthreads();
  pdl_wait();  // every chunk record of the streaming pass
  pdl_trigger();
  if (!s_ok) return;
#pragma unroll
  for (int k = 0; k < 64 / kFinWarps; ++k) {  // warp-uniform
    const int j = warp + k * kFinWarps;
    if (j < B && st[k] >= 1 && st[k] <= need) warp_row_merge<MODE, T>(p, off + j, st[k], g);
  }
  __syncthreads();  // every row result of the sequence written
  if (warp == 0) warp_seq_walk<MODE>(p, b, off, B, g, walk, nullptr);
}

// Completion under rejection sampling, where a row merge also reads the
// draft token's two logits and forms the normalisers (double-float): every
// verified row of every sequence at once, one warp per slot and few warps per
// CTA, so the merges are spread over the SMs; the last merged row of a
// sequence (an arrival count) walks it.
constexpr int kMergeWarps = 4;

template <int MODE, typename T>
__global__ void __launch_bounds__(kMergeWarps * 32) accept_rowmerge_kernel(const AcceptParams p) {
  __shared__ WalkSmem walk[kMergeWarps];
  const int warp = threadIdx.x >> 5;
  const int slot = blockIdx.x * kMergeWarps + warp;
  // Before the wait: the call's inputs only (the streaming kernel writes none
  // of them, and it lets this kernel start only after its own wait) -- the
  // sequence's validity, the row's stage, its draft token and that token's
  // two logits.
  int b = -1, off = 0, B = 0, g = 0, need = 0, st = 0;
  bool mine = false;
  RowInputs in{-1, 0.f, 0.f, 0.f};
  if (slot < p.total_slots) {
    b = find_seq_by_slot(p.slot_off, p.batch, slot);
    if (b >= 0 && warp_seq_valid(p, b)) {
      off = p.slot_off[b];
      B = p.block[b];
      g = p.gamma[b];
      need = min(g + 1, B);
      st = slot < off + B ? p.tau[slot] : 0;
      mine = st >= 1 && st <= need;
      if (mine) in = row_inputs<T>(p, slot, st <= g);
    }
  }
  pdl_wait();  // every chunk record of the streaming pass
  pdl_trigger();
  if (!mine) return;
  warp_row_merge<MODE, T>(p, slot, st, g, &in);
  if (!warp_arrive(&p.cnt_seq[b], 1, need)) return;
  warp_seq_walk<MODE>(p, b, off, B, g, walk[warp], nullptr);
  if ((threadIdx.x & 31) == 0 && need != 1) p.cnt_seq[b] = 0;
}

int device_sm_count() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  return n;
}

template <int MODE, typename T>
cudaError_t launch_t(const AcceptParams& p, cudaStream_t st) {
  using C = StrCfg<MODE, T>;
  static std::once_flag once;
  static cudaError_t attr_err = cudaSuccess;
  std::call_once(once, [] {
    attr_err = cudaFuncSetAttribute(accept_stream_kernel<MODE, T>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    C::kSmem);
  });
  if (attr_err != cudaSuccess) return attr_err;
  const long long units = (long long)p.total_slots * p.nchunks;
  const int sms = device_sm_count();
  if (sms <= 0) return cudaErrorInvalidDevice;
  const int grid = (int)(units < sms ? units : sms);
  cudaError_t e = launch_pdl(accept_stream_kernel<MODE, T>, dim3(grid), dim3(kStrThreads), C::kSmem, st, p);
  if (e != cudaSuccess || p.batch == 0) return e;
  if (MODE != SSV_ACCEPT_REJECT)
    return launch_pdl(accept_finish_kernel<MODE, T>, dim3(p.batch), dim3(kFinWarps * 32), 0, st, p);
  return launch_pdl(accept_rowmerge_kernel<MODE, T>, dim3((p.total_slots + kMergeWarps - 1) / kMergeWarps),
                    dim3(kMergeWarps * 32), 0, st, p);
}

}  // namespace

bool accept_stream_supported(const AcceptParams& p, int mode, bool bf16) {
  const size_t es = bf16 ? 2 : 4;
  if (p.total_slots > kStrMaxRows || p.batch > kStrMaxRows) return false;
  if (((size_t)p.V * es) % 16 != 0 || ((uintptr_t)p.logits & 15u)) return false;
  if (mode == SSV_ACCEPT_REJECT && ((uintptr_t)p.draft_logits & 15u)) return false;
  if (mode == SSV_ACCEPT_GUMBEL && (((size_t)p.V * 4) % 16 != 0 || ((uintptr_t)p.noise & 15u))) return false;
  return device_sm_count() > 0;
}

cudaError_t launch_accept_stream(const AcceptParams& p, int mode, bool bf16, cudaStream_t st) {
  switch (mode) {
    case SSV_ACCEPT_ARGMAX:
      return bf16 ? launch_t<SSV_ACCEPT_ARGMAX, __nv_bfloat16>(p, st) : launch_t<SSV_ACCEPT_ARGMAX, float>(p, st);
    case SSV_ACCEPT_GUMBEL:
      return bf16 ? launch_t<SSV_ACCEPT_GUMBEL, __nv_bfloat16>(p, st) : launch_t<SSV_ACCEPT_GUMBEL, float>(p, st);
    case SSV_ACCEPT_GUMBEL_GEN:
      return bf16 ? launch_t<SSV_ACCEPT_GUMBEL_GEN, __nv_bfloat16>(p, st)
                  : launch_t<SSV_ACCEPT_GUMBEL_GEN, float>(p, st);
    default:
      return bf16 ? launch_t<SSV_ACCEPT_REJECT, __nv_bfloat16>(p, st) : launch_t<SSV_ACCEPT_REJECT, float>(p, st);
  }
}

}  // namespace ssv
