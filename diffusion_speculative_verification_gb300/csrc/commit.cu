// Commit of a verification pass into the KV cache (ssv_commit).
//
// SimSD summary, section 4 "Speculative decoding pipeline" (Acceptance: the
// longest accepted prefix, in the temporal order the draft induces, is
// committed and the loop repeats) and "Main contributions" 3 (the method
// composes with a KV cache).  Sequence b's cache gains, after its C rows, its
// N fresh prompt rows in row order and then the data rows of stages
// 1..n_acc in stage order; mask rows are never committed.
//
// One warp per sequence reports a rejected sequence and writes its new length;
// one warp per fresh row finds its sequence, checks it the same way (stage map
// a permutation of 1..B, n_acc within 0..B, room in the destination), computes
// the row's destination
// (prompt row i -> C + i, data row of stage s <= n_acc -> C + N + s - 1, mask
// row -> none) and moves the key and value rows as 16-byte vectors,
// consecutive lanes on consecutive vectors, loads issued ahead of the stores.
// HBM-bound: reads and writes 2 (K, V) x (N + n_acc) rows x Hkv x d elements
// per sequence.
#include "ssv_internal.cuh"

namespace ssv {
namespace {

constexpr int kCommitWarps = 8;
constexpr int kCommitBatch = 4;  // 16-byte vectors of K and of V in flight per lane

struct CommitParams {
  const uint8_t* k_new;
  const uint8_t* v_new;
  uint8_t* k_dst;
  uint8_t* v_dst;
  const ssv_seq* seqs;
  const int32_t* tau;
  const int32_t* n_acc;
  const int32_t* dst_off;
  const int32_t* dst_cap;
  int32_t* new_len;
  int32_t* dev_status;
  int batch, total_rows, total_slots, dst_rows;
  uint32_t row_bytes;  // Hkv * d * element size, a multiple of 16
};

// Checks sequence b (executed by a whole warp, same answer on every lane):
// 0 if it may be committed, else the status to report.
__device__ __forceinline__ int32_t commit_check(const CommitParams& p, int b, const ssv_seq& s) {
  const int B = s.block, N = s.new_len, C = s.cache_len;
  if (B < 1 || B > 64 || s.tau_off < 0 || (long long)s.tau_off + B > p.total_slots) return SSV_ERR_INVALID;
  if (!warp_tau_is_permutation(p.tau + s.tau_off, B)) return SSV_ERR_BAD_TAU;
  const int na = p.n_acc[b], off = p.dst_off[b], cap = p.dst_cap[b];
  const bool sizes = na >= 0 && na <= B && C >= 0 && N >= 0 && off >= 0 && cap >= 0 &&
                     (long long)C + N + na <= cap && (long long)off + cap <= p.dst_rows;
  return sizes ? 0 : SSV_ERR_INVALID;
}

// warps [0, total_rows): one fresh row each; warps [total_rows, total_rows + batch):
// one sequence each (status and new length)
__global__ void __launch_bounds__(32 * kCommitWarps) commit_kernel(const CommitParams p) {
  pdl_wait();  // n_acc and the fresh rows may come from the kernels before this one
  pdl_trigger();
  const int lane = threadIdx.x & 31;
  const long long w = (long long)blockIdx.x * kCommitWarps + (threadIdx.x >> 5);
  if (w >= p.total_rows) {
    const long long bb = w - p.total_rows;
    if (bb >= p.batch) return;
    const int b = (int)bb;
    const ssv_seq s = p.seqs[b];
    const int32_t bad = commit_check(p, b, s);
    if (lane == 0) {
      if (bad) report(p.dev_status, bad);
      p.new_len[b] = bad ? -1 : s.cache_len + s.new_len + p.n_acc[b];
    }
    return;
  }
  const int row = (int)w;
  // the sequence holding the row: the last one with q_off <= row (sequences are
  // packed in increasing q_off)
  int lo = 0, hi = p.batch - 1, b = -1;
  while (lo <= hi) {
    const int mid = (lo + hi) >> 1;
    if (p.seqs[mid].q_off <= row) { b = mid; lo = mid + 1; } else { hi = mid - 1; }
  }
  if (b < 0) return;
  const ssv_seq s = p.seqs[b];
  const int i = row - s.q_off;
  if (i >= s.new_len + 2 * s.block) return;  // a row between sequences
  if (commit_check(p, b, s)) return;
  const int B = s.block, N = s.new_len, C = s.cache_len;
  const int na = p.n_acc[b], off = p.dst_off[b];
  int dst;
  if (i < N) {
    dst = C + i;  // fresh prompt row
  } else if (i < N + B) {
    const int st = p.tau[s.tau_off + (i - N)];  // data row of slot i - N
    if (st > na) return;                        // stage not accepted
    dst = C + N + st - 1;
  } else {
    return;  // mask row
  }
  const uint8_t* ks = p.k_new + (size_t)row * p.row_bytes;
  const uint8_t* vs = p.v_new + (size_t)row * p.row_bytes;
  uint8_t* kd = p.k_dst + ((size_t)off + dst) * p.row_bytes;
  uint8_t* vd = p.v_dst + ((size_t)off + dst) * p.row_bytes;
  constexpr uint32_t kStep = 32u * 16u;
  for (uint32_t o0 = lane * 16u; o0 < p.row_bytes; o0 += kCommitBatch * kStep) {
    uint4 kx[kCommitBatch], vx[kCommitBatch];
#pragma unroll
    for (int t = 0; t < kCommitBatch; ++t) {
      const uint32_t o = o0 + t * kStep;
      if (o < p.row_bytes) {
        kx[t] = *reinterpret_cast<const uint4*>(ks + o);
        vx[t] = *reinterpret_cast<const uint4*>(vs + o);
      }
    }
#pragma unroll
    for (int t = 0; t < kCommitBatch; ++t) {
      const uint32_t o = o0 + t * kStep;
      if (o < p.row_bytes) {
        *reinterpret_cast<uint4*>(kd + o) = kx[t];
        *reinterpret_cast<uint4*>(vd + o) = vx[t];
      }
    }
  }
}

bool ranges_overlap(const void* a, size_t an, const void* b, size_t bn) {
  const uintptr_t a0 = reinterpret_cast<uintptr_t>(a), b0 = reinterpret_cast<uintptr_t>(b);
  return an > 0 && bn > 0 && a0 < b0 + bn && b0 < a0 + an;
}

}  // namespace
}  // namespace ssv

extern "C" ssv_status ssv_commit(const ssv_commit_args* a, void* stream) {
  using namespace ssv;
  if (!a) return SSV_ERR_INVALID;
  if (a->batch < 0 || a->total_rows < 0 || a->total_slots < 0 || a->dst_rows < 0 || a->Hkv <= 0)
    return SSV_ERR_INVALID;
  if (a->dtype != SSV_F32 && a->dtype != SSV_BF16) return SSV_ERR_INVALID;
  if (a->d != 64 && a->d != 128) return SSV_ERR_UNSUPPORTED;
  if (a->batch == 0) return SSV_OK;
  if (!a->k_new || !a->v_new || !a->k_dst || !a->v_dst || !a->seqs || !a->tau || !a->n_acc || !a->dst_off ||
      !a->dst_cap || !a->new_len)
    return SSV_ERR_INVALID;
  const uintptr_t al = (uintptr_t)a->k_new | (uintptr_t)a->v_new | (uintptr_t)a->k_dst | (uintptr_t)a->v_dst;
  if (al & 15u) return SSV_ERR_INVALID;
  const size_t row_bytes = (size_t)a->Hkv * a->d * (a->dtype == SSV_BF16 ? 2 : 4);
  if (row_bytes > 0x7fffffffu) return SSV_ERR_INVALID;
  const size_t src_bytes = row_bytes * a->total_rows, dst_bytes = row_bytes * a->dst_rows;
  if (ranges_overlap(a->k_new, src_bytes, a->k_dst, dst_bytes) || ranges_overlap(a->k_new, src_bytes, a->v_dst, dst_bytes) ||
      ranges_overlap(a->v_new, src_bytes, a->k_dst, dst_bytes) || ranges_overlap(a->v_new, src_bytes, a->v_dst, dst_bytes))
    return SSV_ERR_INVALID;
  CommitParams p;
  p.k_new = static_cast<const uint8_t*>(a->k_new);
  p.v_new = static_cast<const uint8_t*>(a->v_new);
  p.k_dst = static_cast<uint8_t*>(a->k_dst);
  p.v_dst = static_cast<uint8_t*>(a->v_dst);
  p.seqs = a->seqs;
  p.tau = a->tau;
  p.n_acc = a->n_acc;
  p.dst_off = a->dst_off;
  p.dst_cap = a->dst_cap;
  p.new_len = a->new_len;
  p.dev_status = a->dev_status;
  p.batch = a->batch;
  p.total_rows = a->total_rows;
  p.total_slots = a->total_slots;
  p.dst_rows = a->dst_rows;
  p.row_bytes = (uint32_t)row_bytes;
  const long long warps = (long long)a->total_rows + a->batch;
  const unsigned grid = (unsigned)((warps + kCommitWarps - 1) / kCommitWarps);
  const cudaError_t e =
      launch_pdl(commit_kernel, dim3(grid), dim3(32 * kCommitWarps), 0, static_cast<cudaStream_t>(stream), p);
  return e == cudaSuccess ? SSV_OK : SSV_ERR_CUDA;
}
