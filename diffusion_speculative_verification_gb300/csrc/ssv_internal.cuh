// Internal helpers shared by the libssv translation units (device + host).
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include "../../include/ssv.h"

namespace ssv {

// ---------------------------------------------------------------------------
// status
// ---------------------------------------------------------------------------
__device__ __forceinline__ void report(int32_t* dev_status, int32_t code) {
  if (dev_status) atomicCAS(dev_status, 0, code);
}

// ---------------------------------------------------------------------------
// element conversion
// ---------------------------------------------------------------------------
template <typename T> struct Elem;
template <> struct Elem<float> {
  static __device__ __forceinline__ float load(const float* p) { return *p; }
  static __device__ __forceinline__ float to_f32(float x) { return x; }
  static __device__ __forceinline__ float from_f32(float x) { return x; }
};
template <> struct Elem<__nv_bfloat16> {
  static __device__ __forceinline__ float load(const __nv_bfloat16* p) { return __bfloat162float(*p); }
  static __device__ __forceinline__ float to_f32(__nv_bfloat16 x) { return __bfloat162float(x); }
  static __device__ __forceinline__ __nv_bfloat16 from_f32(float x) { return __float2bfloat16_rn(x); }
};

// ---------------------------------------------------------------------------
// sequence lookup: sequences are packed in increasing q_off order
// ---------------------------------------------------------------------------
__device__ __forceinline__ int find_seq_by_row(const ssv_seq* seqs, int batch, int row) {
  int lo = 0, hi = batch - 1, ans = -1;
  while (lo <= hi) {
    int mid = (lo + hi) >> 1;
    if (seqs[mid].q_off <= row) { ans = mid; lo = mid + 1; } else { hi = mid - 1; }
  }
  return ans;
}

__device__ __forceinline__ int find_seq_by_slot(const int32_t* slot_off, int batch, int slot) {
  int lo = 0, hi = batch - 1, ans = -1;
  while (lo <= hi) {
    int mid = (lo + hi) >> 1;
    if (slot_off[mid] <= slot) { ans = mid; lo = mid + 1; } else { hi = mid - 1; }
  }
  return ans;
}

// ---------------------------------------------------------------------------
// temporal attention rule on the 2B tail keys (SimSD summary, section 2).
// r, t in [0, 2B): rows/keys D_1..D_B then D~_1..D~_B; tau_r / tau_t are the
// stages of their slots.
// ---------------------------------------------------------------------------
__device__ __forceinline__ bool tail_allowed(int r, int t, int B, int tau_r, int tau_t) {
  const bool row_mask = r >= B;
  const bool key_mask = t >= B;
  if (!row_mask) return !key_mask && tau_t <= tau_r;      // data row: revealed data only
  return key_mask ? (tau_t >= tau_r) : (tau_t < tau_r);   // mask row
}

// Checks that tau[0..B) is a permutation of 1..B.  Executed by one warp
// (all 32 lanes must call); returns the same answer on every lane.
__device__ __forceinline__ bool warp_tau_is_permutation(const int32_t* tau, int B) {
  const int lane = threadIdx.x & 31;
  unsigned long long seen = 0ull;
  bool ok = true;
  for (int j = lane; j < B; j += 32) {
    int t = tau[j];
    if (t < 1 || t > B) ok = false; else seen |= 1ull << (t - 1);
  }
  for (int o = 16; o > 0; o >>= 1) {
    seen |= __shfl_xor_sync(0xffffffffu, seen, o);
  }
  ok = __all_sync(0xffffffffu, ok);
  const unsigned long long full = (B >= 64) ? ~0ull : ((1ull << B) - 1ull);
  return ok && seen == full;
}

// The extents of sequence s lie inside the call's buffers: rows
// [q_off, q_off + N + 2B) of the query-side arrays, cache rows
// [kv_off, kv_off + C) and stage-map entries [tau_off, tau_off + B).  The
// attention kernels check this on the device before touching a sequence and
// skip (and report) one that fails.
__host__ __device__ __forceinline__ bool seq_extents_ok(const ssv_seq& s, int total_rows, int total_cache,
                                                        int total_slots) {
  return s.cache_len >= 0 && s.new_len >= 0 && s.block >= 1 && s.block <= 64 && s.q_off >= 0 &&
         (long long)s.q_off + s.new_len + 2LL * s.block <= (long long)total_rows && s.kv_off >= 0 &&
         (long long)s.kv_off + s.cache_len <= (long long)total_cache && s.tau_off >= 0 &&
         (long long)s.tau_off + s.block <= (long long)total_slots;
}

inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Bounded waits give up after this many SM cycles (about one second).
constexpr long long kDefaultWaitBudget = 1ll << 31;

// Test support (ssv_set_fault_injection): the wait budget and the index of
// the copy that CTA 0 leaves out, for a launch of `kernel` (an
// ssv_fault_kernel); {kDefaultWaitBudget, -1} unless that kernel is the one
// chosen.  Read on the host at launch time.
struct FaultSetting {
  long long budget;
  int skip;
};
FaultSetting fault_for(int kernel);

// host-side pieces shared by the entry points (validation, launches with the
// early-read flag of programmatic dependent launch)
ssv_status rope_validate(const ssv_rope_args* a);
ssv_status accept_validate(const ssv_accept_args* a, void* ws, size_t ws_bytes);
ssv_status accept_run(const ssv_accept_args* a, void* ws, size_t ws_bytes, cudaStream_t s, int early);

// ---------------------------------------------------------------------------
// programmatic dependent launch (PDL)
//
// The kernels of the verification step are launched with programmatic
// stream serialisation: a kernel may start while the kernel before it on
// the stream is still running.  pdl_wait() waits for that kernel to
// complete with its memory visible; a kernel reads no input and writes no
// workspace before it, except on an "early" launch inside ssv_verify_step,
// where the host has checked that the preceding kernel of the step writes
// none of the inputs read early.  pdl_trigger() lets the next kernel launch;
// each kernel triggers only once every kernel before it has completed, or on
// an early launch once the step's own predecessor is the only one running,
// so that early reads never overlap work from before the step.  Without the
// launch attribute both are no-ops.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                              Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

}  // namespace ssv

#define SSV_CUDA_CHECK(expr)                                   \
  do {                                                         \
    cudaError_t e_ = (expr);                                   \
    if (e_ != cudaSuccess) return SSV_ERR_CUDA;                \
  } while (0)
