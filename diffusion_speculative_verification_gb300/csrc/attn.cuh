// Verify-attention launch parameters shared by the SIMT and tensor-core
// schedules, and the host entry points of each schedule.
#pragma once

#include "ssv_internal.cuh"

namespace ssv {

struct AttnParams {
  const void* q;
  const void* k_cache;
  const void* v_cache;
  const void* k_new;
  const void* v_new;
  void* o;
  ssv_dtype in_dtype, out_dtype;
  int Hq, Hkv, d;
  float scale;  // softmax scale (1/sqrt(d) unless given)
  const ssv_seq* seqs;
  int batch;
  const int32_t* tau;
  int total_rows, total_cache, total_slots;
  int max_cache, max_new, max_block;
  int32_t* dev_status;
  // 1: the kernel before this one on the stream is the step's rotation kernel,
  // whose outputs overlap none of seqs, tau and the KV cache; those may then
  // be read before that kernel completes (programmatic dependent launch).
  int early;
  // bounded waits give up after wait_budget SM cycles; fault_skip >= 0 makes
  // CTA 0 leave out that key-block copy (test support, ssv_set_fault_injection)
  long long wait_budget;
  int fault_skip;
};

cudaError_t launch_attn_simt(const AttnParams& p, cudaStream_t st);

namespace tc {
bool attn_tc_supported(const AttnParams& p);
size_t attn_tc_workspace(const AttnParams& p);
// ws: attn_tc_workspace(p) bytes, 256-byte aligned, counter area zero on entry (left zero on exit)
cudaError_t launch_attn_tc(const AttnParams& p, void* ws, cudaStream_t st);
}  // namespace tc

}  // namespace ssv
