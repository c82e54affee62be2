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
  // Prompt-only pass (the tree pass's shared prefix, tensor-core schedule
  // only): a sequence has N prompt rows and `block` further query rows, each
  // of which sees the whole prompt (cache + N fresh keys) and nothing else;
  // no stage map is read.  Its fresh keys are rows [tau_off, tau_off + N) of
  // k_new / v_new (total_krows rows), its query and output rows [q_off,
  // q_off + N + block) of q / o (total_rows rows).  lse (when not null):
  // [total_rows][Hq] log2-sum-exp2 of the scaled scores (scale * log2 e) of
  // each output row, -inf for a row that saw no key.
  int prompt_only;
  int total_krows;
  float* lse;
};

cudaError_t launch_attn_simt(const AttnParams& p, cudaStream_t st);

namespace tc {
bool attn_tc_supported(const AttnParams& p);
size_t attn_tc_workspace(const AttnParams& p);
// ws: attn_tc_workspace(p) bytes, 256-byte aligned, counter area zero on entry (left zero on exit)
cudaError_t launch_attn_tc(const AttnParams& p, void* ws, cudaStream_t st);
}  // namespace tc

}  // namespace ssv
