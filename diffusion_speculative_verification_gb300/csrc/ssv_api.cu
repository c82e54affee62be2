// Host side of libssv: argument validation, schedule selection for the
// verification attention, status handling.
#include "ssv_internal.cuh"
#include "attn.cuh"

#include <math.h>
#include <string.h>

#include <atomic>

using namespace ssv;

// ---------------------------------------------------------------------------
// test support: fault injection without a GPU fault (ssv_set_fault_injection)
// ---------------------------------------------------------------------------
namespace {
std::atomic<int> g_fault_kernel{SSV_FAULT_NONE};
std::atomic<int> g_fault_skip{-1};
std::atomic<long long> g_fault_budget{kDefaultWaitBudget};
}  // namespace

namespace ssv {
FaultSetting fault_for(int kernel) {
  if (kernel == SSV_FAULT_NONE || g_fault_kernel.load() != kernel) return {kDefaultWaitBudget, -1};
  return {g_fault_budget.load(), g_fault_skip.load()};
}
}  // namespace ssv

extern "C" ssv_status ssv_set_fault_injection(const ssv_fault_injection* f) {
  if (!f) {
    g_fault_kernel = SSV_FAULT_NONE;
    g_fault_skip = -1;
    g_fault_budget = kDefaultWaitBudget;
    return SSV_OK;
  }
  if (f->kernel < SSV_FAULT_NONE || f->kernel > SSV_FAULT_LMHEAD || f->skip < -1 || f->wait_budget_cycles < 1000 ||
      f->wait_budget_cycles > kDefaultWaitBudget)
    return SSV_ERR_INVALID;
  g_fault_budget = f->wait_budget_cycles;
  g_fault_skip = f->skip;
  g_fault_kernel = f->kernel;
  return SSV_OK;
}

namespace {

ssv_status attn_check(const ssv_attn_args* a) {
  if (!a) return SSV_ERR_INVALID;
  if (a->batch < 0 || a->total_rows < 0 || a->total_cache < 0 || a->total_slots < 0) return SSV_ERR_INVALID;
  if (a->Hq <= 0 || a->Hkv <= 0 || a->Hq % a->Hkv != 0) return SSV_ERR_INVALID;
  if (a->d != 64 && a->d != 128) return SSV_ERR_UNSUPPORTED;
  if (a->in_dtype != SSV_F32 && a->in_dtype != SSV_BF16) return SSV_ERR_INVALID;
  if (a->out_dtype != SSV_F32 && a->out_dtype != SSV_BF16) return SSV_ERR_INVALID;
  if (a->in_dtype == SSV_F32 && a->out_dtype != SSV_F32) return SSV_ERR_UNSUPPORTED;
  if (a->max_block < 1 || a->max_block > 64 || a->max_cache < 0 || a->max_new < 0) return SSV_ERR_INVALID;
  if (!isfinite(a->scale) || a->scale < 0.f) return SSV_ERR_INVALID;
  if (a->batch == 0 || a->total_rows == 0) return SSV_OK;
  if (!a->q || !a->k_new || !a->v_new || !a->o || !a->seqs || !a->tau) return SSV_ERR_INVALID;
  if (a->total_cache > 0 && (!a->k_cache || !a->v_cache)) return SSV_ERR_INVALID;
  const uintptr_t al = (uintptr_t)a->q | (uintptr_t)a->k_cache | (uintptr_t)a->v_cache | (uintptr_t)a->k_new |
                       (uintptr_t)a->v_new | (uintptr_t)a->o;
  if (al & 15u) return SSV_ERR_INVALID;
  return SSV_OK;
}

AttnParams to_params(const ssv_attn_args* a) {
  AttnParams p;
  p.q = a->q;
  p.k_cache = a->k_cache;
  p.v_cache = a->v_cache;
  p.k_new = a->k_new;
  p.v_new = a->v_new;
  p.o = a->o;
  p.in_dtype = a->in_dtype;
  p.out_dtype = a->out_dtype;
  p.Hq = a->Hq;
  p.Hkv = a->Hkv;
  p.d = a->d;
  p.scale = a->scale > 0.f ? a->scale : (float)(1.0 / sqrt((double)a->d));
  p.seqs = a->seqs;
  p.batch = a->batch;
  p.tau = a->tau;
  p.total_rows = a->total_rows;
  p.total_cache = a->total_cache;
  p.total_slots = a->total_slots;
  p.max_cache = a->max_cache;
  p.max_new = a->max_new;
  p.max_block = a->max_block;
  p.dev_status = a->dev_status;
  p.early = 0;
  const FaultSetting f = fault_for(SSV_FAULT_ATTN);
  p.wait_budget = f.budget;
  p.fault_skip = f.skip;
  p.prompt_only = 0;
  p.total_krows = a->total_rows;
  p.lse = nullptr;
  return p;
}

}  // namespace

extern "C" ssv_status ssv_verify_attn_workspace(const ssv_attn_args* a, size_t* bytes) {
  if (!bytes) return SSV_ERR_INVALID;
  const ssv_status st = attn_check(a);
  if (st != SSV_OK) return st;
  *bytes = 256;
  if (a->batch > 0 && a->total_rows > 0) {
    const AttnParams p = to_params(a);
    if (tc::attn_tc_supported(p)) *bytes = tc::attn_tc_workspace(p);
  }
  return SSV_OK;
}

namespace {

ssv_status attn_validate(const ssv_attn_args* a, void* ws, size_t ws_bytes) {
  const ssv_status st = attn_check(a);
  if (st != SSV_OK) return st;
  if (a->batch == 0 || a->total_rows == 0) return SSV_OK;
  size_t need = 0;
  ssv_verify_attn_workspace(a, &need);
  if (need > 0 && (!ws || ((uintptr_t)ws & 255u) || ws_bytes < need)) return SSV_ERR_WORKSPACE;
  return SSV_OK;
}

ssv_status attn_run(const ssv_attn_args* a, void* ws, size_t ws_bytes, cudaStream_t s, int early) {
  const ssv_status st = attn_validate(a, ws, ws_bytes);
  if (st != SSV_OK) return st;
  if (a->batch == 0 || a->total_rows == 0) return SSV_OK;
  AttnParams p = to_params(a);
  p.early = early;
  const cudaError_t e = tc::attn_tc_supported(p) ? tc::launch_attn_tc(p, ws, s) : launch_attn_simt(p, s);
  return e == cudaSuccess ? SSV_OK : SSV_ERR_CUDA;
}

// byte ranges [a, a + na) and [b, b + nb) intersect
bool overlap(const void* a, size_t na, const void* b, size_t nb) {
  if (!a || !b || na == 0 || nb == 0) return false;
  const uintptr_t x = (uintptr_t)a, y = (uintptr_t)b;
  return x < y + nb && y < x + na;
}

size_t esize(ssv_dtype t) { return t == SSV_BF16 ? 2 : 4; }

}  // namespace

extern "C" ssv_status ssv_verify_attn(const ssv_attn_args* a, void* ws, size_t ws_bytes, void* stream) {
  return attn_run(a, ws, ws_bytes, static_cast<cudaStream_t>(stream), 0);
}

extern "C" ssv_status ssv_verify_step(const ssv_rope_args* rope, const ssv_attn_args* attn, void* attn_ws,
                                      size_t attn_ws_bytes, const ssv_accept_args* acc, void* acc_ws,
                                      size_t acc_ws_bytes, void* stream) {
  if (!attn) return SSV_ERR_INVALID;
  ssv_status st;
  if (rope && (st = rope_validate(rope)) != SSV_OK) return st;
  if ((st = attn_validate(attn, attn_ws, attn_ws_bytes)) != SSV_OK) return st;
  if (acc && (st = accept_validate(acc, acc_ws, acc_ws_bytes)) != SSV_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // What each kernel may read before its predecessor completes, and what the
  // predecessors write.
  size_t rq = 0, rk = 0;
  if (rope) {
    const size_t e = rope->dtype == SSV_BF16 ? 2 : 4;
    rq = (size_t)rope->total_rows * rope->Hq * rope->d * e;
    rk = (size_t)rope->total_rows * rope->Hkv * rope->d * e;
  }
  auto written_by_rope = [&](const void* p, size_t n) {
    return rope && (overlap(rope->q_out, rq, p, n) || overlap(rope->k_out, rk, p, n));
  };
  const size_t cache_bytes = (size_t)attn->total_cache * attn->Hkv * attn->d * esize(attn->in_dtype);
  const int early_attn =
      rope && !written_by_rope(attn->seqs, sizeof(ssv_seq) * (size_t)attn->batch) &&
      !written_by_rope(attn->tau, sizeof(int32_t) * (size_t)attn->total_slots) &&
      !written_by_rope(attn->k_cache, cache_bytes) && !written_by_rope(attn->v_cache, cache_bytes);
  int early_acc = 0;
  if (acc) {
    const size_t ob = (size_t)attn->total_rows * attn->Hq * attn->d * esize(attn->out_dtype);
    const void* meta[5] = {acc->tau, acc->block, acc->gamma, acc->slot_off, acc->noise_row};
    const size_t mb[5] = {4 * (size_t)acc->total_slots, 4 * (size_t)acc->batch, 4 * (size_t)acc->batch,
                          4 * (size_t)acc->batch, acc->noise_row ? 4 * (size_t)acc->total_slots : 0};
    early_acc = 1;
    for (int i = 0; i < 5; ++i)
      if (written_by_rope(meta[i], mb[i]) || overlap(attn->o, ob, meta[i], mb[i]) ||
          overlap(attn_ws, attn_ws_bytes, meta[i], mb[i]))
        early_acc = 0;
  }
  if (rope && (st = ssv_rope_copy(rope, stream)) != SSV_OK) return st;
  if ((st = attn_run(attn, attn_ws, attn_ws_bytes, s, early_attn)) != SSV_OK) return st;
  if (acc && (st = accept_run(acc, acc_ws, acc_ws_bytes, s, early_acc)) != SSV_OK) return st;
  return SSV_OK;
}

extern "C" ssv_status ssv_get_status(int32_t* dev_status, void* stream) {
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (!dev_status) {
    return cudaStreamSynchronize(s) == cudaSuccess ? SSV_OK : SSV_ERR_CUDA;
  }
  int32_t h = 0;
  if (cudaMemcpyAsync(&h, dev_status, sizeof(h), cudaMemcpyDeviceToHost, s) != cudaSuccess) return SSV_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return SSV_ERR_CUDA;
  if (h != 0) {
    if (cudaMemsetAsync(dev_status, 0, sizeof(int32_t), s) != cudaSuccess) return SSV_ERR_CUDA;
    if (cudaStreamSynchronize(s) != cudaSuccess) return SSV_ERR_CUDA;
  }
  return static_cast<ssv_status>(h);
}

extern "C" const char* ssv_status_string(ssv_status s) {
  switch (s) {
    case SSV_OK: return "ok";
    case SSV_ERR_INVALID: return "invalid argument";
    case SSV_ERR_UNSUPPORTED: return "unsupported configuration";
    case SSV_ERR_CUDA: return "CUDA error";
    case SSV_ERR_TIMEOUT: return "bounded device wait ran out";
    case SSV_ERR_BAD_TAU: return "stage map is not a permutation of 1..B";
    case SSV_ERR_WORKSPACE: return "workspace missing, misaligned or too small";
    case SSV_ERR_NOT_FINITE: return "temperature not finite or negative";
  }
  return "unknown status";
}

extern "C" const char* ssv_version(void) { return "ssv 0.2 sm_103a"; }
