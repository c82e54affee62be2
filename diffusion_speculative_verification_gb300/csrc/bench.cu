// ssv_bench: native timing of the library on a named synthetic workload:
// rotation, verify attention, acceptance, the commit (each sequence appends
// its prompt rows and gamma / 2 accepted rows) and the fused LM head +
// acceptance (hidden width Hq * head_dim; greedy unless the workload uses
// coupled noise).
//
// Buffers are allocated here (this is a measurement utility, not a hot-path
// call) and filled on the device by a counter-hash generator (splitmix64
// finaliser + Box-Muller); values are only needed to have the right shapes
// and distributions, not to match any other generator.  Each op is timed
// with CUDA events on its stream, one launch per sample, with a 256 MB
// memset between samples so that inputs never start in the 129 MB L2.
#include "ssv_internal.cuh"

#include <algorithm>
#include <math.h>
#include <stdio.h>
#include <string.h>
#include <string>
#include <vector>

namespace {

__device__ __forceinline__ uint64_t mix64(uint64_t x) {
  x += 0x9E3779B97F4A7C15ull;
  x = (x ^ (x >> 30)) * 0xBF58476D1CE4E5B9ull;
  x = (x ^ (x >> 27)) * 0x94D049BB133111EBull;
  return x ^ (x >> 31);
}

__device__ __forceinline__ float unit_open(uint64_t h) {  // (0, 1)
  return ((float)(h >> 40) + 0.5f) * (1.0f / 16777216.0f);
}

template <typename T>
__global__ void fill_normal(T* p, size_t n, uint64_t seed, float std) {
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n; i += (size_t)gridDim.x * blockDim.x) {
    const float u1 = unit_open(mix64(seed ^ (2 * i)));
    const float u2 = unit_open(mix64(seed ^ (2 * i + 1)));
    const float z = sqrtf(-2.f * logf(u1)) * cospif(2.f * u2) * std;
    p[i] = ssv::Elem<T>::from_f32(z);
  }
}

__global__ void fill_gumbel(float* p, size_t n, uint64_t seed) {
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n; i += (size_t)gridDim.x * blockDim.x)
    p[i] = -logf(-logf(unit_open(mix64(seed ^ i))));
}

__global__ void fill_uniform(float* p, size_t n, uint64_t seed) {
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n; i += (size_t)gridDim.x * blockDim.x)
    p[i] = unit_open(mix64(seed ^ i)) * 0.999f;
}

__global__ void fill_tokens(int32_t* p, size_t n, uint64_t seed, int V) {
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n; i += (size_t)gridDim.x * blockDim.x)
    p[i] = (int32_t)(mix64(seed ^ i) % (uint64_t)V);
}

// Plain streaming read, the reference a kernel of the path that reads the same
// bytes is measured against: 16-byte loads, eight independent ones in flight
// per thread, two CTAs of 512 threads per SM, each CTA one contiguous range;
// the XOR of everything read goes to *out so that no load can be dropped.
__global__ void __launch_bounds__(512) stream_read_kernel(const uint4* __restrict__ buf, size_t n16, uint32_t* out) {
  const size_t per = (n16 + gridDim.x - 1) / gridDim.x;
  const size_t b = (size_t)blockIdx.x * per, e = (b + per < n16) ? b + per : n16;
  uint32_t acc = 0u;
  for (size_t i = b + threadIdx.x; i < e; i += (size_t)blockDim.x * 8) {
    uint4 v[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const size_t j = i + (size_t)u * blockDim.x;
      v[u] = j < e ? __ldcs(buf + j) : make_uint4(0u, 0u, 0u, 0u);
    }
#pragma unroll
    for (int u = 0; u < 8; ++u) acc ^= v[u].x ^ v[u].y ^ v[u].z ^ v[u].w;
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) acc ^= __shfl_xor_sync(0xffffffffu, acc, o);
  if ((threadIdx.x & 31) == 0 && acc) atomicXor(out, acc);
}

uint64_t host_mix(uint64_t x) {
  x += 0x9E3779B97F4A7C15ull;
  x = (x ^ (x >> 30)) * 0xBF58476D1CE4E5B9ull;
  x = (x ^ (x >> 27)) * 0x94D049BB133111EBull;
  return x ^ (x >> 31);
}

struct Cfg {
  const char* name;
  int batch, Hq, Hkv, d;
  ssv_dtype dt;
  int mode;
  float T;
  int V;
  int gamma;  // 0 = B
};

const Cfg kCfgs[] = {
    {"tiny", 1, 1, 1, 64, SSV_F32, SSV_ACCEPT_GUMBEL, 1.f, 256, 0},
    {"gqa1p7b", 8, 16, 8, 128, SSV_BF16, SSV_ACCEPT_ARGMAX, 0.f, 151936, 0},
    {"gqa8b", 16, 32, 8, 128, SSV_BF16, SSV_ACCEPT_REJECT, 1.f, 151936, 16},
    {"prefill", 4, 32, 8, 128, SSV_BF16, -1, 0.f, 151936, 0},
    {"sweep", 64, 32, 8, 128, SSV_BF16, SSV_ACCEPT_GUMBEL, 1.f, 151936, 0},
};

void lengths(const Cfg& c, int b, int* C, int* N, int* B) {
  const std::string n = c.name;
  *N = 0;
  if (n == "tiny") { *C = 16; *B = 4; }
  else if (n == "gqa1p7b") { *C = 1024; *B = 8; }
  else if (n == "gqa8b") { *C = 4096; *B = 32; }
  else if (n == "prefill") { *C = 0; *N = 8192; *B = 16; }
  else {
    const uint64_t h = host_mix(0x5eed0000ull + b);
    *C = 256 + (int)(h % (8192 - 256 + 1));
    static const int Bs[4] = {4, 8, 16, 32};
    *B = Bs[(h >> 32) & 3];
  }
}

struct Timing { double med, p10, p90; };

Timing summarize(std::vector<float>& v) {
  std::sort(v.begin(), v.end());
  auto at = [&](double q) { return (double)v[std::min(v.size() - 1, (size_t)(q * (v.size() - 1) + 0.5))]; };
  return {at(0.5) * 1e3, at(0.1) * 1e3, at(0.9) * 1e3};  // microseconds
}

}  // namespace

#define BENCH_CHECK(x)                                          \
  do {                                                          \
    if ((x) != cudaSuccess) { rc = SSV_ERR_CUDA; goto done; }   \
  } while (0)
#define BENCH_SSV(x)                                            \
  do {                                                          \
    ssv_status s_ = (x);                                        \
    if (s_ != SSV_OK) { rc = s_; goto done; }                   \
  } while (0)

extern "C" ssv_status ssv_bench(const char* config, int32_t iters, char* json_out, size_t json_len) {
  if (!config || !json_out || json_len < 64 || iters < 1) return SSV_ERR_INVALID;
  const Cfg* cfg = nullptr;
  for (const Cfg& c : kCfgs)
    if (strcmp(c.name, config) == 0) cfg = &c;
  if (!cfg) return SSV_ERR_INVALID;

  ssv_status rc = SSV_OK;
  const int batch = cfg->batch, Hq = cfg->Hq, Hkv = cfg->Hkv, d = cfg->d;
  const size_t es = cfg->dt == SSV_BF16 ? 2 : 4;
  std::vector<ssv_seq> seqs(batch);
  std::vector<int32_t> blocks(batch), gammas(batch), slot_off(batch), tau_h;
  int rows = 0, cache = 0, slots = 0, max_c = 0, max_n = 0, max_b = 0;
  double pairs = 0;
  for (int b = 0; b < batch; ++b) {
    int C, N, B;
    lengths(*cfg, b, &C, &N, &B);
    seqs[b] = {C, N, B, rows, cache, slots};
    blocks[b] = B;
    gammas[b] = cfg->gamma ? std::min(cfg->gamma, B) : B;
    slot_off[b] = slots;
    for (int k = 0; k < B; ++k) tau_h.push_back((int32_t)((k * 5 + b) % B) + 1);  // a permutation when gcd(5,B)=1
    rows += N + 2 * B;
    cache += C;
    slots += B;
    max_c = std::max(max_c, C); max_n = std::max(max_n, N); max_b = std::max(max_b, B);
    const double P = C + N;
    pairs += N * (N + 1) / 2.0 + (double)N * C + 2.0 * B * P + B * (B + 1) / 2.0 + (double)B * B;
  }
  // 5 is coprime to every block width used (4, 8, 16, 32): tau is a permutation.
  const double attn_flops = pairs * Hq * 4.0 * d;
  const double attn_bytes = (double)cache * Hkv * d * 2 * es + (double)rows * Hq * d * es +
                            (double)rows * Hkv * d * 2 * es + (double)rows * Hq * d * es;
  const double rope_bytes = 2.0 * rows * (Hq + Hkv) * d * es;

  void *q = nullptr, *kn = nullptr, *vn = nullptr, *kc = nullptr, *vc = nullptr, *o = nullptr;
  void *logits = nullptr, *dlogits = nullptr, *noise = nullptr, *flush = nullptr, *ws_a = nullptr, *ws_c = nullptr;
  ssv_seq* d_seqs = nullptr;
  int32_t *d_tau = nullptr, *d_blocks = nullptr, *d_gam = nullptr, *d_soff = nullptr, *d_draft = nullptr;
  int32_t *d_nrow = nullptr, *d_nacc = nullptr, *d_nout = nullptr, *d_tok = nullptr, *d_status = nullptr;
  float *d_ua = nullptr, *d_us = nullptr;
  cudaStream_t st = nullptr;
  cudaEvent_t e0 = nullptr, e1 = nullptr;
  std::vector<float> t_rope, t_attn, t_acc, t_commit, t_lm;
  void *k_dst = nullptr, *v_dst = nullptr, *lm_w = nullptr, *lm_h = nullptr, *ws_l = nullptr;
  int32_t *d_cnacc = nullptr, *d_doff = nullptr, *d_dcap = nullptr, *d_newlen = nullptr;
  double commit_bytes = 0, lm_bytes = 0, lm_flops = 0;
  size_t ws_lm = 0;
  const int hidden = Hq * d;
  ssv_commit_args ma;
  ssv_lmhead_accept_args la;
  memset(&ma, 0, sizeof(ma));
  memset(&la, 0, sizeof(la));
  const size_t flush_bytes = 256u << 20;
  const int V = cfg->V;
  double acc_bytes = 0;
  size_t ws_attn = 0, ws_acc = 0;
  ssv_rope_args ra;
  ssv_attn_args aa;
  ssv_accept_args ca;
  memset(&ra, 0, sizeof(ra));
  memset(&aa, 0, sizeof(aa));
  memset(&ca, 0, sizeof(ca));

  BENCH_CHECK(cudaStreamCreateWithFlags(&st, cudaStreamNonBlocking));
  BENCH_CHECK(cudaEventCreate(&e0));
  BENCH_CHECK(cudaEventCreate(&e1));
  BENCH_CHECK(cudaMalloc(&q, (size_t)rows * Hq * d * es));
  BENCH_CHECK(cudaMalloc(&kn, (size_t)rows * Hkv * d * es));
  BENCH_CHECK(cudaMalloc(&vn, (size_t)rows * Hkv * d * es));
  BENCH_CHECK(cudaMalloc(&kc, std::max<size_t>(16, (size_t)cache * Hkv * d * es)));
  BENCH_CHECK(cudaMalloc(&vc, std::max<size_t>(16, (size_t)cache * Hkv * d * es)));
  BENCH_CHECK(cudaMalloc(&o, (size_t)rows * Hq * d * es));
  BENCH_CHECK(cudaMalloc(&flush, flush_bytes));
  BENCH_CHECK(cudaMalloc((void**)&d_seqs, sizeof(ssv_seq) * batch));
  BENCH_CHECK(cudaMalloc((void**)&d_tau, sizeof(int32_t) * slots));
  BENCH_CHECK(cudaMalloc((void**)&d_status, sizeof(int32_t)));
  BENCH_CHECK(cudaMemsetAsync(d_status, 0, sizeof(int32_t), st));
  BENCH_CHECK(cudaMemcpyAsync(d_seqs, seqs.data(), sizeof(ssv_seq) * batch, cudaMemcpyHostToDevice, st));
  BENCH_CHECK(cudaMemcpyAsync(d_tau, tau_h.data(), sizeof(int32_t) * slots, cudaMemcpyHostToDevice, st));
  if (cfg->dt == SSV_BF16) {
    fill_normal<__nv_bfloat16><<<1024, 256, 0, st>>>((__nv_bfloat16*)q, (size_t)rows * Hq * d, 1, 1.f);
    fill_normal<__nv_bfloat16><<<1024, 256, 0, st>>>((__nv_bfloat16*)kn, (size_t)rows * Hkv * d, 2, 1.f);
    fill_normal<__nv_bfloat16><<<1024, 256, 0, st>>>((__nv_bfloat16*)vn, (size_t)rows * Hkv * d, 3, 1.f);
    fill_normal<__nv_bfloat16><<<1024, 256, 0, st>>>((__nv_bfloat16*)kc, (size_t)cache * Hkv * d, 4, 1.f);
    fill_normal<__nv_bfloat16><<<1024, 256, 0, st>>>((__nv_bfloat16*)vc, (size_t)cache * Hkv * d, 5, 1.f);
  } else {
    fill_normal<float><<<1024, 256, 0, st>>>((float*)q, (size_t)rows * Hq * d, 1, 1.f);
    fill_normal<float><<<1024, 256, 0, st>>>((float*)kn, (size_t)rows * Hkv * d, 2, 1.f);
    fill_normal<float><<<1024, 256, 0, st>>>((float*)vn, (size_t)rows * Hkv * d, 3, 1.f);
    fill_normal<float><<<1024, 256, 0, st>>>((float*)kc, (size_t)cache * Hkv * d, 4, 1.f);
    fill_normal<float><<<1024, 256, 0, st>>>((float*)vc, (size_t)cache * Hkv * d, 5, 1.f);
  }
  BENCH_CHECK(cudaGetLastError());

  ra.q_in = q; ra.k_in = kn; ra.q_out = q; ra.k_out = kn; ra.dtype = cfg->dt;
  ra.Hq = Hq; ra.Hkv = Hkv; ra.d = d; ra.base = 10000.0; ra.seqs = d_seqs; ra.batch = batch; ra.total_rows = rows;

  aa.q = q; aa.k_cache = kc; aa.v_cache = vc; aa.k_new = kn; aa.v_new = vn; aa.o = o;
  aa.in_dtype = cfg->dt; aa.out_dtype = cfg->dt; aa.Hq = Hq; aa.Hkv = Hkv; aa.d = d; aa.scale = 0.f;
  aa.seqs = d_seqs; aa.batch = batch; aa.tau = d_tau; aa.total_rows = rows; aa.total_cache = cache;
  aa.total_slots = slots; aa.max_cache = max_c; aa.max_new = max_n; aa.max_block = max_b; aa.dev_status = d_status;
  BENCH_SSV(ssv_verify_attn_workspace(&aa, &ws_attn));
  BENCH_CHECK(cudaMalloc(&ws_a, std::max<size_t>(ws_attn, 256)));
  BENCH_CHECK(cudaMemsetAsync(ws_a, 0, std::max<size_t>(ws_attn, 256), st));

  if (cfg->mode >= 0) {
    BENCH_CHECK(cudaMalloc(&logits, (size_t)slots * V * 4));
    fill_normal<float><<<2048, 256, 0, st>>>((float*)logits, (size_t)slots * V, 6, 1.4142135f);
    BENCH_CHECK(cudaMalloc((void**)&d_blocks, sizeof(int32_t) * batch));
    BENCH_CHECK(cudaMalloc((void**)&d_gam, sizeof(int32_t) * batch));
    BENCH_CHECK(cudaMalloc((void**)&d_soff, sizeof(int32_t) * batch));
    BENCH_CHECK(cudaMalloc((void**)&d_draft, sizeof(int32_t) * slots));
    BENCH_CHECK(cudaMalloc((void**)&d_nrow, sizeof(int32_t) * slots));
    BENCH_CHECK(cudaMalloc((void**)&d_nacc, sizeof(int32_t) * batch));
    BENCH_CHECK(cudaMalloc((void**)&d_nout, sizeof(int32_t) * batch));
    BENCH_CHECK(cudaMalloc((void**)&d_tok, sizeof(int32_t) * slots));
    BENCH_CHECK(cudaMalloc((void**)&d_ua, sizeof(float) * slots));
    BENCH_CHECK(cudaMalloc((void**)&d_us, sizeof(float) * batch));
    BENCH_CHECK(cudaMemcpyAsync(d_blocks, blocks.data(), sizeof(int32_t) * batch, cudaMemcpyHostToDevice, st));
    BENCH_CHECK(cudaMemcpyAsync(d_gam, gammas.data(), sizeof(int32_t) * batch, cudaMemcpyHostToDevice, st));
    BENCH_CHECK(cudaMemcpyAsync(d_soff, slot_off.data(), sizeof(int32_t) * batch, cudaMemcpyHostToDevice, st));
    {
      std::vector<int32_t> nrow(slots);
      for (int s = 0; s < slots; ++s) nrow[s] = s;
      BENCH_CHECK(cudaMemcpyAsync(d_nrow, nrow.data(), sizeof(int32_t) * slots, cudaMemcpyHostToDevice, st));
      BENCH_CHECK(cudaStreamSynchronize(st));
    }
    fill_tokens<<<64, 256, 0, st>>>(d_draft, slots, 7, V);
    fill_uniform<<<64, 256, 0, st>>>(d_ua, slots, 8);
    fill_uniform<<<64, 256, 0, st>>>(d_us, batch, 9);
    if (cfg->mode == SSV_ACCEPT_REJECT) {
      BENCH_CHECK(cudaMalloc(&dlogits, (size_t)slots * V * 4));
      fill_normal<float><<<2048, 256, 0, st>>>((float*)dlogits, (size_t)slots * V, 10, 1.4142135f);
    }
    if (cfg->mode == SSV_ACCEPT_GUMBEL) {
      BENCH_CHECK(cudaMalloc(&noise, (size_t)slots * V * 4));
      fill_gumbel<<<2048, 256, 0, st>>>((float*)noise, (size_t)slots * V, 11);
    }
    BENCH_CHECK(cudaGetLastError());
    ca.mode = (ssv_accept_mode)cfg->mode; ca.T = cfg->T; ca.V = V; ca.batch = batch; ca.total_slots = slots;
    ca.max_block = max_b; ca.logits_dtype = SSV_F32; ca.logits = logits; ca.draft_logits = dlogits;
    ca.draft_tokens = d_draft; ca.tau = d_tau; ca.block = d_blocks; ca.gamma = d_gam; ca.slot_off = d_soff;
    ca.noise = (const float*)noise; ca.n_noise_rows = slots; ca.noise_row = d_nrow; ca.u_accept = d_ua;
    ca.u_sample = d_us; ca.n_acc = d_nacc; ca.n_out = d_nout; ca.tokens = d_tok; ca.dev_status = d_status;
    BENCH_SSV(ssv_accept_workspace(&ca, &ws_acc));
    BENCH_CHECK(cudaMalloc(&ws_c, ws_acc));
    BENCH_CHECK(cudaMemsetAsync(ws_c, 0, ws_acc, st));
    for (int b = 0; b < batch; ++b) {
      const int need = std::min(gammas[b] + 1, blocks[b]);
      double rowsb = need;
      if (cfg->mode == SSV_ACCEPT_REJECT) rowsb += gammas[b];
      if (cfg->mode == SSV_ACCEPT_GUMBEL && cfg->T > 0.f) rowsb += need;
      acc_bytes += rowsb * V * 4.0;
    }
  }
  {  // commit: every sequence appends its N prompt rows and gamma / 2 accepted data rows
    std::vector<int32_t> nacc(batch), doff(batch), dcap(batch);
    int drows = 0;
    for (int b = 0; b < batch; ++b) {
      nacc[b] = gammas[b] / 2;
      dcap[b] = seqs[b].cache_len + seqs[b].new_len + seqs[b].block;
      doff[b] = drows;
      drows += dcap[b];
      commit_bytes += 2.0 * 2.0 * (seqs[b].new_len + nacc[b]) * Hkv * d * es;
    }
    BENCH_CHECK(cudaMalloc(&k_dst, (size_t)drows * Hkv * d * es));
    BENCH_CHECK(cudaMalloc(&v_dst, (size_t)drows * Hkv * d * es));
    BENCH_CHECK(cudaMalloc((void**)&d_cnacc, sizeof(int32_t) * batch));
    BENCH_CHECK(cudaMalloc((void**)&d_doff, sizeof(int32_t) * batch));
    BENCH_CHECK(cudaMalloc((void**)&d_dcap, sizeof(int32_t) * batch));
    BENCH_CHECK(cudaMalloc((void**)&d_newlen, sizeof(int32_t) * batch));
    BENCH_CHECK(cudaMemcpyAsync(d_cnacc, nacc.data(), sizeof(int32_t) * batch, cudaMemcpyHostToDevice, st));
    BENCH_CHECK(cudaMemcpyAsync(d_doff, doff.data(), sizeof(int32_t) * batch, cudaMemcpyHostToDevice, st));
    BENCH_CHECK(cudaMemcpyAsync(d_dcap, dcap.data(), sizeof(int32_t) * batch, cudaMemcpyHostToDevice, st));
    BENCH_CHECK(cudaStreamSynchronize(st));
    ma.k_new = kn; ma.v_new = vn; ma.k_dst = k_dst; ma.v_dst = v_dst; ma.dtype = cfg->dt; ma.Hkv = Hkv; ma.d = d;
    ma.seqs = d_seqs; ma.batch = batch; ma.tau = d_tau; ma.n_acc = d_cnacc; ma.dst_off = d_doff; ma.dst_cap = d_dcap;
    ma.new_len = d_newlen; ma.total_rows = rows; ma.total_slots = slots; ma.dst_rows = drows;
    ma.dev_status = d_status;
  }
  if (cfg->mode >= 0 && slots <= 2048) {  // fused LM head over the mask slots
    BENCH_CHECK(cudaMalloc(&lm_w, (size_t)V * hidden * 2));
    BENCH_CHECK(cudaMalloc(&lm_h, (size_t)slots * hidden * 2));
    fill_normal<__nv_bfloat16><<<2048, 256, 0, st>>>((__nv_bfloat16*)lm_w, (size_t)V * hidden, 12, 1.f);
    fill_normal<__nv_bfloat16><<<256, 256, 0, st>>>((__nv_bfloat16*)lm_h, (size_t)slots * hidden, 13,
                                                     1.f / sqrtf((float)hidden));
    BENCH_CHECK(cudaGetLastError());
    const bool gumbel = cfg->mode == SSV_ACCEPT_GUMBEL;
    la.mode = gumbel ? SSV_ACCEPT_GUMBEL : SSV_ACCEPT_ARGMAX; la.T = gumbel ? cfg->T : 0.f; la.V = V;
    la.hidden = hidden; la.batch = batch; la.total_slots = slots; la.hidden_states = lm_h; la.lm_head = lm_w;
    la.draft_tokens = d_draft; la.tau = d_tau; la.block = d_blocks; la.gamma = d_gam; la.slot_off = d_soff;
    la.noise = (const float*)noise; la.n_noise_rows = slots; la.noise_row = d_nrow; la.n_acc = d_nacc;
    la.n_out = d_nout; la.tokens = d_tok; la.dev_status = d_status;
    BENCH_SSV(ssv_lmhead_accept_workspace(&la, &ws_lm));
    BENCH_CHECK(cudaMalloc(&ws_l, std::max<size_t>(ws_lm, 256)));
    BENCH_CHECK(cudaMemsetAsync(ws_l, 0, std::max<size_t>(ws_lm, 256), st));
    double ver = 0;
    for (int b = 0; b < batch; ++b) ver += std::min(gammas[b] + 1, blocks[b]);
    lm_bytes = (double)V * hidden * 2 + (double)slots * hidden * 2 + ((gumbel && cfg->T > 0.f) ? ver * V * 4.0 : 0.0);
    lm_flops = 2.0 * ver * V * hidden;
  }
  BENCH_CHECK(cudaStreamSynchronize(st));

  for (int it = -3; it < iters; ++it) {
    float ms;
    BENCH_CHECK(cudaMemsetAsync(flush, it & 0xff, flush_bytes, st));
    BENCH_CHECK(cudaEventRecord(e0, st));
    BENCH_SSV(ssv_rope_copy(&ra, st));
    BENCH_CHECK(cudaEventRecord(e1, st));
    BENCH_CHECK(cudaEventSynchronize(e1));
    BENCH_CHECK(cudaEventElapsedTime(&ms, e0, e1));
    if (it >= 0) t_rope.push_back(ms);
    BENCH_CHECK(cudaMemsetAsync(flush, it & 0xff, flush_bytes, st));
    BENCH_CHECK(cudaEventRecord(e0, st));
    BENCH_SSV(ssv_verify_attn(&aa, ws_a, std::max<size_t>(ws_attn, 256), st));
    BENCH_CHECK(cudaEventRecord(e1, st));
    BENCH_CHECK(cudaEventSynchronize(e1));
    BENCH_CHECK(cudaEventElapsedTime(&ms, e0, e1));
    if (it >= 0) t_attn.push_back(ms);
    if (cfg->mode >= 0) {
      BENCH_CHECK(cudaMemsetAsync(flush, it & 0xff, flush_bytes, st));
      BENCH_CHECK(cudaEventRecord(e0, st));
      BENCH_SSV(ssv_accept(&ca, ws_c, ws_acc, st));
      BENCH_CHECK(cudaEventRecord(e1, st));
      BENCH_CHECK(cudaEventSynchronize(e1));
      BENCH_CHECK(cudaEventElapsedTime(&ms, e0, e1));
      if (it >= 0) t_acc.push_back(ms);
    }
    BENCH_CHECK(cudaMemsetAsync(flush, it & 0xff, flush_bytes, st));
    BENCH_CHECK(cudaEventRecord(e0, st));
    BENCH_SSV(ssv_commit(&ma, st));
    BENCH_CHECK(cudaEventRecord(e1, st));
    BENCH_CHECK(cudaEventSynchronize(e1));
    BENCH_CHECK(cudaEventElapsedTime(&ms, e0, e1));
    if (it >= 0) t_commit.push_back(ms);
    if (lm_w) {
      BENCH_CHECK(cudaMemsetAsync(flush, it & 0xff, flush_bytes, st));
      BENCH_CHECK(cudaEventRecord(e0, st));
      BENCH_SSV(ssv_lmhead_accept(&la, ws_l, std::max<size_t>(ws_lm, 256), st));
      BENCH_CHECK(cudaEventRecord(e1, st));
      BENCH_CHECK(cudaEventSynchronize(e1));
      BENCH_CHECK(cudaEventElapsedTime(&ms, e0, e1));
      if (it >= 0) t_lm.push_back(ms);
    }
  }
  BENCH_SSV(ssv_get_status(d_status, st));
  {
    const Timing tr = summarize(t_rope), ta = summarize(t_attn);
    Timing tc = {0, 0, 0}, tm = summarize(t_commit), tl = {0, 0, 0};
    if (!t_acc.empty()) tc = summarize(t_acc);
    if (!t_lm.empty()) tl = summarize(t_lm);
    const int n = snprintf(
        json_out, json_len,
        "{\"config\": \"%s\", \"iters\": %d, \"rope_us\": [%.3f, %.3f, %.3f], \"rope_bytes\": %.0f, "
        "\"attn_us\": [%.3f, %.3f, %.3f], \"attn_bytes\": %.0f, \"attn_flops\": %.0f, "
        "\"attn_gbs\": %.1f, \"attn_tflops\": %.2f, \"accept_us\": [%.3f, %.3f, %.3f], \"accept_bytes\": %.0f, "
        "\"accept_gbs\": %.1f, \"accept_seq_per_s\": %.1f, \"t_verify_us\": %.3f, "
        "\"commit_us\": [%.3f, %.3f, %.3f], \"commit_bytes\": %.0f, \"lmhead_hidden\": %d, "
        "\"lmhead_us\": [%.3f, %.3f, %.3f], \"lmhead_bytes\": %.0f, \"lmhead_flops\": %.0f}",
        cfg->name, iters, tr.med, tr.p10, tr.p90, rope_bytes, ta.med, ta.p10, ta.p90, attn_bytes, attn_flops,
        attn_bytes / (ta.med * 1e3), attn_flops / (ta.med * 1e6), tc.med, tc.p10, tc.p90, acc_bytes,
        tc.med > 0 ? acc_bytes / (tc.med * 1e3) : 0.0, tc.med > 0 ? batch / (tc.med * 1e-6) : 0.0,
        tr.med + ta.med + tc.med, tm.med, tm.p10, tm.p90, commit_bytes, hidden, tl.med, tl.p10, tl.p90, lm_bytes,
        lm_flops);
    if (n < 0 || (size_t)n >= json_len) rc = SSV_ERR_INVALID;
  }
done:
  cudaStreamSynchronize(st);
  void* bufs[] = {q, kn, vn, kc, vc, o, logits, dlogits, noise, flush, ws_a, ws_c, d_seqs, d_tau, d_blocks,
                  d_gam, d_soff, d_draft, d_nrow, d_nacc, d_nout, d_tok, d_status, d_ua, d_us, k_dst, v_dst,
                  lm_w, lm_h, ws_l, d_cnacc, d_doff, d_dcap, d_newlen};
  for (void* p : bufs)
    if (p) cudaFree(p);
  if (e0) cudaEventDestroy(e0);
  if (e1) cudaEventDestroy(e1);
  if (st) cudaStreamDestroy(st);
  return rc;
}

extern "C" ssv_status ssv_stream_read(const void* buf, size_t bytes, uint32_t* out, void* stream) {
  if (!buf || !out || ((uintptr_t)buf & 15u) || (bytes & 15u)) return SSV_ERR_INVALID;
  if (bytes == 0) return SSV_OK;
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0)
    return SSV_ERR_CUDA;
  const size_t n16 = bytes / 16;
  const size_t want = (n16 + 4095) / 4096;  // at least 64 KB per CTA
  const int grid = (int)std::min<size_t>((size_t)2 * sms, std::max<size_t>(want, 1));
  stream_read_kernel<<<grid, 512, 0, static_cast<cudaStream_t>(stream)>>>(static_cast<const uint4*>(buf), n16, out);
  return cudaGetLastError() == cudaSuccess ? SSV_OK : SSV_ERR_CUDA;
}
