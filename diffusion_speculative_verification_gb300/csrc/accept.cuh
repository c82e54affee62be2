// Shared pieces of the acceptance kernels (ssv_accept).
//
// SimSD summary, section 4 "Acceptance": standard rejection sampling in the
// temporal order the draft induces; the longest accepted prefix is kept.
// SPOT review, section "How it is used": state equality (exact at T = 0) and
// the coupled-noise match argmax(l/T + G[position]) (Proposition 2).
//
// Every verified row (a slot whose stage is <= min(gamma + 1, B)) is cut
// into vocabulary chunks of kAccChunk entries; a reduce kernel writes one
// AccPartial per (row, chunk).  Completion is two-level and lock-free (an
// arrival counter per row and per sequence, no spinning):
//   row merge  the CTA that lands the last chunk of a row merges its chunk
//              records with one warp (lanes over chunks): the decision token
//              (argmax of the score) or, for rejection sampling, the row
//              normalisers and the accept test u < p(d) / q(d);
//   seq walk   the CTA that merges the last row of a sequence walks the
//              stages in tau order with one warp and writes n_acc, n_out,
//              tokens and, for rejection sampling, which row the emitted
//              token is drawn from.
#pragma once

#include "ssv_internal.cuh"
#include "dfloat.cuh"
#include "noisegen.cuh"

#include <limits.h>
#include <math.h>

namespace ssv {

constexpr int kAccChunk = 8192;  // vocabulary entries per (row, chunk) record

struct AccPartial {
  float m_a, m_b;          // chunk max of the raw logits and of the draft logits  (reject)
  float sa_hi, sa_lo;      // compensated sum over the chunk of 2^((l - m_a) c2)   (reject)
  float sb_hi, sb_lo;      // same for the draft row                              (reject)
  float val;               // best decision score                                  (argmax / gumbel)
  int idx;                 // its first index
};

struct __align__(8) SlotNorm {  // row maxima of the logits and the draft logits (p_v = 2^((l_v - m_a) c2) / S_a, q likewise)
  float m_a, m_b;
};

struct __align__(8) RowResult {
  int ok;   // stage tested and accepted
  int dec;  // decision token of the row (argmax / gumbel)
};

struct AcceptParams {
  int mode;
  float T;
  float c2;                // log2(e) / T: rejection-sampling weights are 2^((l - max) * c2)
  int V;
  int vec;                 // rows allow 4-element vector accesses
  int batch;
  int total_slots;
  int nchunks;
  const void* logits;
  const void* draft_logits;
  const int32_t* draft_tokens;
  const int32_t* tau;
  const int32_t* block;
  const int32_t* gamma;
  const int32_t* slot_off;
  const float* noise;
  int n_noise_rows;
  const int32_t* noise_row;
  const float* u_accept;
  const float* u_sample;
  int32_t* n_acc;
  int32_t* n_out;
  int32_t* tokens;
  int32_t* dev_status;
  // 1: the kernel before this one on the stream is the step's attention
  // kernel, whose outputs overlap none of the batch metadata; the metadata
  // may then be read before it completes (programmatic dependent launch).
  int early;
  // workspace carve-up (the counters come first and are contiguous)
  int32_t* unit_ctr;    // [2]            streaming pass: next unit, producers done
  int32_t* cnt_seq;     // [batch]        merged rows of the sequence
  int32_t* cnt_row;     // [total_slots]  chunks of the row done
  int32_t* emit;        // [batch][2] : emission slot (or -1), 1 = residual / 0 = p
  AccPartial* part;     // [total_slots][nchunks]
  SlotNorm* norm;       // [total_slots]
  RowResult* rowres;    // [total_slots]
  // rejection-sampling emission (double-float), per sequence over nsub
  // sub-chunks of kEmitSub vocabulary entries:
  int nsub;
  float4* enorm;        // [batch][nsub]     sums of e_a = 2^((l - m_a) c2) and e_b = 2^((ql - m_b) c2)
  float4* smass;        // [batch][nsub]     residual mass, p mass (each hi, lo)
  float4* wmass;        // [batch][nsub][8]  the same per warp of the sub-chunk's CTA
  // [batch][nsub][8][256]: e_a and e_b (each hi, lo) of every entry
  // of the emitted row, written by the normaliser pass for a residual sample
  // and read back by the sampling pass ([j][t] holds the sub-chunk's entry
  // 8 t + j); null: the sampling pass forms them again from the logits
  float4* eexp;
  // c2 = log2(e) / T split into an fp32 head and tail; 2^(2^i / 256),
  // i = 0..7, likewise (host-computed)
  float c2_hi, c2_lo;
  float2 e2pow[8];
  // bounded waits of the streaming reduce give up after wait_budget SM
  // cycles; fault_skip >= 0 makes its CTA 0 leave out that chunk's copy
  // (test support, ssv_set_fault_injection)
  long long wait_budget;
  int fault_skip;
  uint64_t noise_seed;  // SSV_ACCEPT_GUMBEL_GEN: key of the noise generator
};

constexpr int kEmitSub = 2048;  // vocabulary entries per emission CTA (256 threads x 8)

struct AccWorkspaceLayout {
  size_t unit_ctr, cnt_seq, cnt_row, emit, part, norm, rowres, enorm, smass, wmass, eexp, total;
};

// eexp: room for the emitted rows' stored exponentials (rejection sampling);
// without it L.eexp == L.total and the sampling pass recomputes them.
inline AccWorkspaceLayout accept_layout(int batch, int total_slots, int nchunks, bool eexp) {
  const size_t nsub = (size_t)nchunks * (kAccChunk / kEmitSub);
  AccWorkspaceLayout L;
  size_t o = 0;
  L.unit_ctr = o;   o += sizeof(int32_t) * 2;
  L.cnt_seq = o;    o += sizeof(int32_t) * (size_t)batch;
  L.cnt_row = o;    o = align_up(o + sizeof(int32_t) * (size_t)total_slots, 256);
  L.emit = o;       o = align_up(o + sizeof(int32_t) * 2 * (size_t)batch, 256);
  L.part = o;       o = align_up(o + sizeof(AccPartial) * (size_t)total_slots * nchunks, 256);
  L.norm = o;       o = align_up(o + sizeof(SlotNorm) * (size_t)total_slots, 256);
  L.rowres = o;     o = align_up(o + sizeof(RowResult) * (size_t)total_slots, 256);
  L.enorm = o;      o = align_up(o + sizeof(float) * 4 * (size_t)batch * nsub, 256);
  L.smass = o;      o = align_up(o + sizeof(float) * 4 * (size_t)batch * nsub, 256);
  L.wmass = o;      o = align_up(o + sizeof(float) * 4 * 8 * (size_t)batch * nsub, 256);
  L.eexp = o;       if (eexp) o = align_up(o + sizeof(float) * 4 * (size_t)kEmitSub * batch * nsub, 256);
  L.total = o;
  return L;
}

// ---- arithmetic -------------------------------------------------------------
__device__ __forceinline__ float ex2f(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

template <typename T>
__device__ __forceinline__ float ld_logit(const void* base, size_t i) {
  return Elem<T>::to_f32(static_cast<const T*>(base)[i]);
}

__device__ __forceinline__ void kahan_add(float& s, float& c, float x) {
  const float y = x - c;
  const float t = s + y;
  c = (t - s) - y;
  s = t;
}

// (h1, l1) += (h2, l2) with an error-free transformation of the leading terms
__device__ __forceinline__ void two_sum_acc(float& h1, float& l1, float h2, float l2) {
  const float s = h1 + h2;
  const float bb = s - h1;
  const float err = (h1 - (s - bb)) + (h2 - bb);
  h1 = s;
  l1 = l1 + l2 + err;
}

// larger score wins; equal scores go to the smaller vocabulary index
__device__ __forceinline__ void argmax_combine(float& v, int& i, float ov, int oi) {
  if (ov > v || (ov == v && oi < i)) { v = ov; i = oi; }
}

__device__ __forceinline__ void warp_argmax(float& v, int& i) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1)
    argmax_combine(v, i, __shfl_xor_sync(0xffffffffu, v, o), __shfl_xor_sync(0xffffffffu, i, o));
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

__device__ __forceinline__ void warp_sum2(float& h, float& l) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float a = __shfl_xor_sync(0xffffffffu, h, o), b = __shfl_xor_sync(0xffffffffu, l, o);
    two_sum_acc(h, l, a, b);
  }
}

// ---- per-sequence validity, checked by one warp (all 32 lanes) --------------
__device__ __forceinline__ bool warp_seq_valid(const AcceptParams& p, int b) {
  const int B = p.block[b], g = p.gamma[b];
  bool ok = B >= 1 && B <= 64 && g >= 0 && g <= B && p.slot_off[b] + B <= p.total_slots;
  if (ok) ok = warp_tau_is_permutation(p.tau + p.slot_off[b], B);
  return ok;
}

// Coupled-noise score fl32(fl32(l / T) + G) with G generated from the word x
// (T == 1: l / 1 is exact and skipped).
__device__ __forceinline__ float gen_score(float l, uint32_t x, float T, bool unit_t) {
  return __fadd_rn(unit_t ? l : __fdiv_rn(l, T), noise::gumbel_from_bits(x));
}

// ---- completion steps (one warp, all 32 lanes) ------------------------------

// Lane 0 publishes `add` arrivals on a counter, releasing its own earlier
// writes; returns on every lane whether this call completed the count (then
// every lane has acquire ordering for the other contributors' writes).  A
// caller that brings the whole count at once needs no counter at all.
__device__ __forceinline__ bool warp_arrive(int32_t* counter, int add, int target) {
  if (add == target) {  // every record is this warp's own (lane 0 wrote them)
    __syncwarp();
    asm volatile("fence.acq_rel.gpu;" ::: "memory");
    return true;
  }
  int last = 0;
  if ((threadIdx.x & 31) == 0) {
    int prev;
    asm volatile("atom.acq_rel.gpu.global.add.s32 %0, [%1], %2;" : "=r"(prev) : "l"(counter), "r"(add) : "memory");
    last = (prev + add) == target;
  }
  last = __shfl_sync(0xffffffffu, last, 0);
  if (last) asm volatile("fence.acq_rel.gpu;" ::: "memory");
  return last != 0;
}

// Inputs of a rejection test that come with the call (lane 0 holds them):
// the draft token d, its logit under the target and the draft, u_accept.
struct RowInputs {
  int d;
  float ld, qd, ua;
};

template <typename T>
__device__ __forceinline__ RowInputs row_inputs(const AcceptParams& p, int slot, bool tested) {
  RowInputs in{-1, 0.f, 0.f, 0.f};
  if (tested && (threadIdx.x & 31) == 0) {
    in.d = p.draft_tokens[slot];
    in.ua = p.u_accept[slot];
    if (in.d >= 0 && in.d < p.V) {
      in.ld = ld_logit<T>(p.logits, (size_t)slot * p.V + in.d);
      in.qd = ld_logit<T>(p.draft_logits, (size_t)slot * p.V + in.d);
    }
  }
  return in;
}

// Merge of verified row `slot` (1-based stage st, draft length g): lanes
// over chunks.  Writes rowres[slot] and, for rejection sampling, norm[slot].
// pre: the row's RowInputs when the caller loaded them already, else null.
template <int MODE, typename T>
__device__ void warp_row_merge(const AcceptParams& p, int slot, int st, int g, const RowInputs* pre = nullptr) {
  const int lane = threadIdx.x & 31;
  const AccPartial* pp = p.part + (size_t)slot * p.nchunks;
  const bool tested = st <= g;  // stages past gamma carry no draft token
  RowResult rr;
  rr.ok = 0;
  rr.dec = -1;
  if (MODE != SSV_ACCEPT_REJECT) {
    float v = -INFINITY;
    int i = INT_MAX;
    for (int c = lane; c < p.nchunks; c += 32) argmax_combine(v, i, __ldcg(&pp[c].val), __ldcg(&pp[c].idx));
    warp_argmax(v, i);
    rr.dec = i;
    rr.ok = tested && p.draft_tokens[slot] == i;
    if (lane == 0) p.rowres[slot] = rr;
    return;
  }
  // Rejection sampling: the row maxima (warp max of the chunk maxima), then
  // S = sum over chunks of s_c 2^((m_c - M) c2) in double-float arithmetic
  // (fp32 pairs: fp64 is a narrow pipe on this part, tens of cycles per
  // dependent operation), each scale factor an fp32 exp2 of an argument
  // formed from the exact difference m_c - M (about 5e-7 relative, the order
  // of the chunk sums' own exp2 rounding).  The ratio p(d)/q(d) is then
  // 2^(((l_d - M_a) - (q_d - M_b)) c2) S_b / S_a in fp32.
  RowInputs in = pre ? *pre : row_inputs<T>(p, slot, tested);
  const float c2 = p.c2;
  constexpr int kHeld = 2;  // chunk records held per lane (up to 64 chunks; beyond that, loaded twice)
  float cma[kHeld], cmb[kHeld];
  dfx csa[kHeld], csb[kHeld];
  float ma = -INFINITY, mb = -INFINITY;
#pragma unroll
  for (int h = 0; h < kHeld; ++h) {
    const int c = lane + 32 * h;
    cma[h] = cmb[h] = -INFINITY;
    csa[h] = csb[h] = dfx{0.f, 0.f};
    if (c < p.nchunks) {
      cma[h] = __ldcg(&pp[c].m_a);
      csa[h] = dfx{__ldcg(&pp[c].sa_hi), __ldcg(&pp[c].sa_lo)};
      if (tested) {
        cmb[h] = __ldcg(&pp[c].m_b);
        csb[h] = dfx{__ldcg(&pp[c].sb_hi), __ldcg(&pp[c].sb_lo)};
      }
    }
    ma = fmaxf(ma, cma[h]);
    mb = fmaxf(mb, cmb[h]);
  }
  for (int c = lane + 32 * kHeld; c < p.nchunks; c += 32) {
    ma = fmaxf(ma, __ldcg(&pp[c].m_a));
    if (tested) mb = fmaxf(mb, __ldcg(&pp[c].m_b));
  }
  const float Ma = warp_max(ma), Mb = warp_max(mb);
  // s_c 2^((m_c - M) c2), added into acc
  auto add_scaled = [&](dfx& acc, float m, dfx sc, float M) {
    if (m == -INFINITY) return;
    const dfx dm = dfx_two_sum(m, -M);  // exact m - M <= 0
    const float f = (m == M) ? 1.f : exp2f(__fmaf_rn(dm.hi, c2, __fmul_rn(dm.lo, c2)));
    acc = dfx_add(acc, f == 1.f ? sc : dfx_mul(sc, dfx{f, 0.f}));
  };
  dfx sa{0.f, 0.f}, sb{0.f, 0.f};
#pragma unroll
  for (int h = 0; h < kHeld; ++h) {
    add_scaled(sa, cma[h], csa[h], Ma);
    if (tested) add_scaled(sb, cmb[h], csb[h], Mb);
  }
  for (int c = lane + 32 * kHeld; c < p.nchunks; c += 32) {
    add_scaled(sa, __ldcg(&pp[c].m_a), dfx{__ldcg(&pp[c].sa_hi), __ldcg(&pp[c].sa_lo)}, Ma);
    if (tested) add_scaled(sb, __ldcg(&pp[c].m_b), dfx{__ldcg(&pp[c].sb_hi), __ldcg(&pp[c].sb_lo)}, Mb);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    sa = dfx_add(sa, dfx{__shfl_xor_sync(0xffffffffu, sa.hi, o), __shfl_xor_sync(0xffffffffu, sa.lo, o)});
    sb = dfx_add(sb, dfx{__shfl_xor_sync(0xffffffffu, sb.hi, o), __shfl_xor_sync(0xffffffffu, sb.lo, o)});
  }
  if (lane == 0) {
    SlotNorm nm;
    nm.m_a = Ma;
    nm.m_b = Mb;
    p.norm[slot] = nm;
    if (tested) {
      if (in.d >= 0 && in.d < p.V) {
        // exponent ((l_d - M_a) - (q_d - M_b)) c2 from exact differences
        const dfx ea = dfx_two_sum(in.ld, -Ma), eb = dfx_two_sum(in.qd, -Mb);
        const dfx e = dfx_add(ea, dfx{-eb.hi, -eb.lo});
        const float r = exp2f(__fmaf_rn(e.hi, c2, __fmul_rn(e.lo, c2)));
        // S_b / S_a: a quotient of the high parts plus one correction step
        const float q0 = __fdiv_rn(sb.hi, sa.hi);
        const float q1 = __fdiv_rn(__fadd_rn(__fmaf_rn(-q0, sa.hi, sb.hi), __fmaf_rn(-q0, sa.lo, sb.lo)), sa.hi);
        rr.ok = in.ua < __fmul_rn(r, __fadd_rn(q0, q1));
      } else {
        report(p.dev_status, SSV_ERR_INVALID);
      }
    }
    p.rowres[slot] = rr;
  }
}

// Shared-memory scratch of the warp that walks a sequence.
struct WalkSmem {
  int slot[64];  // slot (offset in the sequence) of each stage
  int ok[64];    // per stage: tested and accepted
  int dec[64];   // per stage: decision token (argmax / gumbel)
  int tok[64];   // per stage: draft token
};

// Walk of sequence b (slots off .. off + B - 1, draft length g) once every
// verified row is merged: one round of loads (row results, draft tokens, and
// the stage map unless the caller holds it in shared memory as stage_s, one
// byte per slot), rearranged into stage order.
template <int MODE>
__device__ void warp_seq_walk(const AcceptParams& p, int b, int off, int B, int g, WalkSmem& w,
                              const unsigned char* stage_s) {
  const int lane = threadIdx.x & 31;
  const int need = min(g + 1, B);
  int st[2], rok[2], rdec[2], dtok[2];
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const int j = lane + 32 * h;
    st[h] = (j < B) ? (stage_s ? (int)stage_s[off + j] : __ldcg(&p.tau[off + j])) : 0;
    dtok[h] = (j < B) ? p.draft_tokens[off + j] : -1;
    const int2 r = (j < B) ? __ldcg(reinterpret_cast<const int2*>(p.rowres + off + j)) : make_int2(0, -1);
    rok[h] = r.x;
    rdec[h] = r.y;
  }
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const int j = lane + 32 * h;
    if (j < B) {
      const int s0 = st[h] - 1;  // a valid sequence's map is a permutation of 1..B
      const bool merged = s0 < need;  // only verified rows hold row results
      w.slot[s0] = j;
      w.ok[s0] = merged ? rok[h] : 0;
      w.dec[s0] = merged ? rdec[h] : -1;
      w.tok[s0] = dtok[h];
    }
  }
  __syncwarp();
  unsigned long long okmask = 0ull;
  for (int base = 0; base < g; base += 32) {
    const int s0 = base + lane;  // 0-based stage
    okmask |= (unsigned long long)__ballot_sync(0xffffffffu, s0 < g && w.ok[s0]) << base;
  }
  const unsigned long long rej = ~okmask;
  int n = rej ? __ffsll((long long)rej) - 1 : 64;
  n = min(n, g);  // longest accepted prefix in stage order
  for (int i = lane; i < B; i += 32) {
    int tok = -1;
    if (i < n) tok = w.tok[i];
    else if (i == n && MODE != SSV_ACCEPT_REJECT) tok = w.dec[n];
    p.tokens[off + i] = tok;
  }
  if (lane == 0) {
    p.n_acc[b] = n;
    p.n_out[b] = (n + 1 <= B) ? n + 1 : n;
    if (MODE == SSV_ACCEPT_REJECT) {
      p.emit[2 * b] = (n < B) ? off + w.slot[n] : -1;
      p.emit[2 * b + 1] = (n + 1 <= g) ? 1 : 0;  // a rejected draft: residual (p - q)_+
    }
  }
  __syncwarp();
}

// `add` more chunk records of row `slot` (stage st of sequence b, whose slots
// start at off; block B, draft length g) are written by lane 0: run the row
// merge and the sequence walk when they complete the counts.  stage_s: the
// stage map in shared memory (one byte per slot), or null.
template <int MODE, typename T>
__device__ void warp_rows_done(const AcceptParams& p, int b, int slot, int add, int st, int off, int B, int g,
                               WalkSmem& w, const unsigned char* stage_s) {
  if (!warp_arrive(&p.cnt_row[slot], add, p.nchunks)) return;
  warp_row_merge<MODE, T>(p, slot, st, g);
  if ((threadIdx.x & 31) == 0 && add != p.nchunks) p.cnt_row[slot] = 0;
  if (!warp_arrive(&p.cnt_seq[b], 1, min(g + 1, B))) return;
  warp_seq_walk<MODE>(p, b, off, B, g, w, stage_s);
  if ((threadIdx.x & 31) == 0 && min(g + 1, B) != 1) p.cnt_seq[b] = 0;
}

// ---- launchers ----------------------------------------------------------------
// Streaming reduce (accept_stream.cu): one CTA per SM, bulk-copy ring.
bool accept_stream_supported(const AcceptParams& p, int mode, bool bf16);
cudaError_t launch_accept_stream(const AcceptParams& p, int mode, bool bf16, cudaStream_t st);

}  // namespace ssv
