/*
 * ssv.h -- C ABI of libssv: the target-model verification pass of
 * speculative decoding for block-diffusion language models, on one GB300
 * (sm_103a).
 *
 * The pass (SimSD, "Simple Speculative Decoding in Diffusion Language
 * Models", summary sections 1-4): after the prompt the target sees a data
 * section D (B reference tokens) and a mask section D~ (B [MASK] slots);
 * the pair (D_k, D~_k) occupies one response position.  A stage map tau,
 * a permutation of 1..B, orders the positions in time and gates attention.
 * One forward pass under that mask yields logits for every drafted
 * position; acceptance then keeps the longest accepted prefix in stage
 * order (SimSD section 4; state equality and the coupled Gumbel-noise match
 * of the SPOT review, section "How it is used").
 *
 * Conventions for every entry point
 *  - All pointers named "device" are CUDA device (or managed) addresses on
 *    the current device; "host" pointers are ordinary CPU memory.  The
 *    caller owns every buffer; the library allocates nothing on these
 *    paths.  Scratch space is caller-provided ("workspace"), sized by the
 *    matching *_workspace query, 256-byte aligned, and must be all-zero
 *    when first used: each call leaves the zero-initialised counter area
 *    zero again on exit.
 *  - `stream` is a cudaStream_t (NULL = legacy default stream).  Calls are
 *    asynchronous on it.  Host-side validation errors return synchronously
 *    and launch nothing.
 *  - Errors found on the device (a stage map that is not a permutation, a
 *    bounded wait that ran out, a non-finite temperature) are written to
 *    `dev_status` (device int32, may be NULL; first error wins) and read
 *    back with ssv_get_status().  Affected outputs are then unspecified,
 *    and after SSV_ERR_TIMEOUT the workspace's counter area may be left
 *    non-zero: clear the workspace before its next use.
 *  - Nothing is thread-local; calls from several host threads on different
 *    streams are safe.  Two calls whose workspaces overlap must not run
 *    concurrently.
 */
#ifndef SSV_H_
#define SSV_H_

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define SSV_API __attribute__((visibility("default")))
#else
#define SSV_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  SSV_OK = 0,
  SSV_ERR_INVALID = 1,      /* bad argument (null pointer, shape, alignment) */
  SSV_ERR_UNSUPPORTED = 2,  /* valid but not implemented (e.g. head_dim 96) */
  SSV_ERR_CUDA = 3,         /* a CUDA runtime call failed */
  SSV_ERR_TIMEOUT = 4,      /* a bounded on-device wait ran out */
  SSV_ERR_BAD_TAU = 5,      /* stage map of some sequence is not a permutation of 1..B */
  SSV_ERR_WORKSPACE = 6,    /* workspace null, misaligned or smaller than the query */
  SSV_ERR_NOT_FINITE = 7    /* temperature not finite / negative */
} ssv_status;

typedef enum { SSV_F32 = 0, SSV_BF16 = 1 } ssv_dtype;

typedef enum {
  SSV_ACCEPT_ARGMAX = 0,    /* T = 0 state equality: accept iff draft == argmax(l) */
  SSV_ACCEPT_GUMBEL = 1,    /* coupled noise: accept iff draft == argmax(fl(l/T) + G[row]) */
  SSV_ACCEPT_REJECT = 2,    /* standard rejection sampling, accept iff u < p(d)/q(d) */
  SSV_ACCEPT_GUMBEL_GEN = 3 /* coupled noise generated on the device: accept iff
                               draft == argmax(fl(l/T) + G(noise_seed, noise_row[k], v)) */
} ssv_accept_mode;

/*
 * One sequence of a packed batch.  Query rows of a sequence are its N fresh
 * prompt rows followed by 2B tail rows (D_1..D_B, then D~_1..D~_B); they sit
 * at rows [q_off, q_off + N + 2B) of Q, K_new, V_new and O.  Its C cached
 * prompt keys sit at rows [kv_off, kv_off + C) of K_cache / V_cache.  Its
 * stage map occupies tau[tau_off .. tau_off + B).  Sequences are packed in
 * increasing q_off order without overlap (q_off[b] + N_b + 2B_b <=
 * q_off[b+1]): kernels find a row's sequence by binary search on q_off.
 * Every kernel checks each sequence's extents on the device before it
 * touches the sequence's rows (q_off + N + 2B <= total_rows, kv_off + C <=
 * the cache rows, tau_off + B <= total_slots, all offsets >= 0, 1 <= B <=
 * 64, and for the attention C, N, B within max_cache, max_new, max_block):
 * a sequence that fails is skipped -- nothing of it is read or written --
 * and SSV_ERR_INVALID is reported through dev_status.  Overlapping or
 * unsorted sequences are not detected (their rows may be processed twice or
 * under the wrong sequence, still inside the buffers).
 */
typedef struct {
  int32_t cache_len;  /* C >= 0 */
  int32_t new_len;    /* N >= 0 */
  int32_t block;      /* B, 1 <= B <= 64 */
  int32_t q_off;
  int32_t kv_off;
  int32_t tau_off;
} ssv_seq;

/* ------------------------------------------------------------------------
 * ssv_rope_copy -- rotary embedding with the RoPE-copy index.
 * SimSD summary, section 3 "Position Encoding Alignment": each mask slot
 * D~_k reuses the RoPE index of its data token D_k.
 *
 * Positions, without a position table (positions == NULL): fresh prompt row
 * i is at C + i; tail row r (0 <= r < 2B) at P + (r mod B), P = C + N.
 * With a table (device int32 [total_rows], entries >= 0): fresh prompt row
 * i of a sequence is at positions[q_off + i], data row D_k at
 * positions[q_off + N + k - 1], and mask row D~_k at D_k's entry (entries
 * at mask rows are not read).  The table serves passes whose positions are
 * not contiguous: after a commit (ssv_commit) the accepted data rows keep
 * the positions of their slots, so the next pass over the same block gives
 * its remaining slots, and the emitted token entering as a fresh prompt
 * row, the positions of their own slots (a reading: the pages do not
 * describe the loop).  Rotate-half pairing (x_i, x_{i+d/2}) with
 * theta_i = base^(-2i/d); angles are formed and reduced in fp64, the
 * rotation is done in fp32 and stored in `dtype`.
 *
 * q_in  [total_rows, Hq, d]  device, dtype     q_out same shape (may equal q_in)
 * k_in  [total_rows, Hkv, d] device, dtype     k_out same shape (may equal k_in)
 * seqs  [batch] device ssv_seq.  Every row of [0, total_rows) must belong to
 *       exactly one sequence (rows outside all sequences are left untouched).
 * d in {64, 128}; pointers 16-byte aligned.
 * Errors: SSV_ERR_INVALID (null, non-positive sizes, misalignment),
 *         SSV_ERR_UNSUPPORTED (d), SSV_ERR_CUDA (launch); on device
 *         SSV_ERR_INVALID for a sequence whose rows leave [0, total_rows)
 *         (or B outside 1..64, or C + N + B beyond int range; its rows are
 *         left untouched) and for a negative table entry (that row is left
 *         untouched).
 * ---------------------------------------------------------------------- */
typedef struct {
  const void* q_in;
  const void* k_in;
  void* q_out;
  void* k_out;
  ssv_dtype dtype;
  int32_t Hq, Hkv, d;
  double base;                 /* RoPE base, e.g. 10000 */
  const ssv_seq* seqs;         /* device */
  int32_t batch;
  int32_t total_rows;
  const int32_t* positions;    /* device [total_rows] or NULL (see above) */
  int32_t* dev_status;         /* device, may be NULL */
} ssv_rope_args;

SSV_API ssv_status ssv_rope_copy(const ssv_rope_args* a, void* stream);

/* ------------------------------------------------------------------------
 * ssv_verify_attn -- attention of the verification pass.
 * SimSD summary, section 2 "Temporal Attention Mask" and section 4
 * "Verification".  For every query row and query head h (kv head h / G,
 * G = Hq / Hkv):  O = softmax(scale * q K^T restricted to allowed keys) V.
 * Keys of a sequence, in order: cache (C), fresh prompt (N), D_1..D_B,
 * D~_1..D~_B.  Allowed keys:
 *   fresh prompt row i : cache and fresh prompt keys 0 .. C+i (causal)
 *   data row D_j       : whole prompt, D_k with tau(k) <= tau(j)  (reading;
 *                        the pages fix only the mask-slot rule)
 *   mask row D~_i      : whole prompt, D_j with tau(j) < tau(i),
 *                        D~_j with tau(j) >= tau(i)
 * The mask is derived on the device from tau; it is never stored.
 *
 * q       [total_rows, Hq, d]   device, in_dtype, post-RoPE
 * k_cache [total_cache, Hkv, d] device, in_dtype, already rotated
 * v_cache [total_cache, Hkv, d] device
 * k_new   [total_rows, Hkv, d]  device, post-RoPE
 * v_new   [total_rows, Hkv, d]  device
 * o       [total_rows, Hq, d]   device, out_dtype (written for every row of
 *                               every sequence)
 * tau     [sum B] int32 device
 * in_dtype: SSV_F32 (exact fp32 SIMT path) or SSV_BF16 (tensor-core path,
 * fp32 accumulation).  out_dtype: SSV_F32 or SSV_BF16 (bf16 input only).
 * d in {64, 128}; Hq % Hkv == 0; 1 <= B <= 64; pointers 16-byte aligned.
 * max_cache / max_new / max_block bound every sequence's C / N / B (used to
 * size grids and workspace).  scale 0 means 1/sqrt(d).
 * Errors: SSV_ERR_INVALID, SSV_ERR_UNSUPPORTED, SSV_ERR_WORKSPACE,
 *         SSV_ERR_CUDA; on device SSV_ERR_BAD_TAU, SSV_ERR_TIMEOUT, and
 *         SSV_ERR_INVALID for a sequence outside the buffers (skipped: its
 *         rows of o are not written).
 * Scheduling: the bf16 path launches one CTA per SM; where a unit of work is
 * split across CTAs, the CTA holding its first key block waits (bounded, about
 * one second of SM clock) for the others' partial results.  Before launching,
 * the host checks that the kernel's resources let one CTA reside on every SM
 * at once (else SSV_ERR_CUDA, nothing launched).  Work on other streams that
 * keeps SMs busy for longer than that second while this kernel runs can
 * still end the call with SSV_ERR_TIMEOUT (never a hang).
 * ---------------------------------------------------------------------- */
typedef struct {
  const void* q;
  const void* k_cache;
  const void* v_cache;
  const void* k_new;
  const void* v_new;
  void* o;
  ssv_dtype in_dtype;
  ssv_dtype out_dtype;
  int32_t Hq, Hkv, d;
  float scale;
  const ssv_seq* seqs;         /* device [batch] */
  int32_t batch;
  const int32_t* tau;          /* device [total_slots] */
  int32_t total_rows;          /* sum of N + 2B */
  int32_t total_cache;         /* sum of C */
  int32_t total_slots;         /* sum of B */
  int32_t max_cache, max_new, max_block;
  int32_t* dev_status;         /* device, may be NULL */
} ssv_attn_args;

SSV_API ssv_status ssv_verify_attn_workspace(const ssv_attn_args* a, size_t* bytes);
SSV_API ssv_status ssv_verify_attn(const ssv_attn_args* a, void* workspace, size_t workspace_bytes, void* stream);

/* ------------------------------------------------------------------------
 * ssv_accept -- acceptance in temporal order, longest accepted prefix.
 * SimSD summary section 4 "Acceptance" (rejection sampling in the draft's
 * temporal order); SPOT review "How it is used" (state equality, exact at
 * T = 0; coupled-noise match with one Gumbel table per absolute output
 * position, which recovers the target distribution, Proposition 2).
 *
 * Per sequence b with block B, verified stages 1..gamma (0 <= gamma <= B):
 * stage s is slot k = tau^{-1}(s).  Walk s = 1..gamma and accept while
 *   ARGMAX : draft_tokens[k] == argmax_v l_k[v]            (ties: lowest v)
 *   GUMBEL : draft_tokens[k] == argmax_v fl32(fl32(l_k[v]/T) + noise[noise_row[k]][v])
 *            (IEEE fp32, no contraction; T = 0 means ARGMAX)
 *   REJECT : u_accept[k] < p(d)/q(d), p = softmax(l_k/T), q = softmax(draft_logits_k/T)
 *   GUMBEL_GEN : as GUMBEL with the table value replaced by one generated on
 *            the device, G(seed, pos, v) = -L(-L(U)), U = (floor(x / 2^9) + 1/2)
 *            2^-23, x = word (v mod 4) of Philox4x32-10 at counter
 *            (floor(v / 4), pos, 0, 0) under key (low, high word of noise_seed),
 *            pos = noise_row[k] (any 32-bit value the caller assigns to the
 *            slot's absolute output position; drafter and target use the same),
 *            L the natural logarithm by one fixed sequence of fp32 operations:
 *            reduction to m in [sqrt(1/2), sqrt 2], s = (m - 1) / (m + 1),
 *            ln m = 2 s + s z (2/3 + z (2/5 + z (2/7 + z 2/9))), z = s^2
 *            (Horner from the inside, every operation rounded to nearest), plus
 *            e ln 2.  Nothing but the logits is read; T = 0 means ARGMAX.
 * n_acc = leading accepted stages.  If c = n_acc + 1 <= B one target token
 * is emitted at stage c: the ARGMAX/GUMBEL decision; for REJECT a sample of
 * (p - q)_+ if c <= gamma, else of p, by inverse CDF with u_sample[b]
 * (smallest v whose cumulative mass exceeds u_sample * total).
 *
 * logits       [total_slots, V] device, logits_dtype, row = slot (slot order);
 *              only rows of stages <= min(gamma + 1, B) are read.
 * draft_logits [total_slots, V] device, logits_dtype (REJECT only, else NULL)
 * draft_tokens, tau, noise_row, u_accept: [total_slots] device
 * block, gamma, slot_off, u_sample: [batch] device; slot_off[b] = first slot;
 *              sequences in increasing slot order without overlap
 *              (slot_off[b] + block[b] <= slot_off[b+1])
 * noise [n_noise_rows, V] fp32 device (GUMBEL with T > 0 only)
 * noise_seed: GUMBEL_GEN only (noise_row then holds positions, not rows)
 * Outputs: n_acc[batch], n_out[batch] (= n_acc + 1 if a token is emitted),
 *          tokens[total_slots]: per sequence, the accepted drafts in stage
 *          order then the emitted token, rest -1.
 * V >= 1; T >= 0 (REJECT needs T > 0); 1 <= block <= 64.
 * Workspace: ssv_accept_workspace bytes.  Under REJECT it includes
 *   16 * batch * 8192 * ceil(V / 8192) bytes in which the first emission
 *   pass keeps the double-float exponentials of each sequence's emitted row
 *   for the second (about 2.4 MB per sequence at V = 151936).
 * Errors: SSV_ERR_INVALID, SSV_ERR_WORKSPACE, SSV_ERR_NOT_FINITE,
 *         SSV_ERR_CUDA; on device SSV_ERR_BAD_TAU.
 * ---------------------------------------------------------------------- */
typedef struct {
  ssv_accept_mode mode;
  float T;
  int32_t V;
  int32_t batch;
  int32_t total_slots;
  int32_t max_block;
  ssv_dtype logits_dtype;
  const void* logits;
  const void* draft_logits;
  const int32_t* draft_tokens;
  const int32_t* tau;
  const int32_t* block;
  const int32_t* gamma;
  const int32_t* slot_off;
  const float* noise;
  int32_t n_noise_rows;
  const int32_t* noise_row;
  const float* u_accept;
  const float* u_sample;
  int32_t* n_acc;
  int32_t* n_out;
  int32_t* tokens;
  int32_t* dev_status;         /* device, may be NULL */
  uint64_t noise_seed;         /* GUMBEL_GEN: key of the noise generator */
} ssv_accept_args;

SSV_API ssv_status ssv_accept_workspace(const ssv_accept_args* a, size_t* bytes);
SSV_API ssv_status ssv_accept(const ssv_accept_args* a, void* workspace, size_t workspace_bytes, void* stream);

/* ------------------------------------------------------------------------
 * ssv_verify_step -- the whole verification step in one call: ssv_rope_copy
 * (rope, may be NULL when Q and K_new are already rotated), ssv_verify_attn
 * (attn), then ssv_accept (acc, may be NULL), in that order on `stream`, with
 * the same arguments, results and workspaces as the three separate calls.
 * SimSD summary sections 2-4 (one verification pass: rotation with the
 * RoPE-copy index, temporal attention, acceptance in temporal order).
 *
 * The difference is overlap: each kernel is launched with programmatic
 * dependent launch and may begin its input-independent set-up while the one
 * before it finishes.  When the rotation's outputs (rope->q_out, k_out)
 * overlap none of attn->seqs, tau, k_cache, v_cache, the attention kernel
 * plans and starts streaming the KV cache before the rotation completes;
 * when neither the rotation's outputs nor attn->o or the attention
 * workspace overlap acc->tau, block, gamma, slot_off, noise_row, the
 * acceptance kernel builds its row list before the attention completes.
 * Everything else is read only after the preceding kernel has completed.
 * Kernels that ran before the call must be complete or ordered by the stream
 * as usual; nothing here relaxes that.
 * All arguments are validated before anything is launched.
 * Errors: those of the three calls.
 * ---------------------------------------------------------------------- */
SSV_API ssv_status ssv_verify_step(const ssv_rope_args* rope, const ssv_attn_args* attn, void* attn_workspace,
                                   size_t attn_workspace_bytes, const ssv_accept_args* acc, void* acc_workspace,
                                   size_t acc_workspace_bytes, void* stream);

/* ------------------------------------------------------------------------
 * ssv_accept_noalloc -- ssv_accept for callers that cannot allocate.
 * The pages have no counterpart: this is an interface addition of the
 * library.  Some callers have no way to obtain device memory of their own:
 * a host runtime that owns every byte of the GPU and hands its plugins no
 * allocator, or a latency-critical path where cudaMalloc (which can
 * synchronise the device) and allocating library routines are not allowed.
 * They pass inputs and outputs exactly as for ssv_accept but no workspace;
 * the scratch lives in a fixed 4 MiB array inside the library, which every
 * GPU that loads libssv holds until the process exits.
 *  - Same arguments, semantics and results as ssv_accept.
 *  - Calls whose scratch would exceed 4 MiB (roughly total_slots *
 *    ceil(V / 8192) > 120000 chunk records, e.g. more than ~6000 slots at
 *    V = 151936) return SSV_ERR_WORKSPACE and launch nothing.  Under REJECT
 *    the stored exponentials of the emitted rows (see ssv_accept) are kept
 *    only when they fit too; otherwise the second emission pass forms them
 *    again from the logits, with identical results.
 *  - Calls nothing that allocates: no cudaMalloc/cudaFree, no allocating
 *    library routine.  It clears its arrival counters with a memset on
 *    `stream` at every call.
 *  - The first call in each CUDA context looks up the array's device
 *    address (cudaGetSymbolAddress with that context current) and caches it
 *    per device together with the context; a later call from another
 *    context on that device (after cudaDeviceReset, or a context the caller
 *    made current) looks it up again.  Make the first call in a context
 *    before any stream capture.  Device ordinals of 64 and above are refused
 *    with SSV_ERR_INVALID.
 *  - All calls share the one array and it keeps the last call's contents:
 *    calls that overlap on the GPU (different streams or host threads)
 *    race and must be serialised by the caller.
 * ---------------------------------------------------------------------- */
SSV_API ssv_status ssv_accept_noalloc(const ssv_accept_args* a, void* stream);

/* ------------------------------------------------------------------------
 * ssv_commit -- commit of a verification pass into the KV cache.
 * SimSD summary, section 4 "Speculative decoding pipeline" (Acceptance: the
 * longest accepted prefix, in the temporal order the draft induces, is
 * committed and the loop repeats) and "Main contributions" 3 (composes with
 * a KV cache).  The pages give no cache layout; the reading taken: after
 * sequence b's pass (C cached rows, N fresh prompt rows, block B, stage map
 * tau, n_acc[b] accepted stages) its cache gains, appended after row C,
 *   - the keys / values of the N fresh prompt rows, in row order, then
 *   - those of the data rows of stages 1..n_acc, in stage order (stage s is
 *     slot k = tau^{-1}(s), fresh row N + k).
 * Mask rows are never committed.  Rows are copied as they are (keys keep the
 * rotation ssv_rope_copy gave them).  new_len[b] = C + N + n_acc[b].
 *
 * k_new, v_new [total_rows, Hkv, d]  device, dtype: the pass's fresh rows
 *                                     (post-RoPE keys), packed per sequence at
 *                                     seqs[b].q_off as for ssv_verify_attn
 * k_dst, v_dst [dst_rows, Hkv, d]    device, dtype: destination caches;
 *                                     sequence b's cache starts at row
 *                                     dst_off[b] and has dst_cap[b] rows of
 *                                     room (rows C .. C + N + n_acc - 1 of it
 *                                     are written, nothing else).  May be the
 *                                     k_cache / v_cache of ssv_verify_attn
 *                                     when its sequences were laid out with
 *                                     room (dst_off = kv_off).
 * seqs, tau, batch, total_rows as for ssv_verify_attn; n_acc [batch] device
 * (as written by ssv_accept); dst_off, dst_cap [batch] device; new_len
 * [batch] device, written (-1 for a sequence rejected on the device).
 * dtype SSV_F32 or SSV_BF16; d in {64, 128}; pointers 16-byte aligned.
 * k_new / v_new must not overlap k_dst / v_dst (checked), and the
 * destination ranges [dst_off[b], dst_off[b] + dst_cap[b]) of different
 * sequences must not overlap (not checked: overlapping ones race).
 * Errors: SSV_ERR_INVALID, SSV_ERR_CUDA; on device SSV_ERR_BAD_TAU (stage
 * map not a permutation of 1..B) and SSV_ERR_INVALID (B outside 1..64, a
 * stage map outside tau[0, total_slots), n_acc outside 0..B, or the
 * appended rows do not fit dst_cap / dst_rows): that sequence's rows are not
 * written and its new_len is -1.  No workspace; asynchronous on `stream`.
 * ---------------------------------------------------------------------- */
typedef struct {
  const void* k_new;
  const void* v_new;
  void* k_dst;
  void* v_dst;
  ssv_dtype dtype;
  int32_t Hkv, d;
  const ssv_seq* seqs;         /* device [batch] */
  int32_t batch;
  const int32_t* tau;          /* device [total_slots] */
  const int32_t* n_acc;        /* device [batch] */
  const int32_t* dst_off;      /* device [batch] */
  const int32_t* dst_cap;      /* device [batch] */
  int32_t* new_len;            /* device [batch], out */
  int32_t total_rows;          /* rows of k_new / v_new */
  int32_t total_slots;         /* entries of tau (sum of B) */
  int32_t dst_rows;            /* rows of k_dst / v_dst */
  int32_t* dev_status;         /* device, may be NULL */
} ssv_commit_args;

SSV_API ssv_status ssv_commit(const ssv_commit_args* a, void* stream);

/* ------------------------------------------------------------------------
 * ssv_lmhead_accept -- LM head over the mask slots fused with acceptance.
 * SimSD summary section 4 (the target scores every drafted position in one
 * pass; acceptance in the temporal order the draft induces); SPOT review
 * "How it is used" (state equality; coupled-noise match).  The pages do not
 * say how the logits are formed; the reading taken: the logits of mask slot
 * k are l_k = W h_k for the LM head W [V, hidden] and the slot's final
 * hidden state h_k.  This call computes, for every verified row (stage
 * <= min(gamma + 1, B)), the decision score over the whole vocabulary
 * without writing logits anywhere:
 *   ARGMAX : argmax_v l_k[v]                                   (ties: lowest v)
 *   GUMBEL : argmax_v fl32(fl32(l_k[v] / T) + noise[noise_row[k]][v])
 *            (IEEE fp32, no contraction; T = 0 means ARGMAX)
 * and then walks the stages exactly as ssv_accept (same n_acc, n_out,
 * tokens).  l_k is accumulated in fp32 on the tensor cores from the bf16
 * operands (exact products, fp32 sums in an unspecified order), so a
 * decision between two tokens whose scores differ by less than that
 * accumulation error may fall either way.  Rejection sampling is not
 * offered here (it needs the draft model's logits as well).
 *
 * hidden_states [total_slots, hidden] bf16 device, row = slot (slot order);
 *               only rows of verified stages are read (when some stages
 *               are not verified, a first kernel copies the verified rows
 *               into the workspace and the GEMM runs over those).
 * lm_head       [V, hidden] bf16 device, row-major.
 * draft_tokens, tau, noise_row: [total_slots] int32 device
 * block, gamma, slot_off: [batch] int32 device (as for ssv_accept)
 * noise [n_noise_rows, V] fp32 device (GUMBEL with T > 0 only, else NULL)
 * Outputs n_acc, n_out [batch], tokens [total_slots] as for ssv_accept.
 * Sizes: hidden % 64 == 0 and >= 64; 1 <= V; 1 <= total_slots <= 2048;
 *        batch <= 2048; pointers 16-byte aligned.
 * Workspace: ssv_lmhead_accept_workspace bytes, zero before first use.
 * Errors: SSV_ERR_INVALID (mode REJECT, sizes, null, alignment),
 *         SSV_ERR_NOT_FINITE (T), SSV_ERR_UNSUPPORTED (total_slots or batch
 *         above 2048), SSV_ERR_WORKSPACE, SSV_ERR_CUDA; on device
 *         SSV_ERR_BAD_TAU (that sequence's outputs are not written),
 *         SSV_ERR_INVALID (a verified slot's noise_row outside the table;
 *         likewise), SSV_ERR_TIMEOUT (a bounded wait ran out).
 * Scheduling: two kernels chained by programmatic dependent launch (a
 * gather of the verified rows, then the GEMM with one CTA per SM); the CTA
 * that finishes an M-tile last merges its rows; no CTA waits on another.
 * ---------------------------------------------------------------------- */
typedef struct {
  ssv_accept_mode mode;        /* SSV_ACCEPT_ARGMAX or SSV_ACCEPT_GUMBEL */
  float T;
  int32_t V;
  int32_t hidden;
  int32_t batch;
  int32_t total_slots;
  const void* hidden_states;   /* bf16 [total_slots, hidden] */
  const void* lm_head;         /* bf16 [V, hidden] */
  const int32_t* draft_tokens;
  const int32_t* tau;
  const int32_t* block;
  const int32_t* gamma;
  const int32_t* slot_off;
  const float* noise;
  int32_t n_noise_rows;
  const int32_t* noise_row;
  int32_t* n_acc;
  int32_t* n_out;
  int32_t* tokens;
  int32_t* dev_status;         /* device, may be NULL */
} ssv_lmhead_accept_args;

SSV_API ssv_status ssv_lmhead_accept_workspace(const ssv_lmhead_accept_args* a, size_t* bytes);
SSV_API ssv_status ssv_lmhead_accept(const ssv_lmhead_accept_args* a, void* workspace, size_t workspace_bytes,
                                     void* stream);

/* ------------------------------------------------------------------------
 * Tree (state-set) verification -- the verification pass over a draft tree
 * of block states and the acceptance by state equality.
 * SPOT review, "How it works" (the drafter grows a tree of candidate block
 * states, each edge committing one position with one token) and "How it is
 * used" (an edge (y, z) is accepted only if z is the target's next state
 * from y, so the accepted set is one path; coupled noise at T > 0); SimSD
 * summary section 2 (in a block state, the mask slot of an undecided
 * position sees the committed data tokens and the undecided mask slots).
 * Readings (the pages give neither a layout nor the target's choice of
 * position):
 *  - Tree of a sequence: E edges (0 <= E <= 63) over B positions
 *    (1 <= B <= 64); edge e hangs under node parent[e] + 1 (parent[e] = -1:
 *    the root, the block state before the pass; parent[e] < e) and commits
 *    position pos[e] (undecided there) with token token[e].  Node 0 is the
 *    root, node e + 1 the child of edge e.
 *  - Query rows at q_off: the N fresh prompt rows, then one mask-slot row per
 *    position p (its query is the same in every state).  New key / value rows
 *    at k_off: the N fresh rows, one data row per edge, one mask row per
 *    position.  Output rows at o_off: the N fresh rows (causal over cache and
 *    fresh prompt), then node-major rows (n, p), n = 0..E, p = 0..B-1: row
 *    (n, p), for p undecided at node n, is mask slot p attending the whole
 *    prompt, the data rows of the edges on the path root -> n and the mask
 *    rows of the positions undecided at n.  Rows of committed positions are
 *    not written.  A chain of edges in stage order gives SimSD's mask rows.
 *  - Target transition from node n: for each undecided p the decision token
 *    dec(n, p) of logits row (n, p) (argmax, or coupled-noise argmax with the
 *    noise row of position p) and its confidence l[dec] - logsumexp(l)
 *    (log-probability under softmax(l)); the most confident position wins
 *    (ties: the lowest).  The walk from the root follows the child edge
 *    carrying that (position, token) (the lowest such edge) while there is
 *    one, and emits the transition where there is none; a node with no
 *    undecided position ends the walk with nothing emitted.
 * Every kernel checks each sequence's extents and tree on the device; a
 * sequence that fails is skipped (its outputs are not written; the
 * acceptance sets n_acc = -1) and SSV_ERR_INVALID is reported.
 * ---------------------------------------------------------------------- */
typedef struct {
  int32_t cache_len;  /* C >= 0 */
  int32_t new_len;    /* N >= 0 */
  int32_t block;      /* B, 1 <= B <= 64 */
  int32_t n_edges;    /* E, 0 <= E <= 63 */
  int32_t q_off;      /* N + B query rows */
  int32_t k_off;      /* N + E + B new key / value rows */
  int32_t kv_off;     /* C cache rows */
  int32_t edge_off;   /* E entries of parent / pos / token */
  int32_t o_off;      /* N + (E + 1) B output rows (and logits rows) */
} ssv_tree_seq;

/* ssv_tree_verify_attn -- the attention of the tree pass.
 * q [total_q, Hq, d], k_new / v_new [total_k, Hkv, d], k_cache / v_cache
 * [total_cache, Hkv, d] device, in_dtype (post-RoPE); o [total_out, Hq, d]
 * device, out_dtype.  parent, pos [total_edges] int32 device.  Sequences in
 * increasing q_off order.  d in {64, 128}, Hq % Hkv == 0, pointers 16-byte
 * aligned; max_cache bounds every C.
 * The part every row shares -- the prompt (cache + fresh rows), the same keys
 * for a mask slot at every node -- is computed once per query row: for bf16
 * inputs with d = 128 on the tensor cores (the verify attention's schedule
 * in a prompt-only form, bf16 P and fp32 accumulation as there), which then
 * leaves each row's normalised output and log-sum-exp in the workspace; a
 * node kernel (fp32) continues that softmax over each node's tail keys.
 * Other inputs run the prompt part in the node kernel itself (fp32 SIMT).
 * Workspace: ssv_tree_verify_attn_workspace bytes (0 when the prompt part
 * runs in fp32), 256-byte aligned, all-zero before its first use and left
 * reusable (as for ssv_verify_attn).
 * Errors: SSV_ERR_INVALID, SSV_ERR_UNSUPPORTED, SSV_ERR_WORKSPACE,
 * SSV_ERR_CUDA; on device SSV_ERR_INVALID (see above). */
typedef struct {
  const void* q;
  const void* k_cache;
  const void* v_cache;
  const void* k_new;
  const void* v_new;
  void* o;
  ssv_dtype in_dtype;
  ssv_dtype out_dtype;
  int32_t Hq, Hkv, d;
  float scale;                 /* 0 => 1/sqrt(d) */
  const ssv_tree_seq* seqs;    /* device [batch] */
  int32_t batch;
  const int32_t* parent;       /* device [total_edges] */
  const int32_t* pos;          /* device [total_edges] */
  int32_t total_q, total_k, total_cache, total_edges, total_out;
  int32_t max_cache;
  int32_t* dev_status;         /* device, may be NULL */
} ssv_tree_attn_args;

SSV_API ssv_status ssv_tree_verify_attn_workspace(const ssv_tree_attn_args* a, size_t* bytes);
SSV_API ssv_status ssv_tree_verify_attn(const ssv_tree_attn_args* a, void* workspace, size_t workspace_bytes,
                                        void* stream);

/* ssv_tree_accept -- acceptance of the tree by state equality.
 * logits [total_out, V] device (row (n, p) of sequence b at o_off + N + n B + p,
 * the numbering of the attention's output rows; fresh rows are not read).
 * mode SSV_ACCEPT_ARGMAX or SSV_ACCEPT_GUMBEL (coupled noise: the table row of
 * position p of sequence b is noise_row[pos_off[b] + p]; T = 0 means argmax).
 * parent, pos, token [total_edges] int32 device.
 * Outputs (device): n_acc [batch] (accepted edges, -1 for a rejected
 * sequence); path [batch * 64] (the accepted edges' ids within the sequence,
 * root first, -1 padded); emit_pos, emit_tok [batch] (the target's
 * transition where the walk stopped, -1 if none).
 * Workspace: ssv_tree_accept_workspace bytes, 256-byte aligned (no state is
 * kept between calls).  Errors: SSV_ERR_INVALID, SSV_ERR_NOT_FINITE,
 * SSV_ERR_WORKSPACE, SSV_ERR_CUDA; on device SSV_ERR_INVALID. */
typedef struct {
  ssv_accept_mode mode;
  float T;
  int32_t V;
  const ssv_tree_seq* seqs;    /* device [batch] */
  int32_t batch;
  ssv_dtype logits_dtype;
  const void* logits;
  const int32_t* parent;
  const int32_t* pos;
  const int32_t* token;
  int32_t total_edges;
  int32_t total_out;
  const float* noise;          /* [n_noise_rows, V] fp32 (GUMBEL, T > 0) */
  int32_t n_noise_rows;
  const int32_t* noise_row;    /* [total_positions] */
  const int32_t* pos_off;      /* [batch] */
  int32_t total_positions;
  int32_t* n_acc;
  int32_t* path;
  int32_t* emit_pos;
  int32_t* emit_tok;
  int32_t* dev_status;         /* device, may be NULL */
} ssv_tree_accept_args;

SSV_API ssv_status ssv_tree_accept_workspace(const ssv_tree_accept_args* a, size_t* bytes);
SSV_API ssv_status ssv_tree_accept(const ssv_tree_accept_args* a, void* workspace, size_t workspace_bytes,
                                   void* stream);

/* ------------------------------------------------------------------------
 * ssv_set_fault_injection -- test support for failure detection.
 * The pages have no counterpart: this lets a test make a bounded device wait
 * run out without faulting, trapping or hanging the GPU.  For the chosen
 * kernel -- the tensor-core attention (SSV_FAULT_ATTN), the streaming
 * acceptance reduce (SSV_FAULT_ACCEPT) or the fused LM head's GEMM
 * (SSV_FAULT_LMHEAD) -- every bounded wait gives up after
 * wait_budget_cycles SM cycles instead of about one second, and, if
 * skip >= 0, CTA 0 leaves out one asynchronous copy: its skip-th key block
 * (attention), its skip-th vocabulary chunk (acceptance) or its skip-th
 * operand stage (LM head), so that the wait for that copy runs out.  The
 * kernel then drains every copy and MMA it issued (bounded), releases its
 * tensor memory, writes SSV_ERR_TIMEOUT to dev_status and returns; its
 * outputs are unspecified and its workspace counters must be cleared before
 * the workspace is used again (as after any SSV_ERR_TIMEOUT).
 * The setting is process-wide and applies to every later launch of that
 * kernel from every host thread, until reset with NULL.  For tests only.
 * f: kernel in SSV_FAULT_NONE..SSV_FAULT_LMHEAD, skip >= -1,
 *    1000 <= wait_budget_cycles <= 2^31.  Errors: SSV_ERR_INVALID.
 * ---------------------------------------------------------------------- */
typedef enum {
  SSV_FAULT_NONE = 0,
  SSV_FAULT_ATTN = 1,
  SSV_FAULT_ACCEPT = 2,
  SSV_FAULT_LMHEAD = 3
} ssv_fault_kernel;

typedef struct {
  ssv_fault_kernel kernel;
  int32_t skip;                /* index of the copy CTA 0 leaves out, or -1 */
  int64_t wait_budget_cycles;  /* budget of every bounded wait of that kernel */
} ssv_fault_injection;

SSV_API ssv_status ssv_set_fault_injection(const ssv_fault_injection* f);

/* ------------------------------------------------------------------------
 * Status and utilities
 * ---------------------------------------------------------------------- */
/* Waits for `stream`, reads the device status word, resets it to 0 and
 * returns it (SSV_OK if dev_status is NULL). */
SSV_API ssv_status ssv_get_status(int32_t* dev_status, void* stream);

SSV_API const char* ssv_status_string(ssv_status s);

/* Library build identification, e.g. "ssv 0.2 sm_103a". */
SSV_API const char* ssv_version(void);

/* ------------------------------------------------------------------------
 * ssv_bench -- native timing of the library on a named synthetic workload
 * ("tiny", "gqa1p7b", "gqa8b", "prefill", "sweep").  Allocates its own
 * device buffers (this is not a hot-path call), fills them with a
 * counter-hash generator, runs `iters` timed iterations per op with an L2
 * flush between them and writes one JSON object (median/p10/p90 times,
 * algorithmic bytes and FLOPs) into json_out.  The DFlash review's latency
 * model L = (T_draft + T_verify) / tau needs T_verify; this reports it.
 * Errors: SSV_ERR_INVALID (unknown config, short buffer), SSV_ERR_CUDA.
 * ---------------------------------------------------------------------- */
SSV_API ssv_status ssv_bench(const char* config, int32_t iters, char* json_out, size_t json_len);

/* ------------------------------------------------------------------------
 * ssv_stream_read -- the measurement reference for a memory-bound kernel
 * of the path: reads `bytes` at device address `buf` once (16-byte loads,
 * two CTAs per SM, each a contiguous range) and XORs every word read into
 * *out (device address; a checksum that keeps the loads live, not a result
 * of the method).  Timed like the kernel it is compared with (same L2
 * flush, same launch mode), it gives the achievable time for reading those
 * bytes, launch and first-byte latency included; on small workloads that is
 * well above bytes / peak bandwidth.  Not a hot-path call.  buf must be
 * 16-byte aligned and bytes a multiple of 16.  Asynchronous on `stream`.
 * Errors: SSV_ERR_INVALID (null or misaligned arguments), SSV_ERR_CUDA.
 * ---------------------------------------------------------------------- */
SSV_API ssv_status ssv_stream_read(const void* buf, size_t bytes, uint32_t* out, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* SSV_H_ */
