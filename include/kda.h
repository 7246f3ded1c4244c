/*
 * kda.h -- C ABI of libkda: the KDA (Kimi Delta Attention) linear-attention mixer step on one
 * GB300 (sm_103a).
 *
 * What the step computes, per sequence b, head h and token t (the pages name the steps; the
 * formulas are the plain gated delta-rule reading of them):
 *   f_b decay projection   graw = W_fb[h] . f_a                          ("KDA fuses the f_b
 *   decay gate             alpha = exp(-exp(A_log[h]) * softplus(graw + dt_bias))   projection,
 *   short causal conv      q,k,v = SiLU(depthwise conv over the last 4 inputs)      convolution,
 *   L2 norms               k /= |k|;  q /= |q| * sqrt(dk)                           FP32 recurrence
 *   FP32 recurrence        S <- Diag(alpha) S;  u = v - S^T k;  S += beta k u^T;    and gated output
 *                          o = S^T q,  beta = sigmoid(beta_logit)                   normalization")
 *   gated output RMSNorm   y = o / rms(o) * norm_w * sigmoid(gate)
 * Sources, cited by page title and section:
 *   [NVFP4-K3] "vsabavat/TensorRT-LLM pull request 1: NVFP4 Kimi K3 targets", Description
 *              (the fused step; FP32 or BF16 recurrent-state storage; FP32 recurrence and FP32
 *              per-token draft records with either storage dtype; typed state stores).
 *   [K3-Rubin] "NVIDIA/TensorRT-LLM pull request 21996: Kimi K3 NVFP4 on Rubin (SM107)", section 3
 *              (KDA mixer with prefill, MTP-decode and fused-projection kernels).
 *   [K3-V2]    "NVIDIA/TensorRT-LLM pull request 19841: Kimi K3 on modeling_v2", section 1
 *              (stateful entries take caller-owned state created before graph capture), section 5
 *              (KDA verify kernels and per-token verify states), section 6 (the KDA mixer returns
 *              its output before o_proj).
 *
 * Conventions for every entry point:
 *   - All tensor pointers are DEVICE pointers owned by the caller; the library allocates
 *     nothing, never synchronises the stream and never reads device memory on the host, so
 *     every call can be captured in a CUDA graph.  `stream` is a cudaStream_t (NULL = legacy
 *     default stream).
 *   - Only dk = dv = 128, r = 128 and conv_size = 4 are supported (KDA_ERR_UNSUPPORTED
 *     otherwise).  Every pointer must be 16-byte aligned and tensors dense row-major.
 *   - Host-visible argument errors return KDA_ERR_INVALID_ARG / KDA_ERR_UNSUPPORTED before
 *     anything is launched; kda_last_error() gives a one-line reason.
 *   - Device data that the host cannot see (slot ids, accepted lengths) is checked in the
 *     kernel: a bad value sets a bit in *pool->err_word and that (sequence, head) tile is
 *     skipped (no trap).  kda_get_error() reads and clears the word.
 *   - Two sequences of one call must not name the same slot (the result is undefined).
 *   - Launch ordering: the kernels of kda_decode, kda_verify, kda_commit and the resume entries
 *     are launched with programmatic dependent launch.  They may start while the kernel
 *     launched before them on the stream is still finishing.  Those that take a layer read its
 *     weights (W_fb, W_fb_scale, A_log, dt_bias, conv_w, norm_w) before waiting for that kernel;
 *     everything else is read for use after the wait (a slot id or accepted length read
 *     earlier only aims an L2 prefetch).  So the weights must not be written by the kernel
 *     launched just before the call on the same stream.  Write them earlier, or separate the
 *     two with an event or a synchronisation.
 *   - Layouts: q, k [.., H*dk]; v, gate, out [.., H*dv]; f_a [.., r]; beta_logit [.., H];
 *     all BF16.  Head h owns channels [h*dk, (h+1)*dk) of q and k and [h*dv, (h+1)*dv) of v,
 *     gate and out.
 */
#ifndef KDA_H
#define KDA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    KDA_OK = 0,
    KDA_ERR_INVALID_ARG = 1,   /* null / misaligned pointer, bad size, bad dtype */
    KDA_ERR_UNSUPPORTED = 2,   /* valid request this build does not implement (dims) */
    KDA_ERR_CUDA = 3,          /* a CUDA runtime call failed (launch error, no device) */
    KDA_ERR_DEVICE = 4         /* kda_get_error() found device-side error bits */
} kda_status;

typedef enum { KDA_STATE_F32 = 0, KDA_STATE_BF16 = 1 } kda_state_dtype;

/* Storage of the f_b projection weights W_fb: BF16, or FP8 E4M3 codes with one FP32 scale per
 * row (the FP8 input path: "FP8 projection weights", [NVFP4-K3] Description; the scale
 * granularity is this library's reading). */
typedef enum { KDA_W_BF16 = 0, KDA_W_FP8_E4M3 = 1 } kda_weight_dtype;

/* Device-side error bits OR-ed into *err_word. */
#define KDA_DEVERR_SLOT      0x1   /* slot id outside [0, num_slots) */
#define KDA_DEVERR_ACCEPTED  0x2   /* accepted length outside [0, T] */
#define KDA_DEVERR_TIMEOUT   0x4   /* an on-chip wait gave up (bounded at 2 s); results invalid */
#define KDA_DEVERR_DECAY     0x8   /* kda_prefill, kda_prefill_varlen: a non-finite per-token
                                      log-decay (NaN inputs, or exp(A_log) beyond FP32); the results
                                      of that chunk and of the sequence after it are invalid.  Any
                                      finite decay is handled. */
#define KDA_DEVERR_TOKENS    0x10  /* kda_verify_resume: n_tokens[b] outside [1, T]; sequence skipped */
#define KDA_DEVERR_SEQLEN    0x20  /* kda_prefill_varlen: cu_seqlens inconsistent for a sequence
                                      (negative, decreasing, past total_tokens or longer than
                                      max_len); that sequence is skipped */

/* Weights of one KDA layer (read only). */
typedef struct {
    int32_t num_heads;      /* H >= 1 */
    int32_t head_k_dim;     /* dk, must be 128 */
    int32_t head_v_dim;     /* dv, must be 128 */
    int32_t fa_rank;        /* r, rank of the f_a/f_b decay factorisation, must be 128 */
    int32_t conv_size;      /* taps of the short convolution, must be 4 */
    const void *W_fb;       /* [H*dk, r] in w_fb_dtype: f_b projection, row i of head h = row h*dk+i */
    const float *A_log;     /* fp32 [H] */
    const float *dt_bias;   /* fp32 [H*dk] */
    const void *conv_w;     /* bf16 [3, H*dk, conv_size]: q, k, v depthwise weights, tap
                               conv_size-1 multiplies the current token */
    const float *norm_w;    /* fp32 [dv]: output RMSNorm weight, shared by the heads */
    float l2_eps;           /* q/k L2-norm epsilon (inside the square root), e.g. 1e-6 */
    float norm_eps;         /* output RMSNorm epsilon, e.g. 1e-5 */
    int32_t w_fb_dtype;     /* kda_weight_dtype of W_fb */
    const float *W_fb_scale;/* fp32 [H*dk] with KDA_W_FP8_E4M3: row h*dk+i of W_fb is
                               W_fb_scale[h*dk+i] times its E4M3 codes (16-byte aligned);
                               ignored with KDA_W_BF16 (may be NULL) */
} kda_layer;

/* Caller-owned pool of recurrent-state slots (one slot per live sequence). */
typedef struct {
    void *state;            /* [num_slots, H, dk, dv] in state_dtype; dv contiguous */
    int32_t state_dtype;    /* kda_state_dtype: storage only, compute is FP32 either way */
    void *conv_state;       /* bf16 [num_slots, 3, conv_size-1, H*dk]: the last conv_size-1
                               pre-conv q, k, v inputs, oldest first */
    int32_t num_slots;
    int32_t *err_word;      /* device int32, zero-initialised by the caller */
} kda_pool;

/* Single-token decode for B sequences ([NVFP4-K3] Description; [K3-V2] section 6).
 * Reads and updates in place, for each b, the state and conv window of slot slot_ids[b].
 *   slot_ids  int32 [B] (device)
 *   q, k      bf16 [B, H*dk]   pre-conv inputs
 *   v, gate   bf16 [B, H*dv]
 *   f_a       bf16 [B, r]      f_a output (shared by the heads)
 *   beta_logit bf16 [B, H]
 *   out       bf16 [B, H*dv]   gated, RMS-normalised mixer output (before o_proj)
 * B = 0 is a no-op.  With a BF16 pool the state is rounded to BF16 (nearest even) once per
 * call, after the FP32 update. */
kda_status kda_decode(const kda_layer *layer, const kda_pool *pool, const int32_t *slot_ids,
                      int32_t B, const void *q, const void *k, const void *v, const void *f_a,
                      const void *beta_logit, const void *gate, void *out, void *stream);

/* Multi-token draft verify ([NVFP4-K3] Description; [K3-V2] section 5).  Runs T draft tokens
 * per sequence, in order, from the state and conv window of slot slot_ids[b], keeping the
 * state in FP32 between tokens, and records after each token:
 *   rec_state fp32 [B, T, H, dk, dv]  the FP32 state after token t (either storage dtype)
 *   rec_conv  bf16 [B, T, 3, conv_size-1, H*dk]  the conv window after token t
 *   out       bf16 [B, T, H*dv]
 * Inputs are laid out [B, T, ...].  The pool is not modified (see kda_commit).  1 <= T <= 16.
 * Record t equals the state after t + 1 kda_decode calls on the same tokens to FP32 rounding (the
 * f_b projection of the draft tokens is summed on the tensor cores here). */
kda_status kda_verify(const kda_layer *layer, const kda_pool *pool, const int32_t *slot_ids,
                      int32_t B, int32_t T, const void *q, const void *k, const void *v,
                      const void *f_a, const void *beta_logit, const void *gate, void *out,
                      float *rec_state, void *rec_conv, void *stream);

/* Commit accepted draft lengths after kda_verify.  For each b with n = accepted[b] >= 1:
 * slot state <- record [b, n-1] (bit copy for an FP32 pool, round-to-nearest-even for a BF16
 * pool) and slot conv window <- conv record [b, n-1].  n = 0 leaves the slot untouched.
 *   accepted int32 [B] (device), each in [0, T]; an out-of-range value sets
 *   KDA_DEVERR_ACCEPTED and that sequence is skipped.
 * num_heads / head dims / conv_size must match the records' layout. */
kda_status kda_commit(const kda_pool *pool, int32_t num_heads, int32_t head_k_dim,
                      int32_t head_v_dim, int32_t conv_size, const int32_t *slot_ids,
                      const int32_t *accepted, int32_t B, int32_t T, const float *rec_state,
                      const void *rec_conv, void *stream);

/* Decode that first commits the previous step's drafts ("fused commit into the next step").
 * For each b, with n = prev_accepted[b]:
 *   n >= 1: the step starts from record [b, n-1] of the previous kda_verify / kda_verify_resume
 *           (state rounded to the pool's storage dtype exactly as kda_commit stores it, and the
 *           conv-window record), not from the slot;
 *   n == 0: the step starts from slot slot_ids[b].
 * Then one token is decoded as by kda_decode and the slot receives the new state and window.
 * The result equals kda_commit(prev_accepted) followed by kda_decode, bit for bit, without the
 * commit's extra pass over the state (one read of the record and one write of the slot per
 * tile).  The pages fuse no commit; decode and draft verify are theirs ([NVFP4-K3] Description;
 * [K3-V2] section 5).
 *   prev_accepted  int32 [B] (device), each in [0, prev_T]; NULL = every n is 0.  An out-of-range
 *                  value sets KDA_DEVERR_ACCEPTED and that sequence is skipped (slot untouched).
 *   prev_rec_state fp32 [B, prev_T, H, dk, dv], prev_rec_conv bf16 [B, prev_T, 3, conv_size-1,
 *                  H*dk]: the previous step's records (may be NULL when prev_accepted is NULL).
 *   other arguments as kda_decode.  The records are only read. */
kda_status kda_decode_resume(const kda_layer *layer, const kda_pool *pool, const int32_t *slot_ids,
                             int32_t B, const int32_t *prev_accepted, int32_t prev_T,
                             const float *prev_rec_state, const void *prev_rec_conv,
                             const void *q, const void *k, const void *v, const void *f_a,
                             const void *beta_logit, const void *gate, void *out, void *stream);

/* Draft verify that first commits the previous step's drafts, with a per-sequence token count
 * so that one launch serves a mixed step (sequences decoding one token next to sequences
 * verifying drafts; the pages' mixed steps run their KDA decode kernel, [K3-V2] manual 16-rank
 * reference, part 5).  For each b, with n = prev_accepted[b]:
 *   n >= 1: slot slot_ids[b] <- record [b, n-1] of the previous step (as kda_commit) and the
 *           verify starts from that state and window;
 *   n == 0: the verify starts from the slot, which is left untouched.
 * Then tokens t < n_tokens[b] (all T when n_tokens is NULL) run as in kda_verify, writing
 * out[b, t] and the records [b, t]; entries t >= n_tokens[b] of out and of the records are not
 * written.  A one-token sequence is a decode step whose commit is the next step's n = 1 (its
 * result equals kda_decode's to FP32 rounding: the verify forms sum the f_b projection on the
 * tensor cores, decode with FMA chains).
 * Equals kda_commit(prev_accepted) followed by kda_verify, bit for bit, on the tokens run.
 *   n_tokens  int32 [B] (device) in [1, T], or NULL; out of range sets KDA_DEVERR_TOKENS and the
 *             sequence is skipped (after its commit).
 *   prev_*    as kda_decode_resume.  The previous records must not overlap rec_state / rec_conv.
 *   other arguments as kda_verify. */
kda_status kda_verify_resume(const kda_layer *layer, const kda_pool *pool, const int32_t *slot_ids,
                             int32_t B, int32_t T, const int32_t *n_tokens,
                             const int32_t *prev_accepted, int32_t prev_T,
                             const float *prev_rec_state, const void *prev_rec_conv,
                             const void *q, const void *k, const void *v, const void *f_a,
                             const void *beta_logit, const void *gate, void *out,
                             float *rec_state, void *rec_conv, void *stream);

/* Chunked prefill ([K3-Rubin] section 3).  L tokens per sequence, starting from the state and
 * conv window held in slot slot_ids[b] (zero them for a fresh sequence) and leaving the final
 * state (rounded once to the storage dtype) and conv window there.
 *   q, k [B, L, H*dk]; v, gate, out [B, L, H*dv]; f_a [B, L, r]; beta_logit [B, L, H]
 *   chunk      tokens per chunk of the chunked (WY) form; must be 64
 *   workspace  device scratch of at least kda_prefill_workspace_size(...) bytes, 256-byte
 *              aligned, owned by the caller; its contents need no initialisation.
 * L = 0 or B = 0 is a no-op. */
size_t kda_prefill_workspace_size(const kda_layer *layer, int32_t B, int32_t L, int32_t chunk);
kda_status kda_prefill(const kda_layer *layer, const kda_pool *pool, const int32_t *slot_ids,
                       int32_t B, int32_t L, int32_t chunk, const void *q, const void *k,
                       const void *v, const void *f_a, const void *beta_logit, const void *gate,
                       void *out, void *workspace, size_t workspace_bytes, void *stream);

/* Variable-length chunked prefill: B sequences of different lengths, packed one after another
 * (the chunked prefill of [K3-Rubin] section 3 over the ragged batches a server forms).
 * Sequence b is rows cu_seqlens[b] .. cu_seqlens[b+1]-1 of the packed inputs; it continues
 * from the state and conv window of slot slot_ids[b] (zero them for a fresh sequence) and
 * leaves its final state and window there, exactly as kda_prefill does for one sequence.
 *   cu_seqlens  int32 [B+1] (device): cu_seqlens[0] = 0, non-decreasing, cu_seqlens[B] <=
 *               total_tokens.  A zero-length sequence leaves its slot untouched.
 *   max_len     a host-side bound on every length (sizes the launch; no device read).
 *   A sequence longer than max_len, or whose offsets cu_seqlens[b-1..b+1] are out of order or
 *   outside [0, total_tokens], sets KDA_DEVERR_SEQLEN and is skipped.  Offsets that decrease
 *   further away can make two sequences share rows: their outputs are then undefined, but no
 *   access leaves the arguments' extents.
 *   q, k [total_tokens, H*dk]; v, gate, out [total_tokens, H*dv]; f_a [total_tokens, r];
 *   beta_logit [total_tokens, H]
 *   workspace   at least kda_prefill_varlen_workspace_size(layer, B, total_tokens, chunk)
 *               bytes, 256-byte aligned, caller-owned, no initialisation needed.
 * B = 0 or total_tokens = 0 is a no-op. */
size_t kda_prefill_varlen_workspace_size(const kda_layer *layer, int32_t B, int32_t total_tokens,
                                         int32_t chunk);
kda_status kda_prefill_varlen(const kda_layer *layer, const kda_pool *pool, const int32_t *slot_ids,
                              int32_t B, const int32_t *cu_seqlens, int32_t total_tokens,
                              int32_t max_len, int32_t chunk, const void *q, const void *k,
                              const void *v, const void *f_a, const void *beta_logit,
                              const void *gate, void *out, void *workspace,
                              size_t workspace_bytes, void *stream);

/* kda_prefill for callers that cannot allocate device memory (no counterpart in the pages:
 * this is a service of this library).  Code inside a CUDA-graph capture, runtimes that reserve
 * a fixed memory budget before serving, or hosts without an allocator of their own cannot
 * provide the prefill's scratch workspace; this entry point uses a scratch region compiled into
 * the library instead and allocates nothing (no cudaMalloc / cudaFree, no allocating library
 * routine).
 *   - The region holds kda_prefill_noalloc_max_bytes() bytes (64 MiB); every GPU that loads
 *     the library keeps it until the process exits.  Calls whose scratch need
 *     (kda_prefill_workspace_size) exceeds it return KDA_ERR_UNSUPPORTED with a message in
 *     kda_last_error(); e.g. H = 8 allows 56 chunks of 64 tokens (3,584 tokens) per call, summed
 *     over the batch with each sequence rounded up to whole chunks.
 *   - The first call on a device looks up the region's device address for that device (with
 *     the device current).  With lazy module loading (CUDA's default) that first call is also
 *     when the device reserves the region, so it can return KDA_ERR_CUDA (out of memory) under
 *     an allocator that already holds the device: make one call at start-up, before any stream
 *     capture or allocator reservation.  A cudaDeviceReset of a device the library has used
 *     invalidates the looked-up address; calls after it are not supported.
 *   - All calls share the region: calls whose kernels can overlap on the GPU (different
 *     streams without ordering) race.  Nothing in it needs clearing between calls.
 * Arguments and results are those of kda_prefill. */
size_t kda_prefill_noalloc_max_bytes(void);
kda_status kda_prefill_noalloc(const kda_layer *layer, const kda_pool *pool, const int32_t *slot_ids,
                               int32_t B, int32_t L, int32_t chunk, const void *q, const void *k,
                               const void *v, const void *f_a, const void *beta_logit,
                               const void *gate, void *out, void *stream);

/* Reads *pool->err_word into *host_err, then clears it (synchronises `stream`).  Returns
 * KDA_ERR_DEVICE when the word was nonzero, KDA_OK otherwise. */
kda_status kda_get_error(const kda_pool *pool, int32_t *host_err, void *stream);

/* Static string for a status code. */
const char *kda_status_string(kda_status s);

/* One-line description of the last host-side argument error on this thread ("" if none). */
const char *kda_last_error(void);

/* ABI version of this header (incremented on any incompatible change). */
#define KDA_ABI_VERSION 3
int32_t kda_abi_version(void);

#ifdef __cplusplus
}
#endif
#endif /* KDA_H */
