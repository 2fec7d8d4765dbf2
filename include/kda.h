/*
 * kda.h -- C ABI of libkda: Kimi Delta Attention (KDA) prefill and decode on
 * NVIDIA GB300 (sm_103a).
 *
 * The operation (Kimi K3 -- Architecture Notes, section 1.1 "Kimi Delta
 * Attention", the two displayed equations), per sequence and per head:
 *
 *     S_t = (I - beta_t k_t k_t^T) Diag(alpha_t) S_{t-1} + beta_t k_t v_t^T
 *     o_t = scale * S_t^T q_t
 *
 * S is the d_k x d_v fp32 recurrent state (same section: S in R^{d_k x d_v},
 * fixed size). alpha_t = exp(g_t) is channel-wise over the d_k key channels,
 * with g_t = max(log_alpha_t, lower_bound) (section 1.2 "The lower-bounded
 * decay": g >= g_min = -5); a NaN log_alpha is not clamped and propagates.
 * beta_t is one scalar per (token, head). q and k are expected L2-normalised
 * by the caller (section 1.1); the library does not normalise them. `scale`
 * multiplies the read-out (the pages print none: pass 1).
 *
 * Conventions shared by every entry point:
 *  - All tensor pointers are DEVICE pointers owned by the caller, contiguous,
 *    16-byte aligned. The library never allocates device memory and keeps no
 *    per-call state; it only enqueues kernels on `stream` (a cudaStream_t,
 *    passed as void*; NULL = the legacy default stream).
 *  - Argument errors are detected on the host before anything is enqueued and
 *    return KDA_ERR_INVALID_ARG or KDA_ERR_UNSUPPORTED; nothing is written.
 *    Launch failures return KDA_ERR_CUDA. Errors found by a kernel while it
 *    runs (a bounded wait that gave up) are recorded in a device error word
 *    that kda_check_device_error() reads.
 *  - in_dtype is the element type of q, k and v; out_dtype that of out (each
 *    KDA_BF16 = bfloat16 or KDA_F32 = float). log_alpha, beta and the states
 *    are always float (fp32). Results are accumulated in fp32; bf16 outputs are
 *    rounded to nearest-even. A bf16 output carries a relative rounding error
 *    of up to 2^-9 per element on top of the computation's own error.
 *  - Outputs must not alias inputs, except that final_state may equal
 *    init_state (in-place continuation of a prefill). Every entry point checks
 *    the byte ranges it is given and returns KDA_ERR_INVALID_ARG on an overlap.
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
  KDA_ERR_INVALID_ARG = 1, /* null/misaligned pointer, bad size, bad enum          */
  KDA_ERR_UNSUPPORTED = 2, /* valid but outside what the kernels implement        */
  KDA_ERR_CUDA = 3,        /* a CUDA runtime call or kernel launch failed          */
  KDA_ERR_TIMEOUT = 4,     /* a kernel's bounded wait gave up (device error word)  */
  KDA_ERR_RANGE = 5        /* an input was outside the range the kernel that ran
                              computes exactly (device error word; see kda_prefill) */
} kda_status;

typedef enum { KDA_F32 = 0, KDA_BF16 = 1 } kda_dtype;

/*
 * kda_prefill -- the chunkwise-parallel prefill form over packed
 * variable-length sequences (Kimi K3 -- Architecture Notes, section 1.2: the
 * kernel is recurrent across chunks and parallel within each chunk).
 *
 *   q, k        [total_tokens, H, d_k]   in_dtype
 *   v           [total_tokens, H, d_v]   in_dtype
 *   log_alpha   [total_tokens, H, d_k]   fp32, clamped below at lower_bound
 *   beta        [total_tokens, H]        fp32
 *   cu_seqlens  [num_seqs + 1]           int32, device; cu_seqlens[0] = 0,
 *               non-decreasing, cu_seqlens[num_seqs] = total_tokens. Sequence
 *               n is tokens cu_seqlens[n] .. cu_seqlens[n+1]-1; empty
 *               sequences are allowed (their final state equals their initial
 *               state). The library trusts these values (it cannot read device
 *               memory before enqueueing): malformed offsets are undefined.
 *   init_state  [num_seqs, H, d_k, d_v]  fp32, or NULL for zeros
 *   out         [total_tokens, H, d_v]   out_dtype, written
 *   final_state [num_seqs, H, d_k, d_v]  fp32, written, or NULL to skip
 *   workspace   device scratch of workspace_bytes bytes (16-byte aligned), or
 *               NULL with workspace_bytes = 0. Its size comes from
 *               kda_prefill_workspace_size(); with at least that much the
 *               library may use its parallel schedules (one long sequence split
 *               into segments over more SMs, see kda_prefill_workspace_size),
 *               with less it runs one CTA per (sequence, head) chain. The
 *               contents need no initialisation and are garbage afterwards; the
 *               workspace must not overlap any tensor argument and may not be
 *               shared by calls that run at the same time.
 *
 * Sizes: 1 <= d_k, d_v <= 128, H >= 1, num_seqs >= 0, total_tokens >= 0.
 * bf16 inputs with d_k = d_v = 128 and lower_bound >= -5 run the tensor-core
 * chunked kernel; every other supported case (fp32 inputs, other head sizes, a
 * lower bound below -5) runs the fp32 token-recurrent kernel.
 *
 * Range of the chunked kernel. It rescales keys and queries around one
 * reference point per 32-token chunk; with every clamped log-decay in
 * [lower_bound, 0] (alpha a retention factor in (0, 1], section 1.1) the
 * factors stay within e^80 (section 1.2) and every operand is finite. It also
 * computes exactly any clamped log-decay up to +1/3 (so that no operand of a
 * 32-token chunk can exceed 2^15.5, inside fp16). A clamped log-decay above
 * +1/3 may overflow an operand: the kernel then records KDA_ERR_RANGE in the
 * device error word (kda_check_device_error reports it) and the results of
 * that call are unspecified. A retention factor above one also makes the state
 * grow: the chunked kernel multiplies the state by its chunk operands through an
 * fp16 copy, so state entries must stay below 65504 in magnitude (with alpha <= 1
 * and unit-norm keys the state's norm grows by at most beta_t |v_t| per token).
 * The token-recurrent kernel (kda_prefill_recurrent) takes any finite log-decay
 * and keeps the state in fp32 throughout.
 * Enqueues work on `stream` and returns without synchronising.
 */
kda_status kda_prefill(const void *q, const void *k, const void *v, const float *log_alpha,
                       const float *beta, const int32_t *cu_seqlens, int32_t num_seqs,
                       int64_t total_tokens, int32_t H, int32_t d_k, int32_t d_v,
                       kda_dtype in_dtype, kda_dtype out_dtype, float lower_bound, float scale,
                       const float *init_state, void *out, float *final_state, void *workspace,
                       size_t workspace_bytes, void *stream);

/*
 * kda_prefill_workspace_size -- bytes of device scratch that let kda_prefill
 * (and kda_prefill_ex) use their parallel schedules for these sizes; 0 when
 * none applies (then no workspace is needed). Pure host function, no CUDA
 * call; the same arguments always give the same answer.
 */
size_t kda_prefill_workspace_size(int64_t total_tokens, int32_t num_seqs, int32_t H, int32_t d_k,
                                  int32_t d_v);

/*
 * kda_prefill_noalloc -- kda_prefill for callers that cannot allocate device memory.
 *
 * Some callers cannot produce the workspace kda_prefill asks for: a serving engine that
 * reserves the whole GPU up front in its own pool and refuses any further cudaMalloc, a
 * plugin inside a host framework that owns every device allocation, or code in a
 * latency-critical region where cudaMalloc/cudaFree would stall or synchronise the device.
 * This entry point takes the same arguments as kda_prefill without the workspace, runs the
 * same validation, schedule and kernels, and allocates nothing (no cudaMalloc, cudaFree or
 * allocating library routine): its scratch is a 16 MiB array inside the library's device
 * code, which every GPU that loads the library holds until the process exits.
 *
 * Limit: the schedule's scratch, kda_prefill_workspace_size() of the same sizes, must fit
 * in 16 MiB (16777216 bytes); larger sizes are refused with KDA_ERR_UNSUPPORTED before
 * anything is enqueued. One long sequence with H heads needs (max(R, m) + m) * H * 64 KiB
 * for its m segments and R segment runs (T = 2^20 with H = 32: 12 MiB); up to 8192 packed
 * sequences need 4 bytes each.
 *
 * Set-up: the first call on a device, with that device current, looks up the array's
 * device address once (it may load the library's device code); make that first call
 * before any stream capture on the device. Later calls only enqueue work.
 *
 * Sharing: every call on a device uses the same array, which keeps the last call's
 * contents; each call writes all the scratch it reads, so nothing needs clearing, but calls
 * that overlap on the GPU (on different streams, or from different threads) race on it:
 * order them on one stream or with events. On an argument error nothing is enqueued.
 *
 * No counterpart in the paper: the method needs no scratch memory at all; this is a
 * deployment variant of the library's own parallel schedule.
 */
kda_status kda_prefill_noalloc(const void *q, const void *k, const void *v, const float *log_alpha,
                               const float *beta, const int32_t *cu_seqlens, int32_t num_seqs,
                               int64_t total_tokens, int32_t H, int32_t d_k, int32_t d_v,
                               kda_dtype in_dtype, kda_dtype out_dtype, float lower_bound,
                               float scale, const float *init_state, void *out,
                               float *final_state, void *stream);

/*
 * kda_prefill_recurrent -- same contract and results as kda_prefill, always on
 * the fp32 token-recurrent kernel (one token at a time, state kept on chip).
 * Exposed for cross-checking the chunked kernels and as the reference-accuracy
 * path for fp32 inputs.
 */
kda_status kda_prefill_recurrent(const void *q, const void *k, const void *v,
                                 const float *log_alpha, const float *beta,
                                 const int32_t *cu_seqlens, int32_t num_seqs,
                                 int64_t total_tokens, int32_t H, int32_t d_k, int32_t d_v,
                                 kda_dtype in_dtype, kda_dtype out_dtype, float lower_bound,
                                 float scale,
                                 const float *init_state, void *out, float *final_state,
                                 void *stream);

/*
 * kda_decode -- one decode step: B independent sequences each take one new
 * token, and their states are updated IN PLACE (Kimi K3 -- Architecture Notes,
 * section 1.1: the fixed-size state replaces a growing KV cache; the update is
 * the same recurrence with T = 1).
 *
 *   q, k        [B, H, d_k]   in_dtype
 *   v           [B, H, d_v]   in_dtype
 *   log_alpha   [B, H, d_k]   fp32
 *   beta        [B, H]        fp32
 *   state       [B, H, d_k, d_v] fp32, read and overwritten with S_t
 *   out         [B, H, d_v]   out_dtype, written with scale * S_t^T q_t
 *
 * Sizes: 1 <= d_k, d_v <= 128 and d_v a multiple of 4; B, H >= 1.
 * No aliasing: state and out must not overlap each other or any input (q, k, v,
 * log_alpha, beta), since every CTA reads its inputs while others write;
 * KDA_ERR_INVALID_ARG otherwise.
 */
kda_status kda_decode(const void *q, const void *k, const void *v, const float *log_alpha,
                      const float *beta, float *state, void *out, int32_t B, int32_t H,
                      int32_t d_k, int32_t d_v, kda_dtype in_dtype, kda_dtype out_dtype,
                      float lower_bound, float scale, void *stream);

/*
 * The gated log-decay (Kimi K3 -- Architecture Notes, section 1.2, the K3 row of
 * the mapping table from decay logits to log-decay): instead of log_alpha, the
 * caller passes the decay logits z and one log-scale A_h per head, and
 *
 *     g_t = g_min * Sigmoid(e^{A_h} z_t),   Sigmoid(x) = 1 / (1 + e^{-x}),
 *
 * is computed inside the kernels. g lies in (g_min, 0) by construction, so no
 * clamp is applied; a NaN logit propagates. z has the element type of q, k, v
 * (so the bf16 path streams 2 bytes per channel instead of the 4 of log_alpha).
 *
 *   z      [total_tokens, H, d_k] (prefill) or [B, H, d_k] (decode)   in_dtype
 *   A_log  [H]   fp32, device; e^{A_h} must be finite in fp32 (A_h < 88)
 *   g_min  the lower end of the log-decay, <= 0 and finite (the pages fix -5)
 *
 * Every other argument, the conventions and the results are those of the
 * clamped entry point with the same suffix. kda_prefill_gated runs the chunked
 * tensor-core kernel when in_dtype is KDA_BF16, d_k = d_v = 128 and
 * g_min >= -5, and the fp32 token-recurrent kernel otherwise;
 * kda_prefill_gated_recurrent always runs the latter.
 */
kda_status kda_prefill_gated(const void *q, const void *k, const void *v, const void *z,
                             const float *A_log, const float *beta, const int32_t *cu_seqlens,
                             int32_t num_seqs, int64_t total_tokens, int32_t H, int32_t d_k,
                             int32_t d_v, kda_dtype in_dtype, kda_dtype out_dtype, float g_min,
                             float scale, const float *init_state, void *out, float *final_state,
                             void *stream);

kda_status kda_prefill_gated_recurrent(const void *q, const void *k, const void *v, const void *z,
                                       const float *A_log, const float *beta,
                                       const int32_t *cu_seqlens, int32_t num_seqs,
                                       int64_t total_tokens, int32_t H, int32_t d_k, int32_t d_v,
                                       kda_dtype in_dtype, kda_dtype out_dtype, float g_min,
                                       float scale, const float *init_state, void *out,
                                       float *final_state, void *stream);

kda_status kda_decode_gated(const void *q, const void *k, const void *v, const void *z,
                            const float *A_log, const float *beta, float *state, void *out,
                            int32_t B, int32_t H, int32_t d_k, int32_t d_v, kda_dtype in_dtype,
                            kda_dtype out_dtype, float g_min, float scale, void *stream);

/*
 * Parameter-block entry points: every option of the calls above in one struct,
 * plus the output gate of Kimi K3 -- Architecture Notes, section 1.3
 * ("Full-rank output gate": y = W_o [Sigmoid(W_g x) (.) RMSNorm(o)]). The two
 * projections W_g and W_o are the caller's matmuls; when `out_gate` is given the
 * library applies the bracket to each read-out before writing it, per token and
 * head over the d_v value channels:
 *
 *     out_t = Sigmoid(r_t) * w * o_t / sqrt(mean_j o_tj^2 + norm_eps),
 *     o_t = scale * S_t^T q_t,   r_t = W_g x_t (the gate logits),
 *
 * with w the RMSNorm weight. The page gives neither eps nor the shape of the
 * weight; this library takes the usual RMSNorm: eps inside the square root and
 * one weight per value channel, shared by the heads. norm_eps = 0 with an
 * all-zero read-out gives NaN (0 / 0), as the formula does.
 *
 * Fields (sizes and layouts as in kda_prefill / kda_decode):
 *   struct_size   sizeof the struct; any other value returns KDA_ERR_INVALID_ARG
 *   decay_form    KDA_DECAY_CLAMPED: `decay` is log_alpha (fp32), A_log must be
 *                 NULL and decay_bound is the lower bound; KDA_DECAY_GATED:
 *                 `decay` is the logits z (in_dtype), A_log [H] and decay_bound
 *                 = g_min as in kda_prefill_gated; KDA_DECAY_UNBOUNDED: the map
 *                 of the earlier models in the same section's table,
 *                 g = -e^{A_h} * Softplus(z), Softplus(x) = log(1 + e^x), from the
 *                 logits z (in_dtype) and A_log [H]; decay_bound is ignored. Its
 *                 decay has no lower bound: a bf16 prefill with d = 128 runs the
 *                 chunked kernel, which forms the diagonal-block entries of channels
 *                 decaying by more than about e^79 over 16 tokens from position
 *                 pairs (Kimi K3 -- Architecture Notes, section 1.2, the Kimi Linear
 *                 treatment of the diagonal tiles); other prefills run the fp32
 *                 token-recurrent kernel
 *   out_gate      gate logits r [rows, H, d_v] in in_dtype, device, 16-byte
 *                 aligned, not overlapping `out`; NULL = no output gate (out = o)
 *   norm_weight   w [d_v] fp32, device; NULL = ones. Must be NULL without out_gate
 *   norm_eps      finite, >= 0 (ignored without out_gate)
 *   force_recurrent (prefill) nonzero runs the fp32 token-recurrent kernel
 *   conv_weight, conv_state, l2_eps (decode) the input prologue of kda_prologue
 *                 applied to the token's raw q, k, v, with the sequence's
 *                 convolution state shifted in place (NULL state = no prologue)
 * The output gate is fused into every kernel (the chunked tensor-core kernel,
 * the token-recurrent kernel and decode); it adds one read of the gate logits
 * and no other memory traffic.
 */
typedef enum { KDA_DECAY_CLAMPED = 0, KDA_DECAY_GATED = 1, KDA_DECAY_UNBOUNDED = 2 } kda_decay_form;

typedef struct kda_prefill_params {
  uint32_t struct_size;
  kda_dtype in_dtype, out_dtype;
  kda_decay_form decay_form;
  int32_t num_seqs, H, d_k, d_v;
  int64_t total_tokens;
  const void *q, *k, *v;
  const void *decay;          /* log_alpha (fp32) or z (in_dtype), [total_tokens, H, d_k] */
  const float *A_log;         /* [H], gated form only                                     */
  const float *beta;          /* [total_tokens, H]                                        */
  const int32_t *cu_seqlens;  /* [num_seqs + 1]                                           */
  const float *init_state;    /* [num_seqs, H, d_k, d_v] or NULL                          */
  const void *out_gate;       /* [total_tokens, H, d_v] or NULL                           */
  const float *norm_weight;   /* [d_v] or NULL                                            */
  void *out;                  /* [total_tokens, H, d_v], out_dtype                        */
  float *final_state;         /* [num_seqs, H, d_k, d_v] or NULL                          */
  float decay_bound;          /* lower_bound (clamped) or g_min (gated)                   */
  float scale;
  float norm_eps;
  int32_t force_recurrent;
  void *workspace;            /* device scratch or NULL, as in kda_prefill            */
  size_t workspace_bytes;
} kda_prefill_params;

typedef struct kda_decode_params {
  uint32_t struct_size;
  kda_dtype in_dtype, out_dtype;
  kda_decay_form decay_form;
  int32_t B, H, d_k, d_v;
  const void *q, *k, *v;
  const void *decay;          /* log_alpha (fp32) or z (in_dtype), [B, H, d_k] */
  const float *A_log;         /* [H], gated form only                          */
  const float *beta;          /* [B, H]                                        */
  float *state;               /* [B, H, d_k, d_v], updated in place            */
  const void *out_gate;       /* [B, H, d_v] or NULL                           */
  const float *norm_weight;   /* [d_v] or NULL                                 */
  void *out;                  /* [B, H, d_v], out_dtype                        */
  const float *conv_weight;   /* prologue: [H, 2 d_k + d_v, 4] fp32, or NULL   */
  void *conv_state;           /* prologue: [B, H, 3, 2 d_k + d_v] in_dtype,
                                 read and shifted in place; NULL = q, k, v are
                                 used as given (no prologue)                   */
  float decay_bound;
  float scale;
  float norm_eps;
  float l2_eps;               /* prologue: eps of the L2 norm, finite, >= 0    */
} kda_decode_params;

kda_status kda_prefill_ex(const kda_prefill_params *params, void *stream);
kda_status kda_decode_ex(const kda_decode_params *params, void *stream);

/*
 * kda_prologue -- the input prologue of a KDA layer over packed sequences (Kimi K3 --
 * Architecture Notes, section 1.1: the q/k/v projections pass a short convolution,
 * then Swish, and q and k are then L2-normalised; kernel size 4 from the visualiser
 * page "Kimi K3"). Per token t, head h and channel c of each projection x:
 *
 *     conv_t = sum_{j=0..3} w[h, c, j] * x_{t-3+j}    (causal, depthwise, no bias)
 *     u_t    = conv_t * Sigmoid(conv_t)                (Swish)
 *     q_t, k_t = u_t / sqrt(sum_c u_tc^2 + l2_eps);    v_t = u_t
 *
 * Inputs before a sequence's first token come from its convolution state (its three
 * previous raw inputs, oldest first), or are zero.
 *
 *   q_raw, k_raw [total_tokens, H, d_k], v_raw [total_tokens, H, d_v]   dtype
 *   conv_weight  [H, 2 d_k + d_v, 4] fp32: the q channels, then k, then v
 *   cu_seqlens   [num_seqs + 1] int32, as in kda_prefill (trusted)
 *   conv_init    [num_seqs, H, 3, 2 d_k + d_v] dtype, or NULL for zeros
 *   q, k, v      outputs, shaped as the raw inputs, dtype (bf16 rounds to nearest-even)
 *   conv_final   [num_seqs, H, 3, 2 d_k + d_v] dtype, written, or NULL: each
 *                sequence's last three raw inputs (shifted in from conv_init when
 *                the sequence is shorter), ready for kda_decode_ex's conv_state
 *
 * Outputs must not overlap the inputs or each other (conv_final may not alias
 * conv_init). Sizes: 1 <= d_k, d_v <= 128, 1 <= H <= 65535. The results are the inputs of
 * kda_prefill / kda_prefill_ex. One HBM-bound pass: reads each raw input once and
 * writes each result once. Enqueues on `stream`.
 */
kda_status kda_prologue(const void *q_raw, const void *k_raw, const void *v_raw,
                        const float *conv_weight, const int32_t *cu_seqlens, int32_t num_seqs,
                        int64_t total_tokens, int32_t H, int32_t d_k, int32_t d_v, kda_dtype dtype,
                        const void *conv_init, float l2_eps, void *q, void *k, void *v,
                        void *conv_final, void *stream);

/*
 * kda_check_device_error -- reads and clears the library's device error word in
 * one atomic exchange, enqueued on `stream` behind the work already there, then
 * synchronises `stream` and returns what the word held: KDA_OK, KDA_ERR_TIMEOUT
 * if a kernel's bounded wait gave up, KDA_ERR_RANGE if a kernel met an input
 * outside its range (KDA_ERR_TIMEOUT wins when both are set), or KDA_ERR_CUDA
 * if a CUDA call failed. There is one word per device, shared by every stream
 * and every call in the process: the check covers the work finished on
 * `stream` and anything that any other stream recorded before the exchange;
 * a code recorded after it is kept for the next check. Concurrent checks from
 * several host threads are serialised by the library.
 */
kda_status kda_check_device_error(void *stream);

/* Human-readable name of a status code (static string, never NULL). */
const char *kda_status_string(kda_status status);

/* Library version as MAJOR*10000 + MINOR*100 + PATCH. */
int32_t kda_version(void);

#ifdef __cplusplus
}
#endif

#endif /* KDA_H */
