/*
 * kda.h -- C ABI of the GB300 gated-delta-rule forward library (libkda.so).
 *
 * The library computes the forward pass of the gated delta rule in its general
 * per-channel form, Kimi Delta Attention (KDA), and its special cases Gated
 * DeltaNet (one decay per head and token) and DeltaNet (no decay, log-decay 0).
 * For each sequence b, value head h and token t of the sequence, with key head
 * kh = h / (num_v_heads / num_k_heads) and S the d_v x d_k state of the
 * derivation ("You Could Have Come Up With Kimi Delta Attention", sec. 4, the
 * boxed KDA update; Modular MAX "gated_delta" module, the five per-token steps):
 *
 *     k^ = k[t,kh] / sqrt(|k[t,kh]|^2 + 1e-6)        (when l2norm_qk != 0)
 *     q^ = scale * q[t,kh] / sqrt(|q[t,kh]|^2 + 1e-6)
 *     S  = S Diag(exp(g[t,h]))                         forget (per key channel)
 *     e  = beta[t,h] (v[t,h] - S k^)                   predict and correct
 *     S  = S + e k^T                                   write
 *     o[t,h] = S q^                                    read, after the write
 *
 * Prefill runs the chunkwise (WY/UT) schedule of the same recurrence ("From
 * Attention to Learned Memory", sec. 4; KDA page sec. 6), which is exact up to
 * rounding; decode runs one token per sequence.
 *
 * Conventions shared by every entry point
 *   - All data pointers are DEVICE pointers; the caller allocates and owns every
 *     buffer (inputs, outputs, state pool, workspace).  The library never
 *     allocates, frees or synchronises on these paths.
 *   - Work is enqueued asynchronously on `stream` (a cudaStream_t, passed as
 *     void*; NULL is the legacy default stream).  Inputs must stay valid until
 *     the stream reaches the enqueued work.
 *   - Layouts are row-major, token-major (ragged batches are concatenated along
 *     the token axis, as in the Modular gated_delta module):
 *         q, k          [T, num_k_heads, d_k]   (row stride settable, see below)
 *         v             [T, num_v_heads, d_v]
 *         beta          [T, num_v_heads]                     fp32
 *         log_decay g   [T, num_v_heads]        (SCALAR)     fp32, g = log alpha <= 0
 *                       [T, num_v_heads, d_k]   (PER_CHANNEL)
 *         state_pool    [num_slots, num_v_heads, d_k, d_v]   (the transpose of the
 *                       derivation's d_v x d_k state: key channel = row)
 *         o             [T, num_v_heads, d_v]                fp32
 *   - q/k/v/beta/g are read only, o is write only; the pool slots named by
 *     slot_idx are read, then overwritten in place with the final state; every
 *     other slot is left untouched.  Slots named twice in one call race.
 *   - Errors: argument problems are found on the host before anything is
 *     enqueued and returned as a status; nothing is launched then.  Problems
 *     only the device can see (offsets not monotone or not ending at
 *     total_tokens, a slot index >= num_slots, repeated slots under
 *     KDA_FLAG_CHECKED; on the tensor-core prefill path, a per-channel
 *     log-decay outside its domain, see KDA_DEVERR_DECAY_RANGE) set a device
 *     error word and the affected work is skipped -- no trap, no fault; read it
 *     with kda_get_device_error().
 */
#ifndef KDA_H_
#define KDA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define KDA_ABI_VERSION 1

typedef enum kda_status {
  KDA_OK = 0,
  KDA_ERR_INVALID_ARG = 1, /* null/misaligned pointer, bad size, bad enum value */
  KDA_ERR_UNSUPPORTED = 2, /* valid but not implemented: head size, chunk, dtype combination */
  KDA_ERR_WORKSPACE = 3,   /* workspace missing or smaller than kda_prefill_workspace_size */
  KDA_ERR_CUDA = 4,        /* a CUDA runtime call or a launch failed */
  KDA_ERR_DEVICE = 5       /* kda_get_device_error: the device flagged bad offsets/slots */
} kda_status_t;

typedef enum kda_dtype { KDA_DTYPE_F32 = 0, KDA_DTYPE_BF16 = 1 } kda_dtype_t;

typedef enum kda_decay_kind {
  KDA_DECAY_SCALAR = 0,     /* Gated DeltaNet: one log-decay per (token, value head) */
  KDA_DECAY_PER_CHANNEL = 1 /* KDA: one log-decay per (token, value head, key channel) */
} kda_decay_kind_t;

/* Check every sequence's offsets and slot and that slots are distinct on the
 * device (without it, offsets and slot ranges are still checked, distinctness is not). */
#define KDA_FLAG_CHECKED 1u
/* Run the prefill on CUDA cores in fp32 even where the tensor-core path applies
 * (bf16 q/k/v, d = 128, chunk 64, whose operands are fp16/bf16 with fp32
 * accumulation).  fp32 q/k/v and the other head sizes and chunks always use it. */
#define KDA_FLAG_CUDA_CORES 2u
/* Tensor-core path only: run it as one kernel per (sequence, value head, value
 * tile) that walks the sequence's chunks, with only the chunk table (16 bytes per
 * chunk) and one flag per sequence and value head as workspace; its per-channel
 * factors are anchored at each chunk's middle token, which bounds the decay it takes
 * (see KDA_DEVERR_DECAY_RANGE).  Without it the path runs as two kernels: a chunk-parallel
 * one that writes every chunk's operands of the state recurrence to the workspace
 * (57,856 bytes per chunk and value head) and a sequential one over each
 * sequence's chunks, which keeps the chunk-local work off the sequential path.
 * The two forms round the same operands the same way; their results agree to
 * the tolerance, not bit for bit.  In kda_prefill_bwd the flag bounds the
 * workspace instead (see there). */
#define KDA_FLAG_COMPACT 4u
/* Additive write in place of the delta rule: the correction subtracts no
 * prediction, e_t = beta_t v_t, so S_t = Diag(alpha_t) S_{t-1} + beta_t k_t v_t^T
 * (stored orientation: row = key channel).  With per-channel decay this is Gated
 * Linear Attention, with scalar decay Mamba-2 (beta_t its write step size) or
 * RetNet (a constant decay), and with zero log-decay and beta = 1 plain causal
 * linear attention ("Linear attention visualized": the naive linear attention,
 * RetNet, Mamba-2 and GLA sections; "From Attention to Learned Memory", sec. 1-2).
 * Accepted by every prefill path, the decode step and the verify window (whose
 * records then hold beta_t v_t); the Gated DeltaProduct entry points, whose method
 * is defined on the delta rule, return KDA_ERR_UNSUPPORTED for it. */
#define KDA_FLAG_NO_DELTA 8u

/* Device error codes (kda_get_device_error). */
#define KDA_DEVERR_NONE 0
#define KDA_DEVERR_OFFSETS 1   /* input_row_offsets not monotone / not 0..total_tokens */
#define KDA_DEVERR_SLOT_RANGE 2 /* slot_idx[b] >= num_slots */
#define KDA_DEVERR_SLOT_DUP 3   /* a slot named twice (KDA_FLAG_CHECKED only) */
#define KDA_DEVERR_TIMEOUT 4    /* a bounded wait inside a kernel gave up; its work is incomplete */
/* KDA_DEVERR_DECAY_RANGE: tensor-core prefill path, per-channel decay outside its domain.
 * The default two-kernel form takes any log-decay g <= 1/64 (a forget gate up to
 * exp(1/64)); a larger g is outside it.  The compact form (KDA_FLAG_COMPACT) also needs
 * every channel's cumulative log-decay to stay within 79 nats of its value at the chunk's
 * middle token.  The (sequence, value head) pairs with such a chunk are skipped: their o rows
 * and their slot's state keep their previous contents, every other pair is computed.  The
 * fp32 CUDA-core path (KDA_FLAG_CUDA_CORES) takes any finite log-decay. */
#define KDA_DEVERR_DECAY_RANGE 5
#define KDA_DEVERR_ACCEPTED 6    /* kda_fold_accepted: accepted[b] > window */

typedef struct kda_params {
  int32_t num_seqs;    /* B: sequences in the ragged batch (prefill) or decode batch */
  int32_t num_k_heads; /* HK: heads of q and k */
  int32_t num_v_heads; /* HV: heads of v, beta, g, o and the state; HV % HK == 0 */
  int32_t d_k;         /* key head size; 16 or 128 */
  int32_t d_v;         /* value head size; must equal d_k */
  int32_t num_slots;   /* slots in state_pool */
  int64_t total_tokens;/* T: rows of the token-major tensors (prefill; ignored by decode) */
  int32_t chunk;       /* prefill chunk length C: 16, 32 or 64 (ignored by decode) */
  int32_t qkv_dtype;   /* kda_dtype_t of q, k, v */
  int32_t state_dtype; /* kda_dtype_t of state_pool (bf16 is rounded to nearest even) */
  int32_t decay_kind;  /* kda_decay_kind_t of log_decay */
  float scale;         /* query scale; <= 0 selects 1/sqrt(d_k) */
  int32_t l2norm_qk;   /* nonzero: L2-normalise q and k rows before use */
  uint32_t flags;      /* KDA_FLAG_* */
  /* Elements between consecutive tokens of q, k, v; 0 means dense
   * (HK*d_k, HK*d_k, HV*d_v).  Lets q, k, v be column blocks of one packed
   * [T, 2*HK*d_k + HV*d_v] buffer.  Must keep rows 16-byte aligned. */
  int64_t q_row_stride;
  int64_t k_row_stride;
  int64_t v_row_stride;
} kda_params_t;

/* Version of this ABI (KDA_ABI_VERSION).  Never fails. */
int kda_abi_version(void);

/* Static, NUL-terminated description of a status code.  Never fails. */
const char *kda_status_string(kda_status_t status);

/*
 * Bytes of device workspace kda_prefill_fwd needs for these parameters
 * (an upper bound that depends only on the params, not on the offsets).
 * Returns KDA_ERR_INVALID_ARG / KDA_ERR_UNSUPPORTED for parameters that
 * kda_prefill_fwd would reject; *bytes is then left unchanged.
 */
kda_status_t kda_prefill_workspace_size(const kda_params_t *p, size_t *bytes);

/*
 * 1 if kda_prefill_fwd would run these parameters on the tensor-core path
 * (bf16 q/k/v, d = 128, chunk 64, KDA_FLAG_CUDA_CORES clear: fp16/bf16 MMA
 * operands with fp32 accumulation), 0 if on the fp32 CUDA-core path, -1 if the
 * parameters are invalid.  Never touches the GPU.
 */
int kda_prefill_uses_tensor_cores(const kda_params_t *p);

/*
 * Chunkwise prefill over a ragged batch ("You Could Have Come Up With Kimi
 * Delta Attention", sec. 6 and the pipeline of sec. 6.6; "From Attention to
 * Learned Memory", sec. 4, WY/UT transform and blocked triangular inverse;
 * Modular "gated_delta" module for the ragged batch, GQA and slot pool).
 *
 *   q, k               [T, HK, d_k], qkv_dtype, rows 16-byte aligned
 *   v                  [T, HV, d_v], qkv_dtype
 *   beta               [T, HV] fp32
 *   log_decay          [T, HV] or [T, HV, d_k] fp32 (decay_kind); 4-byte aligned, and
 *                      16-byte aligned for KDA_DECAY_PER_CHANNEL (its rows are copied in
 *                      16-byte pieces), else KDA_ERR_INVALID_ARG
 *   input_row_offsets  [B+1] uint32: sequence b is tokens [off[b], off[b+1]);
 *                      off[0] = 0, non-decreasing, off[B] = T.  Empty sequences
 *                      are allowed and leave their slot untouched.
 *   slot_idx           [B] uint32, each < num_slots: the pool slot holding
 *                      sequence b's initial state, overwritten with its final state
 *   state_pool         [num_slots, HV, d_k, d_v], state_dtype, in place
 *   o                  [T, HV, d_v] fp32, written for every token
 *   workspace          device scratch of >= kda_prefill_workspace_size bytes,
 *                      256-byte aligned; contents on entry are ignored
 * Returns KDA_OK once the work is enqueued.
 */
kda_status_t kda_prefill_fwd(const kda_params_t *p, const void *q, const void *k, const void *v,
                             const float *beta, const float *log_decay,
                             const uint32_t *input_row_offsets, const uint32_t *slot_idx,
                             void *state_pool, float *o, void *workspace, size_t workspace_bytes,
                             void *stream);

/*
 * The front end before the recurrence ("Pass 1" of the Modular "gated_delta" module, which
 * consumes its output; SiLU features as in "From Attention to Learned Memory", sec. 1; the
 * decay built from a log-rate and a softplus step as in the Mamba-2 section of "Linear
 * attention visualized"): over the packed projection x = [Q | K | V] (conv_dim = 2 HK d_k +
 * HV d_v channels per token) a depthwise causal convolution of `width` (1..4) taps and SiLU,
 *
 *     y[t, c] = SiLU(conv_bias[c] + sum_{i < width} conv_weight[c, i] x[t - width + 1 + i, c]),
 *
 * where the width - 1 inputs before a sequence's first token come from its slot of conv_state
 * (oldest first; zeros when conv_state is NULL), and afterwards the slot holds the sequence's
 * last width - 1 inputs (an empty sequence leaves it alone); plus the gates
 *
 *     beta = sigmoid(b),   log_decay = -exp(A_log[h]) softplus(a + dt_bias).
 *
 *   x, y         [T, conv_dim], qkv_dtype, 16-byte aligned; y's column blocks are q, k, v for
 *                kda_prefill_fwd through q/k/v_row_stride = conv_dim
 *   conv_weight  [conv_dim, width] fp32       conv_bias [conv_dim] fp32 or NULL
 *   a            [T, HV] (SCALAR) or [T, HV, d_k] (PER_CHANNEL) fp32; b [T, HV] fp32
 *   A_log        [HV] fp32 or NULL (rate 1)   dt_bias [HV] or [HV * d_k] fp32 or NULL
 *   input_row_offsets  [B + 1] as kda_prefill_fwd (T = total_tokens), or NULL for the
 *                decode form: one token per sequence, T = num_seqs
 *   slot_idx     [B] (required with conv_state)
 *   conv_state   [num_slots, conv_dim, width - 1], qkv_dtype, or NULL; read and written in place
 *   log_decay    the shape of a, fp32;  beta [T, HV] fp32
 * The row strides in p must be 0 (dense x and y).  Offsets out of order and slots out of
 * range set the device error word; nothing is read or written out of bounds.
 */
kda_status_t kda_conv_gates_fwd(const kda_params_t *p, int32_t width, const void *x,
                                const float *conv_weight, const float *conv_bias, const float *a,
                                const float *b, const float *A_log, const float *dt_bias,
                                const uint32_t *input_row_offsets, const uint32_t *slot_idx,
                                void *conv_state, void *y, float *log_decay, float *beta,
                                void *stream);

/*
 * Backward pass of kda_prefill_fwd: the gradients of a loss w.r.t. every input,
 * given its gradients w.r.t. the outputs o and the final states.  The chunk form
 * of the forward ("You Could Have Come Up With Kimi Delta Attention", sec. 6) is
 * differentiated by the chain rule: the state gradient runs as a reverse scan
 * over each sequence's chunks (the transpose of the forward's state recursion),
 * the rest chunk-parallel; the L2 normalisation of q and k and the query scale
 * are differentiated too ("From Attention to Learned Memory", sec. 3, gives the
 * linear-attention backward in full; the delta rule's follows the same recurrence).
 * fp32 arithmetic throughout; with bf16 q/k/v at d = 128 and chunk 64 the scan's
 * two directions and the contractions over the value dimension run on tensor
 * cores with tf32 operands (10-bit mantissa, fp32 range) and fp32 accumulation,
 * everything else on CUDA cores.
 *
 *   q, k, v, beta, log_decay, input_row_offsets, slot_idx: as kda_prefill_fwd
 *   state_pool  [num_slots, HV, d_k, d_v], state_dtype, read only: the INITIAL
 *               states (the pool as it was before the forward call)
 *   d_o         [T, HV, d_v] fp32: dLoss/do
 *   d_state     [num_slots, HV, d_k, d_v] fp32 or NULL (zero): dLoss/d(final
 *               state) of the touched slots
 *   dq, dk      [T, HK, d_k] fp32 (summed over the value heads of each key head)
 *   dv          [T, HV, d_v] fp32          dbeta [T, HV] fp32
 *   dlog_decay  the shape of log_decay, fp32
 *   d_state0    [num_slots, HV, d_k, d_v] fp32 or NULL: dLoss/d(initial state),
 *               written at the touched slots only; may alias d_state
 *   workspace   >= kda_prefill_bwd_workspace_size bytes, 256-byte aligned
 * q, k, v 16-byte aligned with 16-byte aligned rows (as for the forward), every
 * other array 4-byte aligned.  KDA_FLAG_NO_DELTA differentiates the additive
 * write; KDA_FLAG_CUDA_CORES is ignored.  Device-side checks (offsets, slots) set
 * the error word and skip the work, as in the forward.
 *
 * Workspace.  By default it holds every chunk's per-(chunk, value head) matrices,
 * about 0.6 MB per chunk and value head (9.3 GB for 2 x 16384 tokens, 32 heads).
 * KDA_FLAG_COMPACT (bf16 q/k/v, d = 128, chunk 64; ignored elsewhere) bounds it:
 * the chunks run in windows of wc chunk positions per sequence,
 * wc = max(1, 512 / (num_seqs * HV)), so the per-chunk matrices exist for
 * max(512, num_seqs * HV) (chunk, value head) slots, plus the state entering
 * every window after a sequence's first (64 KB per window and value head at
 * d = 128) and one state gradient per (sequence, value head): 421 MiB for
 * 2 x 16384 tokens, 32 heads.  A forward sweep over the windows stores those
 * entering states; the backward sweep then reruns each window's chunk-local stage
 * and forward scan from its checkpoint, latest window first, with the same
 * arithmetic per chunk, so the gradients equal the default form's bit for bit.
 * The call reads the longest sequence's chunk count back to the host once (a
 * synchronisation of `stream`) to size the sweeps.
 */
kda_status_t kda_prefill_bwd_workspace_size(const kda_params_t *p, size_t *bytes);
kda_status_t kda_prefill_bwd(const kda_params_t *p, const void *q, const void *k, const void *v,
                             const float *beta, const float *log_decay,
                             const uint32_t *input_row_offsets, const uint32_t *slot_idx,
                             const void *state_pool, const float *d_o, const float *d_state,
                             float *dq, float *dk, float *dv, float *dbeta, float *dlog_decay,
                             float *d_state0, void *workspace, size_t workspace_bytes,
                             void *stream);

/*
 * One recurrent decode step: one token for each of B = num_seqs sequences
 * ("You Could Have Come Up With Kimi Delta Attention", sec. 5, fused recurrent
 * kernel; Modular "gated_delta" module, the five per-token steps).
 *
 *   q, k        [B, HK, d_k], qkv_dtype     v  [B, HV, d_v], qkv_dtype
 *   beta        [B, HV] fp32                log_decay [B, HV] or [B, HV, d_k] fp32
 *   slot_idx    [B] uint32, each < num_slots
 *   state_pool  [num_slots, HV, d_k, d_v], state_dtype, updated in place
 *   o           [B, HV, d_v] fp32
 * total_tokens and chunk are ignored.  Needs no workspace.
 */
kda_status_t kda_decode_step(const kda_params_t *p, const void *q, const void *k, const void *v,
                             const float *beta, const float *log_decay, const uint32_t *slot_idx,
                             void *state_pool, float *o, void *stream);

/*
 * Speculative-decode verification (Modular MAX "gated_delta" module: the verify
 * kernel runs the recurrence over a verify window and records a ring instead of
 * writing the state back; the fold applies a verify's accepted records to the
 * pool).  The module does not spell out a record; here one record is what a
 * token's state update needs, so that folding it replays that update exactly:
 *
 *     record = [ k^ (d_k) | e (d_v) | alpha (d_k; for SCALAR decay one value
 *                followed by 3 padding elements) ]   fp32
 *     fold:    S <- S Diag(alpha) + e k^T     (the forget and write steps)
 *
 * kda_ring_record_elems returns the record length in fp32 elements
 * (2 d_k + d_v, or d_k + d_v + 4), or -1 for invalid parameters.
 */
int kda_ring_record_elems(const kda_params_t *p);

/*
 * Runs `window` tokens of each of B = num_seqs sequences from its pool slot
 * without modifying the pool: writes every token's output and ring record.
 *   q, k        [B*window, HK, d_k]  (token t of sequence b is row b*window + t)
 *   v           [B*window, HV, d_v]     beta [B*window, HV] fp32
 *   log_decay   [B*window, HV] or [B*window, HV, d_k] fp32
 *   slot_idx    [B] uint32              state_pool read only
 *   o           [B*window, HV, d_v] fp32
 *   ring        [B, window, HV, kda_ring_record_elems] fp32, 16-byte aligned
 * window must be 1..64.  total_tokens and chunk are ignored.
 */
kda_status_t kda_verify_window(const kda_params_t *p, const void *q, const void *k, const void *v,
                               const float *beta, const float *log_decay, const uint32_t *slot_idx,
                               int32_t window, const void *state_pool, float *o, float *ring,
                               void *stream);

/*
 * Applies the first accepted[b] records of sequence b's verify window to its
 * pool slot, in token order (accepted[b] = 0 leaves the slot unchanged).  The
 * result equals accepted[b] decode steps of those tokens from the same state.
 *   ring       as written by kda_verify_window with the same p and window
 *   accepted   [B] uint32, each <= window (larger values set KDA_DEVERR_ACCEPTED
 *              on the device and leave that slot unchanged)
 *   slot_idx   [B] uint32; state_pool updated in place
 */
kda_status_t kda_fold_accepted(const kda_params_t *p, const float *ring, int32_t window,
                               const uint32_t *accepted, const uint32_t *slot_idx,
                               void *state_pool, void *stream);

/*
 * Gated DeltaProduct ("Linear attention visualized", Gated Delta Product section and
 * its virtual-sequence table).  Every token carries n_h transitions, each with its own
 * key, value and gate; the state decays once (by the token's log_decay) before the
 * first, the n_h predict / correct / write steps follow in order, and the token's query
 * reads the state after the last.  n_h = 1 is kda_prefill_fwd.  Computed as the gated
 * delta rule over the virtual sequence of T * n_h positions (decay on the first
 * substep, query on the last, every n_h-th output kept) on the same prefill path.
 *
 *   n_h                1..64 substeps per token
 *   q                  [T, HK, d_k], one query per token (q_row_stride between tokens)
 *   k                  [T, n_h, HK, d_k] (k_row_stride between substep rows)
 *   v                  [T, n_h, HV, d_v] (v_row_stride between substep rows)
 *   beta               [T, n_h, HV] fp32
 *   log_decay          [T, HV] or [T, HV, d_k] fp32, one per token
 *   input_row_offsets, slot_idx, state_pool: as kda_prefill_fwd, over tokens
 *   o                  [T, HV, d_v] fp32, one output per token
 *   workspace          >= kda_gdp_workspace_size(p, n_h, 0) bytes, 256-byte aligned
 * The workspace also holds the virtual queries, log-decays and outputs
 * (T * n_h * (HK*d_k*qkv size + HV*gate width*4 + HV*d_v*4) bytes) ahead of the
 * prefill's own workspace.  Errors as kda_prefill_fwd; n_h outside 1..64 is
 * KDA_ERR_INVALID_ARG, T * n_h >= 2^31 is KDA_ERR_UNSUPPORTED.
 */
kda_status_t kda_gdp_prefill_fwd(const kda_params_t *p, int32_t n_h, const void *q,
                                 const void *k, const void *v, const float *beta,
                                 const float *log_decay, const uint32_t *input_row_offsets,
                                 const uint32_t *slot_idx, void *state_pool, float *o,
                                 void *workspace, size_t workspace_bytes, void *stream);

/*
 * One Gated DeltaProduct decode step: one token (n_h transitions) for each of
 * B = num_seqs sequences, read from and written back to slot_idx[b] of the pool.
 * Arrays as kda_gdp_prefill_fwd with T = B and no offsets; total_tokens is ignored,
 * chunk 0 means 64.  Workspace: kda_gdp_workspace_size(p, n_h, 1) bytes.
 */
kda_status_t kda_gdp_decode_step(const kda_params_t *p, int32_t n_h, const void *q,
                                 const void *k, const void *v, const float *beta,
                                 const float *log_decay, const uint32_t *slot_idx,
                                 void *state_pool, float *o, void *workspace,
                                 size_t workspace_bytes, void *stream);

/*
 * Workspace bytes of kda_gdp_prefill_fwd (decode = 0) or kda_gdp_decode_step
 * (decode = 1) for these parameters and n_h.  Returns the status the call would
 * return for invalid parameters; *bytes is then left unchanged.
 */
kda_status_t kda_gdp_workspace_size(const kda_params_t *p, int32_t n_h, int32_t decode,
                                    size_t *bytes);

/*
 * Waits for `stream`, then returns the device error word of the current device
 * in *code (KDA_DEVERR_*) and clears it.  Returns KDA_ERR_DEVICE when the word
 * was set, KDA_OK when it was clear, KDA_ERR_CUDA when a CUDA call failed.
 */
kda_status_t kda_get_device_error(void *stream, int32_t *code);

/*
 * Prefill without any device allocation: same inputs, outputs and results as
 * kda_prefill_fwd, but its scratch lives in a fixed array inside the library
 * instead of a caller-provided workspace.  There is no counterpart on the pages.
 *
 * For callers that cannot allocate device memory at the point where they run
 * the prefill: code hosted inside an engine that owns the device's memory
 * budget and hands out no allocator, or a runtime that reserves all of its
 * memory at start-up.  They still pass every input and output buffer.
 *
 *   - The scratch is KDA_NO_ALLOC_SCRATCH_BYTES (64 MiB) of device memory that
 *     every GPU which loads the library holds until the process exits.
 *     Problems whose workspace exceeds it are rejected with KDA_ERR_WORKSPACE
 *     before anything is enqueued.
 *   - The default two-kernel tensor-core form needs the chunk table and 57,856
 *     bytes of chunk records per chunk and value head: about 1,150 chunk-heads
 *     (some 4,600 tokens x 16 value heads at chunk 64) fit.  Larger problems run
 *     the compact single-kernel form instead (as with KDA_FLAG_COMPACT: the chunk
 *     table and a flag per sequence and value head, which fits any practical
 *     batch), which is slower and takes a narrower per-channel decay range (see
 *     KDA_DEVERR_DECAY_RANGE); kda_prefill_no_alloc_form() says which form a call
 *     with these parameters runs.  The fp32 CUDA-core path needs about 150 KB per
 *     chunk and value head (roughly 1,700 tokens x 16 heads at d = 128, chunk 64).
 *   - The first call on each device looks up the array's device address
 *     (cudaGetSymbolAddress, with that device current); make that first call
 *     before any stream capture.  Later calls allocate nothing and enqueue
 *     nothing on the stream but the kernel launches.
 *   - All calls share the one array and it keeps the last call's contents
 *     (nothing in it needs to start at zero).  Calls whose work overlaps on the
 *     GPU -- different streams, or different host threads -- race on it: order
 *     them on one stream.
 * Arguments, layouts, errors and the device error word are as in
 * kda_prefill_fwd.  This entry point calls no cudaMalloc / cudaFree.
 */
#define KDA_NO_ALLOC_SCRATCH_BYTES (64u << 20)
kda_status_t kda_prefill_fwd_no_alloc(const kda_params_t *p, const void *q, const void *k,
                                      const void *v, const float *beta, const float *log_decay,
                                      const uint32_t *input_row_offsets, const uint32_t *slot_idx,
                                      void *state_pool, float *o, void *stream);

/*
 * Which form kda_prefill_fwd_no_alloc runs for these parameters (no counterpart on
 * the pages): 0 the two-kernel tensor-core form, 1 the compact single-kernel
 * tensor-core form (the chunk records do not fit the scratch, or KDA_FLAG_COMPACT is
 * set), 2 the fp32 CUDA-core path, -1 rejected (invalid parameters, or a workspace
 * larger than KDA_NO_ALLOC_SCRATCH_BYTES).  Never touches the GPU.
 */
int kda_prefill_no_alloc_form(const kda_params_t *p);

/*
 * Measurement aid (no counterpart on the pages).  Registers up to 8 CUDA events
 * (cudaEvent_t handles passed as void*, created by the caller) that later
 * kda_prefill_fwd / kda_decode_step calls on this process record on their
 * stream: events[0] before the first kernel, events[i] after the i-th kernel.
 * Lets a benchmark time each kernel with CUDA events on the stream the kernel
 * runs on.  count = 0 (or events = NULL) clears the registration.  The handles
 * must stay valid while registered; calls from several threads share it.
 * Returns KDA_ERR_INVALID_ARG for count < 0 or > 8.
 */
kda_status_t kda_set_stage_events(void *const *events, int32_t count);

#ifdef __cplusplus
}
#endif

#endif /* KDA_H_ */
