/*
 * gdn.h -- C ABI of libgdn: the gated delta-rule recurrent state scan
 * (Gated DeltaNet linear attention) on one NVIDIA GB300 (sm_103a).
 *
 * The operation (onnx-runtime-ep-cuda 0.1.0-dev.6, src/kernels/linear_attention.rs,
 * `linear_attention_core`, Steps 1-4, and its fused gate chain): for every
 * sequence n and value head h there is a state S[d_k][d_v] in fp32.  For each
 * token t of the sequence, in order,
 *     g_t    = -exp(A_log[h]) * softplus(a[t,h] + dt_bias[h])      (log-space decay)
 *     beta_t = sigmoid(b[t,h])
 *     S      = exp(g_t) * S                                        (Step 1, decay)
 *     r      = S^T k_t                                             (Step 2, retrieval)
 *     S      = S + k_t (x) beta_t (v_t - r)                        (Step 3, delta update)
 *     o_t    = scale * S^T q_t      (with the updated S)           (Step 4, readout)
 * Value head h reads query/key head h / (h_v / h_qk): consecutive value heads
 * share one q/k head (the GQA mapping of the same page and of nuvec-core 0.6.1,
 * src/fast/imp.rs, `gated_delta_graph`).
 *
 * Conventions for every call below:
 *  - All tensor pointers are DEVICE pointers to contiguous row-major arrays,
 *    owned by the caller; the library never allocates, frees or keeps them.
 *  - Layouts (T = tokens per sequence, or the packed total for varlen):
 *        q, k   [B, T, h_qk, d_k]   io dtype
 *        v, o   [B, T, h_v,  d_v]   io dtype
 *        a, b   [B, T, h_v]         io dtype (raw gate logits)
 *        A_log, dt_bias [h_v]       fp32
 *        state  [N, h_v, d_k, d_v]  fp32 (N = number of sequences)
 *  - `stream` is a cudaStream_t passed as void* (NULL = the legacy default
 *    stream).  Calls are asynchronous on that stream; nothing synchronises.
 *  - Errors found on the host return a status and launch nothing.  Errors only
 *    the device can see (a malformed device cu_seqlens, a slot outside a state
 *    pool) set a device check word, skip the affected work without faulting, and
 *    are reported by gdn_last_device_status().
 *  - Internal resources: gdn_prefill may create, once per device, a CUDA stream and
 *    two events (see gdn_prefill_workspace_bytes); gdn_prefill_noalloc and every
 *    other call create nothing.  No call allocates device memory or uses a library
 *    kernel.
 *
 * Entry points: gdn_prefill (and gdn_prefill_noalloc, gdn_prefill_plan,
 * gdn_prefill_workspace_bytes), gdn_decode_step, gdn_decode_step_slots (a state
 * pool), gdn_scan_window (the states after each of the last W steps),
 * gdn_scan_variant and gdn_prefill_variant (other update rules and gate layouts; with
 * gdn_prefill_variant_workspace_bytes and gdn_prefill_variant_plan),
 * the layer ops around the scan: gdn_causal_conv, gdn_causal_conv_slots and
 * gdn_gated_rmsnorm, gdn_prefill_norm (the prefill and the norm in one call),
 * gdn_decode_layer (conv -> decode step -> norm in one kernel) and gdn_prefill_layer
 * (conv -> prefill -> norm, the convolution inside the chunk prep; with
 * gdn_prefill_layer_workspace_bytes).
 *  - gdn_last_error_message() gives a human-readable detail of the last
 *    non-OK status returned on the calling thread.
 */
#ifndef GDN_H
#define GDN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    GDN_OK = 0,
    GDN_ERR_INVALID_ARG = 1,   /* bad shape, null or misaligned pointer, bad size  */
    GDN_ERR_UNSUPPORTED = 2,   /* valid arguments, geometry not built (d_k > 256)   */
    GDN_ERR_CUDA = 3,          /* a CUDA runtime call or launch failed              */
    GDN_ERR_DEVICE_CHECK = 4,  /* the device found malformed cu_seqlens or a slot
                                  outside the pool                                  */
    GDN_ERR_TIMEOUT = 5        /* a bounded device-side wait gave up                */
} gdn_status;

typedef enum { GDN_F32 = 0, GDN_BF16 = 1, GDN_F16 = 2 } gdn_dtype;

/* The update rules of the onnx-runtime-ep-cuda page's rule list (UpdateRule). */
typedef enum {
    GDN_RULE_GATED_DELTA = 0,   /* decay, retrieval, delta update, readout (the default) */
    GDN_RULE_DELTA = 1,         /* no decay: S += k (x) beta (v - S^T k)                  */
    GDN_RULE_GATED = 2,         /* decay, then S += k (x) v                              */
    GDN_RULE_LINEAR = 3         /* S += k (x) v                                           */
} gdn_rule;

/* Gate and rule variant of gdn_scan_variant (all zero: gdn_prefill's gates). */
typedef struct gdn_variant {
    int32_t rule;            /* gdn_rule                                                   */
    int32_t decay_per_key;   /* 0: a [.., h_v], A_log and dt_bias [h_v];
                                1: a [.., h_v, d_k], A_log and dt_bias [h_v, d_k] (fp32):
                                   row i of S decays by exp(-exp(A_log[h,i]) *
                                   softplus(a[..,h,i] + dt_bias[h,i]))                    */
    int32_t beta_shared;     /* 0: b [.., h_v]; 1: b [B, T, 1], one beta for every head  */
} gdn_variant;

/* Problem geometry shared by every entry point. */
typedef struct gdn_shape {
    int32_t io_dtype;   /* gdn_dtype of q, k, v, a, b and o                          */
    int32_t batch;      /* B; must be 1 when cu_seqlens is given                       */
    int64_t seqlen;     /* T per sequence, or the packed token total with cu_seqlens   */
    int32_t num_seqs;   /* N: equals batch, or len(cu_seqlens) - 1 with cu_seqlens     */
    int32_t h_qk;       /* query/key heads; h_v % h_qk == 0                            */
    int32_t h_v;        /* value heads (one state per value head)                      */
    int32_t d_k;        /* key dim, 1..256 (the tensor-core prefill needs 128)         */
    int32_t d_v;        /* value dim, 1..256, a multiple of 4                          */
} gdn_shape;

/*
 * gdn_prefill -- run the recurrence over whole sequences.
 *
 *   q, k, v, a, b  inputs in the layouts above.
 *   A_log, dt_bias per-value-head gate parameters (fp32 [h_v]).
 *   state_in       initial states [N, h_v, d_k, d_v] fp32, or NULL for zeros.
 *   cu_seqlens     NULL for B sequences of length shape->seqlen; else a DEVICE
 *                  int32 array [N+1] of token offsets into the packed axis
 *                  (cu[0] = 0, non-decreasing, cu[N] = shape->seqlen).  A
 *                  sequence whose entries break these rules is skipped and the
 *                  device check word is set.  Empty sequences are allowed.
 *   scale          readout scale; 0 means 1/sqrt(d_k).
 *   o              output [B, T, h_v, d_v] io dtype, written for every token.
 *   state_out      final states [N, h_v, d_k, d_v] fp32; may alias state_in.
 *                  A sequence with no tokens gets state_in (zeros if NULL),
 *                  as the onnxruntime-ep-mlx ssm.rs page does for an empty
 *                  time axis.
 *   workspace      device scratch of at least gdn_prefill_workspace_bytes(shape)
 *                  bytes (may be NULL when that is 0); its contents need no
 *                  initialisation and are not preserved.
 *
 * bf16/f16 I/O with d_k = d_v = 128 runs the chunked tensor-core path (q, k, v
 * and o must then be 16-byte aligned, else the SIMT path runs); other shapes and
 * fp32 I/O run the token-sequential SIMT path.  State math is fp32 always.
 *
 * On the tensor-core path a batched call whose scan uses few SMs is cut along the
 * time axis into segments that are scanned at once (each from a zero state and, for
 * the correction, from the identity with the values zeroed), then combined; a last
 * kernel adds the correction o += R S_k of each later segment on the tensor cores,
 * with S_k taken in fp32.  That needs the full gdn_prefill_workspace_bytes(shape); a
 * workspace that holds only the chunk records (65 KiB per chunk and value head)
 * instead splits the call into chunk segments whose preparation runs on a stream
 * internal to the library (one per device, created on first use) beside the scan of
 * the earlier one.  Either way the work is ordered after what `stream` held at the
 * call and the call's last kernel is ordered after it, so the call keeps the
 * stream-ordered semantics above.
 */
size_t gdn_prefill_workspace_bytes(const gdn_shape *shape);

gdn_status gdn_prefill(const gdn_shape *shape, const void *q, const void *k, const void *v,
                       const void *a, const void *b, const float *A_log, const float *dt_bias,
                       const float *state_in, const int32_t *cu_seqlens, float scale, void *o,
                       float *state_out, void *workspace, size_t workspace_bytes, void *stream);

/*
 * gdn_prefill_noalloc -- gdn_prefill without a caller-provided workspace.  The
 * pages have no counterpart to this entry point; it exists for callers that may
 * not allocate device memory: a plugin inside a host engine that owns the whole
 * device-memory budget and hands out no allocator, or a latency-bound caller
 * that cannot accept cudaMalloc's implicit device synchronisation.
 *
 * Arguments, layouts, results and errors are those of gdn_prefill, minus
 * `workspace` and `workspace_bytes`.  The scratch is instead a fixed array of
 * GDN_PREFILL_NOALLOC_SCRATCH_BYTES (96 MiB) inside the library, one per device,
 * created when the library's module is first used on that device; the call
 * allocates nothing and frees nothing.  It runs the records-only path (no
 * time-parallel scan, no internal stream), so it needs the chunk records alone: a
 * shape needing more than that size returns GDN_ERR_INVALID_ARG and launches
 * nothing.  A record covers one (64-token chunk, value head) and takes 66,560 bytes, so
 * 96 MiB holds 1,512 records.  The count is read the way the call itself runs: a batched
 * call (cu_seqlens NULL) needs batch * ceil(seqlen / 64) * h_v records, a packed call
 * (cu_seqlens given) (floor(seqlen / 64) + num_seqs + 1) * h_v.  One batched sequence of
 * up to 6,016 tokens at 16 value heads fits (94 x 16 = 1,504 records); 6,017 does not.
 * Shapes off the tensor-core path need no scratch and run as in gdn_prefill.
 *
 * All calls on a device share the one array.  Each call writes every scratch
 * byte it reads before reading it, so no clearing is needed between calls, but
 * two calls whose kernels overlap on the GPU (different streams, no ordering
 * between them) race on the array and give wrong results: order such calls on
 * one stream or with events.
 */
#define GDN_PREFILL_NOALLOC_SCRATCH_BYTES (96u * 1024u * 1024u)

gdn_status gdn_prefill_noalloc(const gdn_shape *shape, const void *q, const void *k,
                               const void *v, const void *a, const void *b, const float *A_log,
                               const float *dt_bias, const float *state_in,
                               const int32_t *cu_seqlens, float scale, void *o,
                               float *state_out, void *stream);

/*
 * gdn_decode_step -- one token per sequence (shape->seqlen must be 1 and
 * cu_seqlens is not taken): B = shape->batch = shape->num_seqs.  `state`
 * [B, h_v, d_k, d_v] fp32 is read and overwritten in place with the updated
 * state.  o [B, 1, h_v, d_v] receives the readout.  Same gates and scale as
 * gdn_prefill; the result equals gdn_prefill on T = 1.
 */
gdn_status gdn_decode_step(const gdn_shape *shape, const void *q, const void *k, const void *v,
                           const void *a, const void *b, const float *A_log,
                           const float *dt_bias, float *state, float scale, void *o,
                           void *stream);

/*
 * gdn_decode_step_slots -- gdn_decode_step against a pool of states, for continuous
 * batching: sequence b (b < B = shape->batch = shape->num_seqs) reads and updates
 * pool entry slots[b] in place.  Follows the `gated_delta_slots` op of the nuvec-core
 * page (src/fast/imp.rs, the fallback graph of FastOp::GatedDeltaSlots): the states at
 * the slots are taken, the rule runs, and the new states are put back at the slots.
 *
 *   pool        DEVICE fp32 [pool_size, h_v, d_k, d_v], 16-byte aligned; entries not
 *               named by `slots` are neither read nor written.
 *   pool_size   number of pool entries (> 0).
 *   slots       DEVICE int32 [B].  The rows should name distinct entries: with a
 *               repeated entry, which row's state lands there, and what those rows
 *               read, is unspecified.  A slot outside [0, pool_size) skips its row
 *               (its o row is left as it was, no pool entry changes) and sets the
 *               device check word, reported by gdn_last_device_status() as
 *               GDN_ERR_DEVICE_CHECK.
 *   q .. o, scale   as gdn_decode_step.
 */
gdn_status gdn_decode_step_slots(const gdn_shape *shape, const void *q, const void *k,
                                 const void *v, const void *a, const void *b, const float *A_log,
                                 const float *dt_bias, float *pool, int64_t pool_size,
                                 const int32_t *slots, float scale, void *o, void *stream);

/*
 * gdn_scan_window -- run B sequences of T tokens each (shape->batch = num_seqs = B,
 * shape->seqlen = T, no cu_seqlens) and emit, instead of the final state, the states
 * after each of the last `window_len` steps: window[w] for w < window_len is the state
 * after step T - window_len + w; when T < window_len the first window_len - T slabs are
 * zero (the `state_window` output of the onnxruntime-ep-mlx ssm.rs page,
 * LinearAttention; with window_len = T this is every step's state, the
 * `gated_delta_steps` output of the nuvec-core page).  Meant for speculative decoding:
 * run the T draft tokens, then restore the state after the last accepted one.
 *
 *   window      DEVICE fp32 [window_len, B, h_v, d_k, d_v], 16-byte aligned, written
 *               in full.
 *   window_len  >= 1.
 *   the rest    as gdn_prefill (state_in may be NULL for zeros).
 * Runs the token-sequential path for every shape and I/O type.
 */
gdn_status gdn_scan_window(const gdn_shape *shape, const void *q, const void *k, const void *v,
                           const void *a, const void *b, const float *A_log, const float *dt_bias,
                           const float *state_in, float scale, void *o, float *window,
                           int32_t window_len, void *stream);

/*
 * gdn_prefill_variant -- gdn_prefill with a gate / rule variant (see gdn_scan_variant for
 * the variants and how they shape a, b, A_log and dt_bias), taking the path gdn_prefill
 * takes: for 16-bit I/O at d_k = d_v = 128 the chunked tensor-core prefill, on which the
 * four update rules and the shared beta are switches of the same algebra (no decay:
 * g = 0; no delta term: A = 0, beta = 1 and W = 0, so the chunk update adds K^T V).
 * A per-key-dim decay (Step 1 scaling row i of the state by e^{g_i}) runs there too, with
 * the gates inside the operands: the chunk's A and P entries are sums over the key
 * dimension of k_t k_s e^{G_t - G_s} (G the running decay sum per dimension), formed on
 * the FP32 cores, and Q and K reach the state scan scaled by e^G and e^{G_C - G}.  That
 * needs the larger workspace gdn_prefill_variant_workspace_bytes reports (two arrays of
 * tokens x h_v x 128 16-bit values more) and `a` 16-byte aligned; with only
 * gdn_prefill_workspace_bytes, an `a` off 16 bytes, or off the tensor-core shapes, a
 * per-key decay runs the token-sequential path.  workspace and
 * workspace_bytes are otherwise gdn_prefill's.  Errors are gdn_scan_variant's plus
 * gdn_prefill's workspace rule.
 */
gdn_status gdn_prefill_variant(const gdn_shape *shape, const gdn_variant *variant, const void *q,
                               const void *k, const void *v, const void *a, const void *b,
                               const float *A_log, const float *dt_bias, const float *state_in,
                               const int32_t *cu_seqlens, float scale, void *o, float *state_out,
                               void *workspace, size_t workspace_bytes, void *stream);

/*
 * gdn_prefill_variant_workspace_bytes -- the workspace gdn_prefill_variant needs for
 * `shape` and `variant` to take its fastest path: gdn_prefill_workspace_bytes(shape), plus,
 * for a per-key-dim decay with a decaying rule, 2 x seqlen x batch x h_v x 128 x 2 bytes
 * (rounded up to 1 KiB each) for the scaled Q and K.  0 when the shape is off the
 * tensor-core path; never fails (a NULL variant reads as the default one).
 */
size_t gdn_prefill_variant_workspace_bytes(const gdn_shape *shape, const gdn_variant *variant);

/*
 * gdn_prefill_variant_plan -- gdn_prefill_plan for gdn_prefill_variant with a workspace of
 * gdn_prefill_variant_workspace_bytes: every rule, the shared beta and the per-key-dim
 * decay take the same kernel path and launch count as the default rule.  Errors:
 * GDN_ERR_INVALID_ARG for a NULL variant or an unknown rule, else gdn_prefill_plan's.
 */
gdn_status gdn_prefill_variant_plan(const gdn_shape *shape, const gdn_variant *variant, int32_t *path,
                                    int32_t *launches);

/*
 * gdn_scan_variant -- gdn_prefill with the gate and rule variants of the
 * onnx-runtime-ep-cuda page's LinearAttention: the update rules {gated_delta,
 * delta, gated, linear} (UpdateRule), Step 1's per-key-dim decay
 * (`decay_per_key_dim`) and a beta shared by all heads (`beta_per_head` false).
 * Arguments and layouts are gdn_prefill's, with a, A_log and dt_bias shaped by
 * variant->decay_per_key and b by variant->beta_shared.  Rules without decay do
 * not read a, A_log or dt_bias (which may be NULL); rules without the delta term do
 * not read b (which may be NULL).  Runs the token-sequential path for every shape
 * and I/O type, including T = 1 with state_out aliasing state_in (a decode step).
 */
gdn_status gdn_scan_variant(const gdn_shape *shape, const gdn_variant *variant, const void *q,
                            const void *k, const void *v, const void *a, const void *b,
                            const float *A_log, const float *dt_bias, const float *state_in,
                            const int32_t *cu_seqlens, float scale, void *o, float *state_out,
                            void *stream);

/* ------------------------------------------------------------------------------------
 * The layer ops around the scan (onnxruntime-ep-mlx 0.31.1, src/ops/ssm.rs): the causal
 * depthwise convolution that produces q, k, v, and the gated RMS norm of the output.
 * ---------------------------------------------------------------------------------- */

/* Activations: the convolution takes NONE or SILU, the norm SILU or SIGMOID. */
typedef enum { GDN_ACT_NONE = 0, GDN_ACT_SILU = 1, GDN_ACT_SIGMOID = 2 } gdn_activation;

/* Geometry of a causal depthwise convolution; carry = (kernel - 1) * dilation. */
typedef struct gdn_conv_shape {
    int32_t io_dtype;        /* gdn_dtype of x, weight, bias, state and y alike           */
    int32_t batch;           /* B rows                                                      */
    int64_t seqlen;          /* L tokens per row (0 allowed)                                */
    int32_t channels;        /* C                                                           */
    int32_t kernel;          /* K taps, 1..64                                               */
    int32_t dilation;        /* >= 1, with carry <= 4096                                    */
    int32_t channels_last;   /* 1: x, y [B, L, C], state [B, carry, C];
                                0: x, y [B, C, L], state [B, C, carry]                      */
    int32_t activation;      /* GDN_ACT_NONE or GDN_ACT_SILU                                */
    int32_t state_window;    /* 0, or W in 1..8: state_in and state_out gain a leading [W]
                                axis (the states after each of the last W tokens)          */
} gdn_conv_shape;

/*
 * gdn_causal_conv -- CausalConvWithState (ssm.rs `causal_conv_op`).  Every channel c of
 * row b is convolved on its own over the padded sequence pad = [past state ; x]:
 *   y[b, t, c] = act(bias[c] + sum_{j<K} weight[c, j] * pad[t + j * dilation])
 * (taps in order, no flip), computed in fp32 and rounded once to the I/O dtype.
 *   weight   [C, 1, K] (the same memory as [C, K, 1]); bias [C] or NULL.
 *   state_in the past state (NULL = zeros); with state_window W only slab W - 1 is read.
 *   state_out the present state (NULL = not written): pad[L .. L + carry), an exact copy;
 *            with a window, slab s holds the carry positions ending at token L - W + s,
 *            zero slabs first when L < W, and the past window itself when L = 0.
 * state_out may be state_in itself (the update is then in place); other overlaps, or y
 * overlapping an input, give undefined results.  All pointers are device memory owned by
 * the caller and aligned to the I/O element size.  Bad geometry or pointers return
 * GDN_ERR_INVALID_ARG before anything is launched.
 */
gdn_status gdn_causal_conv(const gdn_conv_shape *shape, const void *x, const void *weight,
                           const void *bias, const void *state_in, void *y, void *state_out,
                           void *stream);

/*
 * gdn_causal_conv_slots -- gdn_causal_conv against a pool of states, for continuous
 * batching (nuvec-core 0.6.1, src/fast/imp.rs, `causal_conv1d_slots`): row b starts from
 * pool[slots[b]] and its present state is written back there, in place.  Channels last
 * and no state window: x, y [B, L, C], pool [pool_size, carry, C], slots int32 [B] on the
 * device, distinct.  A slot outside [0, pool_size) skips its row (y untouched, pool
 * unchanged) and sets the device check word (gdn_last_device_status).
 */
gdn_status gdn_causal_conv_slots(const gdn_conv_shape *shape, const void *x, const void *weight,
                                 const void *bias, void *pool, int64_t pool_size,
                                 const int32_t *slots, void *y, void *stream);

/*
 * gdn_gated_rmsnorm -- GatedRMSNorm (ssm.rs `gated_rms_norm_op`) over `rows` rows of
 * `width` consecutive values (width = the scale's length; x, gate and y are [rows, width]
 * in memory, any leading shape):
 *   y = x / sqrt(mean(x^2) + epsilon) * scale * act(gate),
 *   act(g) = g * sigmoid(g) (GDN_ACT_SILU) or sigmoid(g) (GDN_ACT_SIGMOID),
 * in fp32, rounded once to io_dtype, which x, scale, gate and y share.  y may be x.
 * Bad arguments return GDN_ERR_INVALID_ARG before anything is launched.
 */
gdn_status gdn_gated_rmsnorm(int32_t io_dtype, int64_t rows, int32_t width, const void *x,
                             const void *scale, const void *gate, float epsilon,
                             int32_t activation, void *y, void *stream);

/*
 * gdn_prefill_norm -- gdn_prefill followed by the gated RMS norm of its output over each
 * d_v row, the two steps on either side of o in the layer (the CUDA page's
 * linear_attention_core Steps 1-4, then the onnxruntime-ep-mlx ssm.rs page's
 * GatedRMSNorm): y[t, h, :] = o * rsqrt(mean(o^2) + epsilon) * norm_scale * act(gate[t, h, :]),
 * with o rounded to the I/O type first, as gdn_prefill would store it, and act as in
 * gdn_gated_rmsnorm.
 *   norm_scale  DEVICE [d_v], io dtype.
 *   gate        DEVICE, o's layout ([B, T, h_v, d_v], or packed), io dtype; must not
 *               overlap y (GDN_ERR_INVALID_ARG).
 *   epsilon     finite and >= 0; activation GDN_ACT_SILU or GDN_ACT_SIGMOID.
 *   y           DEVICE, o's layout.  o itself is not an output.
 *   the rest    as gdn_prefill (workspace sized by gdn_prefill_workspace_bytes).
 *   fuse        0: the prefill writes o into y and the norm runs after it, in place (two
 *               launches of this library's kernels on top of the prefill's; the faster
 *               form on GB300).  1: on the chunked tensor-core path (16-bit I/O,
 *               d_k = d_v = 128) with a 16-byte aligned gate, the norm runs in the state
 *               scan's readout: the two CTAs that own a head's two 64-column halves of the
 *               state run as a thread-block cluster and exchange each row's sum of squares
 *               through shared memory, so o never reaches global memory (that path never
 *               takes the time-parallel scan); elsewhere as 0.  The results agree to one
 *               rounding of the I/O type.
 * Errors: gdn_prefill's, and gdn_gated_rmsnorm's argument rules.
 */
gdn_status gdn_prefill_norm(const gdn_shape *shape, const void *q, const void *k, const void *v,
                            const void *a, const void *b, const float *A_log,
                            const float *dt_bias, const float *state_in,
                            const int32_t *cu_seqlens, float scale, const void *norm_scale,
                            const void *gate, float epsilon, int32_t activation, int32_t fuse,
                            void *y, float *state_out, void *workspace, size_t workspace_bytes,
                            void *stream);

/*
 * gdn_layer_params -- the neighbouring ops of gdn_decode_layer.
 */
typedef struct gdn_layer_params {
    int32_t conv_kernel;       /* K taps of the causal convolution, 1..8 (dilation 1)      */
    int32_t conv_activation;   /* GDN_ACT_NONE or GDN_ACT_SILU                              */
    int32_t norm_activation;   /* GDN_ACT_SILU or GDN_ACT_SIGMOID                           */
    float norm_epsilon;        /* finite, >= 0                                              */
} gdn_layer_params;

/*
 * gdn_decode_layer -- one decode token of a whole gated delta-rule layer in one launch:
 * the three ops gdn_causal_conv (onnxruntime-ep-mlx ssm.rs `causal_conv_op`),
 * gdn_decode_step (onnx-runtime-ep-cuda linear_attention.rs `linear_attention_core`,
 * Steps 1-4) and gdn_gated_rmsnorm (ssm.rs `gated_rms_norm_op`) applied in that order,
 * with q, k and v taken from the convolution's output and the norm applied to the step's
 * output o.  Each intermediate is rounded to io_dtype exactly as the separate calls would
 * store it, but none is written to memory.
 *   x            [B, 1, C] the layer's mixed row, C = 2 h_qk d_k + h_v d_v, read as
 *                [q (h_qk x d_k) | k (h_qk x d_k) | v (h_v x d_v)], heads outer.
 *   conv_weight  [C, 1, K]; conv_bias [C] or NULL; the convolution uses dilation 1.
 *   conv_state_in  [B, K - 1, C] (channels last, oldest position first) or NULL (zeros);
 *   conv_state_out [B, K - 1, C] or NULL (not written): the last K - 1 inputs.  It must
 *                not overlap conv_state_in: several CTAs read the same q and k channels, so
 *                the update cannot be in place.  Callers alternate two buffers.
 *   a, b         [B, 1, h_v]; A_log, dt_bias [h_v] fp32; state [B, h_v, d_k, d_v] fp32,
 *                updated in place; scale 0 means 1 / sqrt(d_k).
 *   norm_scale   [d_v]; gate [B, 1, h_v, d_v]; y [B, 1, h_v, d_v], the normed output:
 *                y = o / sqrt(mean(o^2) + norm_epsilon) * norm_scale * act(gate) per
 *                (sequence, value head) row.
 * Shape (gdn_shape): seqlen 1, no cu_seqlens, d_k = 128, d_v a multiple of 64 up to 256,
 * any io_dtype, which x, conv_weight, conv_bias, the conv states, a, b, norm_scale, gate
 * and y share.  Every pointer is device memory owned by the caller and 16-byte aligned.
 * Bad arguments return GDN_ERR_INVALID_ARG before anything is launched.  The pages run
 * these ops as three kernels; the fused form exists to read q, k, v and o from no
 * intermediate buffer.
 */
gdn_status gdn_decode_layer(const gdn_shape *shape, const gdn_layer_params *layer, const void *x,
                            const void *conv_weight, const void *conv_bias,
                            const void *conv_state_in, void *conv_state_out, const void *a,
                            const void *b, const float *A_log, const float *dt_bias, float *state,
                            float scale, const void *norm_scale, const void *gate, void *y,
                            void *stream);

/*
 * gdn_prefill_layer -- the prefill of a whole gated delta-rule layer: gdn_causal_conv
 * (onnxruntime-ep-mlx ssm.rs `causal_conv_op`) on the layer's mixed input, gdn_prefill
 * (onnx-runtime-ep-cuda linear_attention.rs `linear_attention_core`, Steps 1-4) on its q,
 * k and v, then gdn_gated_rmsnorm (ssm.rs `gated_rms_norm_op`) on o, in that order, with
 * packed sequences handled by the convolution as by the prefill.  fuse = 0 (the faster
 * form on GB300): one streaming pass convolves every token of x into q, k and v in the
 * workspace, then the chunked prefill reads them.  fuse = 1: the prefill's prep kernel
 * convolves each chunk's q, k and v channels straight into its operand tiles, and v never
 * reaches memory.  The norm then runs in place on y.  Each intermediate is rounded to
 * io_dtype as the separate calls would store it, and the convolution sums in their order,
 * so the results equal conv -> prefill -> norm.
 *   x            [tokens, C] (packed with cu_seqlens, or [B, T, C]), C = 2 h_qk d_k +
 *                h_v d_v, read as [q (h_qk x d_k) | k (h_qk x d_k) | v (h_v x d_v)].
 *   conv_weight  [C, 1, K] with K = layer->conv_kernel in 1..4; conv_bias [C] or NULL;
 *                dilation 1; layer->conv_activation GDN_ACT_NONE or GDN_ACT_SILU.
 *   conv_state_in  [sequences, K - 1, C] (oldest position first) or NULL (zeros): the
 *                inputs before each sequence's first token.
 *   conv_state_out [sequences, K - 1, C]: each sequence's last K - 1 inputs (state rows
 *                first when the sequence is shorter).  It must not overlap conv_state_in.
 *   a, b, A_log, dt_bias, state_in, cu_seqlens, scale, state_out: as gdn_prefill.
 *   norm_scale [d_v]; gate like y; layer->norm_activation and norm_epsilon as
 *                gdn_gated_rmsnorm; y [tokens, h_v, d_v], 16-byte aligned, not overlapping
 *                gate.
 *   workspace    at least gdn_prefill_layer_workspace_bytes(shape) bytes: gdn_prefill's
 *                plus the convolved q, k and v (tokens x (2 h_qk + h_v) x 128 16-bit values;
 *                fuse = 1 needs only q and k).
 * Shape: io_dtype bf16 or f16 and d_k = d_v = 128 (GDN_ERR_UNSUPPORTED otherwise); x and
 * the conv states 16-byte aligned.  Every pointer is device memory owned by the caller.
 * Errors are gdn_prefill's and gdn_causal_conv's argument rules, checked before anything
 * is launched.
 */
gdn_status gdn_prefill_layer(const gdn_shape *shape, const gdn_layer_params *layer, const void *x,
                             const void *conv_weight, const void *conv_bias, const void *conv_state_in,
                             void *conv_state_out, const void *a, const void *b, const float *A_log,
                             const float *dt_bias, const float *state_in, const int32_t *cu_seqlens,
                             float scale, const void *norm_scale, const void *gate, void *y,
                             float *state_out, int32_t fuse, void *workspace, size_t workspace_bytes,
                             void *stream);

/* gdn_prefill_layer_workspace_bytes -- the workspace gdn_prefill_layer needs for `shape`
 * (0 off the tensor-core shapes); never fails. */
size_t gdn_prefill_layer_workspace_bytes(const gdn_shape *shape);

/*
 * gdn_last_device_status -- synchronise `stream`, read the device check word
 * set by any earlier call on the current device, clear it, and return GDN_OK or
 * GDN_ERR_DEVICE_CHECK (malformed cu_seqlens, or a slot outside the pool) /
 * GDN_ERR_TIMEOUT.
 */
gdn_status gdn_last_device_status(void *stream);

/*
 * gdn_prefill_plan -- report, without launching anything, which kernel path
 * gdn_prefill takes for `shape` (*path: 1 = token-sequential SIMT scan,
 * 2 = chunked tensor-core scan, 3 = chunked tensor-core scan run time-parallel) and how
 * many kernels one call launches (*launches).  Path 3 assumes the workspace that
 * gdn_prefill_workspace_bytes reports; with less (down to the records alone) the call
 * takes path 2.  Returns the same status gdn_prefill's shape checks would.
 */
gdn_status gdn_prefill_plan(const gdn_shape *shape, int32_t *path, int32_t *launches);

/*
 * gdn_set_wait_budget -- a test hook, process-wide and not part of the operation: the
 * cycles a bounded wait of the tensor-core prefill kernels (chunk prep and state scan)
 * or of the causal conv's bulk-copy pipeline (16-bit rows of 64 tokens or more) may take
 * before the waiting CTA gives up, for calls made after it (0 = the default, about two
 * seconds).  A wait that runs out makes the CTA let the copies and MMAs it has issued
 * finish under the full two-second budget, free its tensor memory and leave;
 * gdn_last_device_status() then returns GDN_ERR_TIMEOUT and the call's outputs are
 * undefined.  Nothing is left running or waiting on the device.
 * A negative value returns GDN_ERR_INVALID_ARG.
 */
gdn_status gdn_set_wait_budget(int64_t cycles);

/* Static name of a status code. */
const char *gdn_status_string(gdn_status status);

/* Detail of the last non-OK status returned on the calling host thread. */
const char *gdn_last_error_message(void);

#ifdef __cplusplus
}
#endif

#endif /* GDN_H */
