// gdn_api.cu -- the C ABI of libgdn: argument checks, status codes, dispatch.
//
// The checks mirror the host validation of onnx-runtime-ep-cuda 0.1.0-dev.6,
// src/kernels/linear_attention.rs (`LinearAttentionKernel::execute`): shapes,
// head divisibility, d_k <= 256, pointer presence; bad arguments return
// GDN_ERR_INVALID_ARG and unbuilt geometry GDN_ERR_UNSUPPORTED, and in both
// cases nothing is launched.  Unlike that page the calls never synchronise.
#include <math.h>
#include <stdarg.h>
#include <stdio.h>
#include <string.h>

#include "gdn_internal.cuh"

namespace gdn {

// Device check word: kernels OR error bits into it instead of trapping.
__device__ int g_device_status = 0;

namespace {

thread_local char g_message[512] = "";

gdn_status fail(gdn_status s, const char *fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_message, sizeof(g_message), fmt, ap);
    va_end(ap);
    return s;
}

gdn_status cuda_fail(cudaError_t e, const char *what) {
    return fail(GDN_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

// Address of the check word in the current device's context, looked up on every call so
// that a context created again after cudaDeviceReset never sees a stale address.
gdn_status status_word(int **out) {
    void *ptr = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&ptr, g_device_status);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(check word)");
    *out = static_cast<int *>(ptr);
    return GDN_OK;
}

bool aligned(const void *p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

size_t io_size(int32_t io) { return io == GDN_F32 ? 4 : 2; }

// Shape rules common to both calls.
gdn_status check_shape(const gdn_shape *s, bool varlen) {
    if (s == nullptr) return fail(GDN_ERR_INVALID_ARG, "shape is NULL");
    if (s->io_dtype != GDN_F32 && s->io_dtype != GDN_BF16 && s->io_dtype != GDN_F16)
        return fail(GDN_ERR_INVALID_ARG, "io_dtype %d is not F32/BF16/F16", s->io_dtype);
    if (s->seqlen < 0) return fail(GDN_ERR_INVALID_ARG, "seqlen %lld < 0", (long long)s->seqlen);
    if (s->num_seqs < 0) return fail(GDN_ERR_INVALID_ARG, "num_seqs %d < 0", s->num_seqs);
    if (varlen) {
        if (s->batch != 1)
            return fail(GDN_ERR_INVALID_ARG, "batch must be 1 with cu_seqlens (got %d)", s->batch);
    } else if (s->batch != s->num_seqs) {
        return fail(GDN_ERR_INVALID_ARG, "num_seqs (%d) must equal batch (%d)", s->num_seqs,
                    s->batch);
    }
    if (s->h_qk <= 0 || s->h_v <= 0)
        return fail(GDN_ERR_INVALID_ARG, "head counts must be positive (h_qk %d, h_v %d)",
                    s->h_qk, s->h_v);
    if (s->h_v % s->h_qk != 0)
        return fail(GDN_ERR_INVALID_ARG, "h_v (%d) must be a multiple of h_qk (%d)", s->h_v,
                    s->h_qk);
    if (s->d_k <= 0 || s->d_v <= 0)
        return fail(GDN_ERR_INVALID_ARG, "d_k (%d) and d_v (%d) must be positive", s->d_k, s->d_v);
    if (s->d_k > 256 || s->d_v > 256)
        return fail(GDN_ERR_UNSUPPORTED, "d_k (%d) and d_v (%d) above 256 are not built", s->d_k,
                    s->d_v);
    if (s->d_v % 4 != 0)
        return fail(GDN_ERR_UNSUPPORTED, "d_v (%d) must be a multiple of 4", s->d_v);
    return GDN_OK;
}

gdn_status check_inputs(const gdn_shape *s, int64_t tokens, const void *q, const void *k,
                        const void *v, const void *a, const void *b, const float *A_log,
                        const float *dt_bias, const void *o) {
    if (tokens > 0) {
        const void *ptrs[] = {q, k, v, a, b, A_log, dt_bias, o};
        const char *names[] = {"q", "k", "v", "a", "b", "A_log", "dt_bias", "o"};
        for (int i = 0; i < 8; ++i)
            if (ptrs[i] == nullptr) return fail(GDN_ERR_INVALID_ARG, "%s is NULL", names[i]);
        const size_t es = io_size(s->io_dtype);
        const void *io_ptrs[] = {q, k, v, a, b, o};
        for (int i = 0; i < 6; ++i)
            if (!aligned(io_ptrs[i], es))
                return fail(GDN_ERR_INVALID_ARG, "pointer is not %zu-byte aligned", es);
        if (!aligned(A_log, 4) || !aligned(dt_bias, 4))
            return fail(GDN_ERR_INVALID_ARG, "A_log/dt_bias must be 4-byte aligned");
    }
    return GDN_OK;
}

// Inputs of a call with a gate / rule variant: q, k, v and o always; a, A_log and
// dt_bias for a decaying rule, b for a delta rule (the others may be NULL).
gdn_status check_variant(const gdn_shape *shape, const gdn_variant *variant, int64_t tokens,
                         const void *q, const void *k, const void *v, const void *a, const void *b,
                         const float *A_log, const float *dt_bias, const void *o) {
    if (variant->rule < GDN_RULE_GATED_DELTA || variant->rule > GDN_RULE_LINEAR)
        return fail(GDN_ERR_INVALID_ARG, "rule %d is not a gdn_rule", variant->rule);
    const bool has_decay = variant->rule == GDN_RULE_GATED_DELTA || variant->rule == GDN_RULE_GATED;
    const bool has_delta = variant->rule == GDN_RULE_GATED_DELTA || variant->rule == GDN_RULE_DELTA;
    if (tokens > 0) {
        if (!q || !k || !v || !o) return fail(GDN_ERR_INVALID_ARG, "q, k, v or o is NULL");
        if (has_decay && (!a || !A_log || !dt_bias))
            return fail(GDN_ERR_INVALID_ARG, "a decaying rule needs a, A_log and dt_bias");
        if (has_delta && !b) return fail(GDN_ERR_INVALID_ARG, "a delta rule needs b");
        const size_t es = io_size(shape->io_dtype);
        const void *io_ptrs[] = {q, k, v, a, b, o};
        for (const void *ptr : io_ptrs)
            if (ptr && !aligned(ptr, es))
                return fail(GDN_ERR_INVALID_ARG, "pointer is not %zu-byte aligned", es);
        if ((A_log && !aligned(A_log, 4)) || (dt_bias && !aligned(dt_bias, 4)))
            return fail(GDN_ERR_INVALID_ARG, "A_log/dt_bias must be 4-byte aligned");
    }
    return GDN_OK;
}

}  // namespace

// Record `message` as the calling thread's last error detail and return `status`
// (for entry points defined in other translation units).
gdn_status report_error(gdn_status status, const char *message) {
    return fail(status, "%s", message);
}

}  // namespace gdn

using namespace gdn;

extern "C" {

const char *gdn_status_string(gdn_status st) {
    switch (st) {
        case GDN_OK: return "GDN_OK";
        case GDN_ERR_INVALID_ARG: return "GDN_ERR_INVALID_ARG";
        case GDN_ERR_UNSUPPORTED: return "GDN_ERR_UNSUPPORTED";
        case GDN_ERR_CUDA: return "GDN_ERR_CUDA";
        case GDN_ERR_DEVICE_CHECK: return "GDN_ERR_DEVICE_CHECK";
        case GDN_ERR_TIMEOUT: return "GDN_ERR_TIMEOUT";
    }
    return "GDN_ERR_UNKNOWN";
}

const char *gdn_last_error_message(void) { return g_message; }

gdn_status gdn_prefill_plan(const gdn_shape *shape, int32_t *path, int32_t *launches) {
    gdn_status st = check_shape(shape, shape != nullptr && shape->batch == 1 &&
                                           shape->num_seqs != 1);
    if (st != GDN_OK) return st;
    const bool varlen = shape->batch == 1 && shape->num_seqs != 1;
    const int64_t tokens = varlen ? shape->seqlen : shape->seqlen * (int64_t)shape->batch;
    const bool tc = prefill_tc_shape_ok((gdn_dtype)shape->io_dtype, shape->d_k, shape->d_v, tokens);
    // Time-parallel scan: prep, scan, one combine per segment boundary and the correction;
    // else the prep and scan of every chunk segment.
    const int tps = tc ? prefill_tc_tp_nseg(varlen, shape->seqlen, shape->batch, shape->h_v) : 1;
    if (path) *path = tc ? (tps > 1 ? 3 : 2) : 1;
    const int nseg = tc ? prefill_tc_segments(varlen, shape->seqlen, shape->batch, shape->h_v) : 1;
    if (launches) *launches = shape->num_seqs > 0 ? (tc ? (tps > 1 ? 2 + tps : 2 * nseg) : 1) : 0;
    return GDN_OK;
}

// Packed sequences come with batch == 1; a single batch-1 sequence is sized as packed too,
// which covers both readings.
size_t gdn_prefill_workspace_bytes(const gdn_shape *shape) {
    const size_t records = gdn::prefill_records_bytes(shape);
    if (records == 0) return 0;
    // Records, plus the time-parallel scan's buffers when a batched call of this shape
    // would use it (with batch 1 the shape may also be a packed call: the sum covers both).
    return records + prefill_tc_tp_bytes(false, shape->seqlen, shape->batch, shape->h_v);
}

size_t gdn_prefill_variant_workspace_bytes(const gdn_shape *shape, const gdn_variant *variant) {
    const size_t base = gdn_prefill_workspace_bytes(shape);
    if (base == 0 || variant == nullptr || !variant->decay_per_key) return base;
    if (variant->rule != GDN_RULE_GATED_DELTA && variant->rule != GDN_RULE_GATED) return base;
    // Q o e^G and K o e^{G_C - G} per value head, for the packed or batched reading alike.
    return base + prefill_tc_pk_bytes(shape->seqlen * (int64_t)shape->batch, shape->h_v);
}

gdn_status gdn_prefill_variant_plan(const gdn_shape *shape, const gdn_variant *variant, int32_t *path,
                                    int32_t *launches) {
    if (variant == nullptr) return fail(GDN_ERR_INVALID_ARG, "variant is NULL");
    if (variant->rule < GDN_RULE_GATED_DELTA || variant->rule > GDN_RULE_LINEAR)
        return fail(GDN_ERR_INVALID_ARG, "rule %d is not a gdn_rule", variant->rule);
    // Every variant takes gdn_prefill's path, given gdn_prefill_variant_workspace_bytes.
    return gdn_prefill_plan(shape, path, launches);
}

gdn_status gdn_set_wait_budget(int64_t cycles) {
    if (cycles < 0) return fail(GDN_ERR_INVALID_ARG, "wait budget %lld < 0", (long long)cycles);
    __atomic_store_n(&g_wait_budget, (long long)cycles, __ATOMIC_RELAXED);
    return GDN_OK;
}

gdn_status gdn_prefill(const gdn_shape *shape, const void *q, const void *k, const void *v,
                       const void *a, const void *b, const float *A_log, const float *dt_bias,
                       const float *state_in, const int32_t *cu_seqlens, float scale, void *o,
                       float *state_out, void *workspace, size_t workspace_bytes, void *stream) {
    return prefill_impl(shape, q, k, v, a, b, A_log, dt_bias, state_in, cu_seqlens, scale, o,
                        state_out, workspace, workspace_bytes, true, stream);
}

gdn_status gdn_prefill_norm(const gdn_shape *shape, const void *q, const void *k, const void *v,
                            const void *a, const void *b, const float *A_log,
                            const float *dt_bias, const float *state_in,
                            const int32_t *cu_seqlens, float scale, const void *norm_scale,
                            const void *gate, float epsilon, int32_t activation, int32_t fuse,
                            void *y, float *state_out, void *workspace, size_t workspace_bytes,
                            void *stream) {
    const NormEpilogue norm{norm_scale, gate, epsilon, activation, fuse != 0};
    return prefill_impl(shape, q, k, v, a, b, A_log, dt_bias, state_in, cu_seqlens, scale, y,
                        state_out, workspace, workspace_bytes, true, stream, nullptr, &norm);
}

size_t gdn_prefill_layer_workspace_bytes(const gdn_shape *shape) {
    const size_t base = gdn_prefill_workspace_bytes(shape);
    if (base == 0) return 0;
    const int64_t tokens = shape->seqlen * (int64_t)shape->batch;
    return base + prefill_tc_conv_bytes(tokens, shape->h_qk) + prefill_tc_conv_v_bytes(tokens, shape->h_v);
}

gdn_status gdn_prefill_layer(const gdn_shape *shape, const gdn_layer_params *layer, const void *x,
                             const void *conv_weight, const void *conv_bias, const void *conv_state_in,
                             void *conv_state_out, const void *a, const void *b, const float *A_log,
                             const float *dt_bias, const float *state_in, const int32_t *cu_seqlens,
                             float scale, const void *norm_scale, const void *gate, void *y,
                             float *state_out, int32_t fuse, void *workspace, size_t workspace_bytes,
                             void *stream) {
    gdn_status st = check_shape(shape, cu_seqlens != nullptr);
    if (st != GDN_OK) return st;
    if (layer == nullptr) return fail(GDN_ERR_INVALID_ARG, "layer is NULL");
    if (layer->conv_kernel < 1 || layer->conv_kernel > 4)
        return fail(GDN_ERR_INVALID_ARG, "conv_kernel %d is not in 1..4", layer->conv_kernel);
    if (layer->conv_activation != GDN_ACT_NONE && layer->conv_activation != GDN_ACT_SILU)
        return fail(GDN_ERR_INVALID_ARG, "the convolution's activation is NONE or SILU");
    if (shape->io_dtype == GDN_F32 || shape->d_k != 128 || shape->d_v != 128)
        return fail(GDN_ERR_UNSUPPORTED, "the layer prefill runs on the tensor-core path: 16-bit I/O, d_k = d_v = 128");
    const int64_t tokens = cu_seqlens ? shape->seqlen : shape->seqlen * (int64_t)shape->batch;
    const size_t es = io_size(shape->io_dtype);
    const int64_t C = 2LL * shape->h_qk * shape->d_k + (int64_t)shape->h_v * shape->d_v;
    const int64_t nseq = shape->num_seqs;
    const size_t state_bytes = (size_t)nseq * (size_t)(layer->conv_kernel - 1) * (size_t)C * es;
    if (nseq > 0 && tokens > 0) {
        if (x == nullptr || conv_weight == nullptr) return fail(GDN_ERR_INVALID_ARG, "x or conv_weight is NULL");
        if (!aligned(x, 16) || !aligned(conv_state_in, 16) || !aligned(conv_state_out, 16))
            return fail(GDN_ERR_INVALID_ARG, "x and the conv states must be 16-byte aligned");
        if (!aligned(conv_weight, es) || !aligned(conv_bias, es))
            return fail(GDN_ERR_INVALID_ARG, "conv_weight / conv_bias is misaligned");
    }
    if (state_bytes > 0 && nseq > 0) {
        if (conv_state_out == nullptr) return fail(GDN_ERR_INVALID_ARG, "conv_state_out is NULL");
        if (conv_state_in != nullptr) {
            const uintptr_t i0 = reinterpret_cast<uintptr_t>(conv_state_in), o0 = reinterpret_cast<uintptr_t>(conv_state_out);
            if (i0 < o0 + state_bytes && o0 < i0 + state_bytes)
                return fail(GDN_ERR_INVALID_ARG, "conv_state_out overlaps conv_state_in (the update cannot be in place)");
        }
    }
    const NormEpilogue norm{norm_scale, gate, layer->norm_epsilon, layer->norm_activation, false};
    if (tokens == 0 || nseq == 0) {
        // No token: the present conv state is the past one, and the prefill copies its state.
        if (state_bytes > 0 && nseq > 0) {
            const cudaError_t e = conv_state_in != nullptr
                                      ? cudaMemcpyAsync(conv_state_out, conv_state_in, state_bytes,
                                                        cudaMemcpyDeviceToDevice, (cudaStream_t)stream)
                                      : cudaMemsetAsync(conv_state_out, 0, state_bytes, (cudaStream_t)stream);
            if (e != cudaSuccess) return cuda_fail(e, "conv state copy");
        }
        return prefill_impl(shape, x, x, x, a, b, A_log, dt_bias, state_in, cu_seqlens, scale, y,
                            state_out, workspace, workspace_bytes, true, stream, nullptr, &norm);
    }
    const ConvPrologue conv{x, conv_weight, conv_bias, conv_state_in, conv_state_out, layer->conv_kernel,
                            layer->conv_activation == GDN_ACT_SILU, fuse != 0};
    // q, k and v are x's channels: x stands in for them in the argument checks.
    return prefill_impl(shape, x, x, x, a, b, A_log, dt_bias, state_in, cu_seqlens, scale, y,
                        state_out, workspace, workspace_bytes, true, stream, nullptr, &norm, &conv);
}

}  // extern "C"

size_t gdn::prefill_records_bytes(const gdn_shape *shape) {
    return prefill_records_bytes_for(shape, shape != nullptr && shape->batch == 1);
}

size_t gdn::prefill_records_bytes_for(const gdn_shape *shape, bool varlen) {
    if (shape == nullptr || shape->seqlen < 0 || shape->batch < 0 || shape->num_seqs < 0 ||
        shape->h_v <= 0)
        return 0;
    const int64_t tokens = varlen ? shape->seqlen : shape->seqlen * (int64_t)shape->batch;
    if (!prefill_tc_shape_ok((gdn_dtype)shape->io_dtype, shape->d_k, shape->d_v, tokens)) return 0;
    return prefill_tc_workspace(varlen, shape->seqlen, shape->batch, shape->num_seqs, shape->h_v);
}

gdn_status gdn::prefill_impl(const gdn_shape *shape, const void *q, const void *k, const void *v,
                             const void *a, const void *b, const float *A_log, const float *dt_bias,
                             const float *state_in, const int32_t *cu_seqlens, float scale, void *o,
                             float *state_out, void *workspace, size_t workspace_bytes,
                             bool allow_overlap, void *stream, const gdn_variant *variant,
                             const NormEpilogue *norm, const ConvPrologue *conv) {
    gdn_status st = check_shape(shape, cu_seqlens != nullptr);
    if (st != GDN_OK) return st;
    const int64_t tokens = cu_seqlens ? shape->seqlen : shape->seqlen * (int64_t)shape->batch;
    if (variant == nullptr) {
        st = check_inputs(shape, tokens, q, k, v, a, b, A_log, dt_bias, o);
    } else {
        st = check_variant(shape, variant, tokens, q, k, v, a, b, A_log, dt_bias, o);
    }
    if (st != GDN_OK) return st;
    const size_t es = io_size(shape->io_dtype);
    if (norm != nullptr) {
        if (norm->activation != GDN_ACT_SILU && norm->activation != GDN_ACT_SIGMOID)
            return fail(GDN_ERR_INVALID_ARG, "the norm's activation is SILU or SIGMOID");
        if (!(norm->eps >= 0.0f) || isinf(norm->eps))
            return fail(GDN_ERR_INVALID_ARG, "epsilon must be finite and >= 0");
        if (tokens > 0) {
            if (!norm->scale || !norm->gate) return fail(GDN_ERR_INVALID_ARG, "norm_scale or gate is NULL");
            if (!aligned(norm->scale, es) || !aligned(norm->gate, es))
                return fail(GDN_ERR_INVALID_ARG, "norm_scale/gate is not %zu-byte aligned", es);
            const size_t bytes = (size_t)tokens * shape->h_v * shape->d_v * es;
            const uintptr_t g0 = reinterpret_cast<uintptr_t>(norm->gate), y0 = reinterpret_cast<uintptr_t>(o);
            if (g0 < y0 + bytes && y0 < g0 + bytes)
                return fail(GDN_ERR_INVALID_ARG, "y overlaps gate");
        }
    }
    if (shape->num_seqs == 0) return GDN_OK;
    if (state_out == nullptr) return fail(GDN_ERR_INVALID_ARG, "state_out is NULL");
    if (!aligned(state_out, 16) || !aligned(state_in, 16))
        return fail(GDN_ERR_INVALID_ARG, "state_in/state_out must be 16-byte aligned");
    if (!(scale == scale) || isinf(scale)) return fail(GDN_ERR_INVALID_ARG, "scale is not finite");
    int *word = nullptr;
    st = status_word(&word);
    if (st != GDN_OK) return st;

    ScanParams p{};
    p.q = q; p.k = k; p.v = v; p.a = a; p.b = b;
    p.A_log = A_log; p.dt_bias = dt_bias;
    p.state_in = state_in; p.state_out = state_out; p.o = o;
    p.cu_seqlens = cu_seqlens;
    p.seqlen = shape->seqlen;
    p.num_seqs = shape->num_seqs;
    p.h_qk = shape->h_qk; p.h_v = shape->h_v; p.d_k = shape->d_k; p.d_v = shape->d_v;
    p.scale = scale == 0.0f ? 1.0f / sqrtf((float)shape->d_k) : scale;
    p.status = word;
    if (variant != nullptr) {
        p.rule = variant->rule;
        p.decay_per_key = variant->decay_per_key != 0;
        p.beta_shared = variant->beta_shared != 0;
    }
    if (conv != nullptr) {
        p.conv_x = conv->x; p.conv_w = conv->weight; p.conv_b = conv->bias;
        p.conv_in = conv->state_in; p.conv_out = conv->state_out;
        p.conv_k = conv->kernel; p.conv_silu = conv->silu;
        p.conv_fuse = conv->fuse;
    }
    const gdn_dtype io = (gdn_dtype)shape->io_dtype;
    cudaError_t e;
    bool norm_after = norm != nullptr && tokens > 0;   // the norm as its own launch, in place
    // One decay per key dimension (with a decaying rule) takes the tensor-core path when
    // the workspace also holds its Q~ and K~ arrays, else the token-sequential one.
    const bool per_key = p.decay_per_key && (p.rule == GDN_RULE_GATED_DELTA || p.rule == GDN_RULE_GATED);
    const size_t pk_bytes = per_key ? prefill_tc_pk_bytes(tokens, shape->h_v) : 0;
    const size_t records = prefill_tc_workspace(cu_seqlens != nullptr, shape->seqlen, shape->batch,
                                                shape->num_seqs, shape->h_v);
    // (The per-key path reads a's [64 tokens x 128] tiles by TMA: a must be 16-byte aligned.)
    const bool pk_room = !per_key || (workspace != nullptr && workspace_bytes >= records + pk_bytes &&
                                      aligned(a, 16));
    const size_t conv_bytes = conv == nullptr ? 0
                              : prefill_tc_conv_bytes(tokens, shape->h_qk) +
                                    (conv->fuse ? 0 : prefill_tc_conv_v_bytes(tokens, shape->h_v));
    if (conv != nullptr && !prefill_tc_supported(p, io, tokens))
        return fail(GDN_ERR_UNSUPPORTED, "the convolution prologue runs on the tensor-core prefill only");
    if (pk_room && prefill_tc_supported(p, io, tokens)) {
        if (norm_after && norm->fuse && aligned(norm->gate, 16)) {
            p.norm_scale = norm->scale;
            p.norm_gate = norm->gate;
            p.norm_eps = norm->eps;
            p.norm_silu = norm->activation == GDN_ACT_SILU;
            norm_after = false;
        }
        const size_t need = records + pk_bytes + conv_bytes;
        if (workspace == nullptr || workspace_bytes < need)
            return fail(GDN_ERR_INVALID_ARG, "workspace of %zu bytes is below the %zu this call needs",
                        workspace == nullptr ? (size_t)0 : workspace_bytes, need);
        if (!aligned(workspace, 16)) return fail(GDN_ERR_INVALID_ARG, "workspace must be 16-byte aligned");
        e = launch_prefill_tc(p, io, tokens, workspace, workspace_bytes, allow_overlap,
                              (cudaStream_t)stream);
        if (e != cudaSuccess) return cuda_fail(e, "tensor-core prefill launch");
    } else {
        e = launch_scan_simt(p, io, (cudaStream_t)stream);
        if (e != cudaSuccess) return cuda_fail(e, "prefill launch");
    }
    if (norm_after) {
        bool vec4 = shape->d_v % 4 == 0;
        const void *ptrs[] = {o, norm->scale, norm->gate};
        for (const void *ptr : ptrs)
            if (!aligned(ptr, 4 * es)) vec4 = false;
        e = launch_gated_rmsnorm(io, tokens * shape->h_v, shape->d_v, o, norm->scale, norm->gate,
                                 norm->eps, norm->activation, o, vec4, (cudaStream_t)stream);
        if (e != cudaSuccess) return cuda_fail(e, "gated RMS norm launch");
    }
    return GDN_OK;
}

extern "C" {

gdn_status gdn_decode_step(const gdn_shape *shape, const void *q, const void *k, const void *v,
                           const void *a, const void *b, const float *A_log,
                           const float *dt_bias, float *state, float scale, void *o,
                           void *stream) {
    gdn_status st = check_shape(shape, false);
    if (st != GDN_OK) return st;
    if (shape->seqlen != 1)
        return fail(GDN_ERR_INVALID_ARG, "decode takes seqlen 1 (got %lld)", (long long)shape->seqlen);
    st = check_inputs(shape, shape->batch, q, k, v, a, b, A_log, dt_bias, o);
    if (st != GDN_OK) return st;
    if (shape->batch == 0) return GDN_OK;
    if (state == nullptr) return fail(GDN_ERR_INVALID_ARG, "state is NULL");
    if (!aligned(state, 16)) return fail(GDN_ERR_INVALID_ARG, "state must be 16-byte aligned");
    if (!(scale == scale) || isinf(scale)) return fail(GDN_ERR_INVALID_ARG, "scale is not finite");
    int *word = nullptr;
    st = status_word(&word);
    if (st != GDN_OK) return st;

    ScanParams p{};
    p.q = q; p.k = k; p.v = v; p.a = a; p.b = b;
    p.A_log = A_log; p.dt_bias = dt_bias;
    p.state_in = state; p.state_out = state; p.o = o;
    p.cu_seqlens = nullptr;
    p.seqlen = 1;
    p.num_seqs = shape->batch;
    p.h_qk = shape->h_qk; p.h_v = shape->h_v; p.d_k = shape->d_k; p.d_v = shape->d_v;
    p.scale = scale == 0.0f ? 1.0f / sqrtf((float)shape->d_k) : scale;
    p.status = word;
    cudaError_t e = launch_scan_simt(p, (gdn_dtype)shape->io_dtype, (cudaStream_t)stream);
    if (e != cudaSuccess) return cuda_fail(e, "decode launch");
    return GDN_OK;
}

gdn_status gdn_decode_step_slots(const gdn_shape *shape, const void *q, const void *k,
                                 const void *v, const void *a, const void *b, const float *A_log,
                                 const float *dt_bias, float *pool, int64_t pool_size,
                                 const int32_t *slots, float scale, void *o, void *stream) {
    gdn_status st = check_shape(shape, false);
    if (st != GDN_OK) return st;
    if (shape->seqlen != 1)
        return fail(GDN_ERR_INVALID_ARG, "decode takes seqlen 1 (got %lld)", (long long)shape->seqlen);
    st = check_inputs(shape, shape->batch, q, k, v, a, b, A_log, dt_bias, o);
    if (st != GDN_OK) return st;
    if (shape->batch == 0) return GDN_OK;
    if (pool == nullptr || slots == nullptr) return fail(GDN_ERR_INVALID_ARG, "pool or slots is NULL");
    if (pool_size <= 0) return fail(GDN_ERR_INVALID_ARG, "pool_size %lld <= 0", (long long)pool_size);
    if (!aligned(pool, 16) || !aligned(slots, 4))
        return fail(GDN_ERR_INVALID_ARG, "pool must be 16-byte and slots 4-byte aligned");
    if (!(scale == scale) || isinf(scale)) return fail(GDN_ERR_INVALID_ARG, "scale is not finite");
    int *word = nullptr;
    st = status_word(&word);
    if (st != GDN_OK) return st;

    ScanParams p{};
    p.q = q; p.k = k; p.v = v; p.a = a; p.b = b;
    p.A_log = A_log; p.dt_bias = dt_bias;
    p.state_in = pool; p.state_out = pool; p.o = o;
    p.cu_seqlens = nullptr;
    p.seqlen = 1;
    p.num_seqs = shape->batch;
    p.h_qk = shape->h_qk; p.h_v = shape->h_v; p.d_k = shape->d_k; p.d_v = shape->d_v;
    p.scale = scale == 0.0f ? 1.0f / sqrtf((float)shape->d_k) : scale;
    p.status = word;
    p.slots = slots;
    p.pool_size = pool_size;
    cudaError_t e = launch_scan_simt(p, (gdn_dtype)shape->io_dtype, (cudaStream_t)stream);
    if (e != cudaSuccess) return cuda_fail(e, "slot decode launch");
    return GDN_OK;
}

gdn_status gdn_scan_window(const gdn_shape *shape, const void *q, const void *k, const void *v,
                           const void *a, const void *b, const float *A_log, const float *dt_bias,
                           const float *state_in, float scale, void *o, float *window,
                           int32_t window_len, void *stream) {
    gdn_status st = check_shape(shape, false);
    if (st != GDN_OK) return st;
    const int64_t tokens = shape->seqlen * (int64_t)shape->batch;
    st = check_inputs(shape, tokens, q, k, v, a, b, A_log, dt_bias, o);
    if (st != GDN_OK) return st;
    if (window_len < 1) return fail(GDN_ERR_INVALID_ARG, "window_len %d < 1", window_len);
    if (shape->batch == 0) return GDN_OK;
    if (window == nullptr) return fail(GDN_ERR_INVALID_ARG, "window is NULL");
    if (!aligned(window, 16) || !aligned(state_in, 16))
        return fail(GDN_ERR_INVALID_ARG, "state_in and window must be 16-byte aligned");
    if (!(scale == scale) || isinf(scale)) return fail(GDN_ERR_INVALID_ARG, "scale is not finite");
    int *word = nullptr;
    st = status_word(&word);
    if (st != GDN_OK) return st;

    ScanParams p{};
    p.q = q; p.k = k; p.v = v; p.a = a; p.b = b;
    p.A_log = A_log; p.dt_bias = dt_bias;
    p.state_in = state_in; p.state_out = nullptr; p.o = o;
    p.cu_seqlens = nullptr;
    p.seqlen = shape->seqlen;
    p.num_seqs = shape->batch;
    p.h_qk = shape->h_qk; p.h_v = shape->h_v; p.d_k = shape->d_k; p.d_v = shape->d_v;
    p.scale = scale == 0.0f ? 1.0f / sqrtf((float)shape->d_k) : scale;
    p.status = word;
    p.window = window;
    p.window_len = window_len;
    cudaError_t e = launch_scan_simt(p, (gdn_dtype)shape->io_dtype, (cudaStream_t)stream);
    if (e != cudaSuccess) return cuda_fail(e, "window scan launch");
    return GDN_OK;
}

gdn_status gdn_prefill_variant(const gdn_shape *shape, const gdn_variant *variant, const void *q,
                               const void *k, const void *v, const void *a, const void *b,
                               const float *A_log, const float *dt_bias, const float *state_in,
                               const int32_t *cu_seqlens, float scale, void *o, float *state_out,
                               void *workspace, size_t workspace_bytes, void *stream) {
    if (variant == nullptr) return fail(GDN_ERR_INVALID_ARG, "variant is NULL");
    return prefill_impl(shape, q, k, v, a, b, A_log, dt_bias, state_in, cu_seqlens, scale, o,
                        state_out, workspace, workspace_bytes, true, stream, variant);
}

gdn_status gdn_scan_variant(const gdn_shape *shape, const gdn_variant *variant, const void *q,
                            const void *k, const void *v, const void *a, const void *b,
                            const float *A_log, const float *dt_bias, const float *state_in,
                            const int32_t *cu_seqlens, float scale, void *o, float *state_out,
                            void *stream) {
    gdn_status st = check_shape(shape, cu_seqlens != nullptr);
    if (st != GDN_OK) return st;
    if (variant == nullptr) return fail(GDN_ERR_INVALID_ARG, "variant is NULL");
    const int64_t tokens = cu_seqlens ? shape->seqlen : shape->seqlen * (int64_t)shape->batch;
    st = check_variant(shape, variant, tokens, q, k, v, a, b, A_log, dt_bias, o);
    if (st != GDN_OK) return st;
    if (shape->num_seqs == 0) return GDN_OK;
    if (state_out == nullptr) return fail(GDN_ERR_INVALID_ARG, "state_out is NULL");
    if (!aligned(state_out, 16) || !aligned(state_in, 16))
        return fail(GDN_ERR_INVALID_ARG, "state_in/state_out must be 16-byte aligned");
    if (!(scale == scale) || isinf(scale)) return fail(GDN_ERR_INVALID_ARG, "scale is not finite");
    int *word = nullptr;
    st = status_word(&word);
    if (st != GDN_OK) return st;

    ScanParams p{};
    p.q = q; p.k = k; p.v = v; p.a = a; p.b = b;
    p.A_log = A_log; p.dt_bias = dt_bias;
    p.state_in = state_in; p.state_out = state_out; p.o = o;
    p.cu_seqlens = cu_seqlens;
    p.seqlen = shape->seqlen;
    p.num_seqs = shape->num_seqs;
    p.h_qk = shape->h_qk; p.h_v = shape->h_v; p.d_k = shape->d_k; p.d_v = shape->d_v;
    p.scale = scale == 0.0f ? 1.0f / sqrtf((float)shape->d_k) : scale;
    p.status = word;
    p.rule = variant->rule;
    p.decay_per_key = variant->decay_per_key != 0;
    p.beta_shared = variant->beta_shared != 0;
    cudaError_t e = launch_scan_simt(p, (gdn_dtype)shape->io_dtype, (cudaStream_t)stream);
    if (e != cudaSuccess) return cuda_fail(e, "variant scan launch");
    return GDN_OK;
}

namespace {

// Geometry rules of the convolution; with_window: the state window is allowed.
gdn_status check_conv(const gdn_conv_shape *s, bool with_window) {
    if (s == nullptr) return fail(GDN_ERR_INVALID_ARG, "shape is NULL");
    if (s->io_dtype != GDN_F32 && s->io_dtype != GDN_BF16 && s->io_dtype != GDN_F16)
        return fail(GDN_ERR_INVALID_ARG, "io_dtype %d is not a gdn_dtype", s->io_dtype);
    if (s->batch < 0 || s->seqlen < 0 || s->channels <= 0)
        return fail(GDN_ERR_INVALID_ARG, "batch, seqlen must be >= 0 and channels > 0");
    if (s->kernel < 1 || s->kernel > 64 || s->dilation < 1)
        return fail(GDN_ERR_INVALID_ARG, "kernel must be in 1..64 and dilation >= 1");
    if ((int64_t)(s->kernel - 1) * s->dilation > 4096)
        return fail(GDN_ERR_INVALID_ARG, "carry (kernel - 1) * dilation exceeds 4096");
    if (s->channels_last != 0 && s->channels_last != 1)
        return fail(GDN_ERR_INVALID_ARG, "channels_last must be 0 or 1");
    if (s->activation != GDN_ACT_NONE && s->activation != GDN_ACT_SILU)
        return fail(GDN_ERR_INVALID_ARG, "the convolution's activation is NONE or SILU");
    if (s->state_window < 0 || s->state_window > 8 || (!with_window && s->state_window != 0))
        return fail(GDN_ERR_INVALID_ARG, "state_window must be in 0..8 (0 with slots)");
    return GDN_OK;
}

gdn_status conv_impl(const gdn_conv_shape *shape, const void *x, const void *weight,
                     const void *bias, const void *state_in, void *y, void *state_out,
                     const int32_t *slots, int64_t pool_size, void *stream) {
    const size_t es = io_size(shape->io_dtype);
    const bool any = shape->batch > 0 && shape->seqlen > 0;
    if (any && (!x || !y)) return fail(GDN_ERR_INVALID_ARG, "x or y is NULL");
    if (shape->batch > 0 && !weight) return fail(GDN_ERR_INVALID_ARG, "weight is NULL");
    const void *ptrs[] = {x, weight, bias, state_in, y, state_out};
    for (const void *ptr : ptrs)
        if (ptr && !aligned(ptr, es))
            return fail(GDN_ERR_INVALID_ARG, "pointer is not %zu-byte aligned", es);
    if (shape->batch == 0) return GDN_OK;
    int *word = nullptr;
    gdn_status st = status_word(&word);
    if (st != GDN_OK) return st;
    ConvLaunch l{};
    l.io = (gdn_dtype)shape->io_dtype;
    l.x = x; l.w = weight; l.bias = bias; l.state_in = state_in;
    l.y = y; l.state_out = state_out;
    l.batch = shape->batch; l.seqlen = shape->seqlen;
    l.channels = shape->channels; l.kernel = shape->kernel; l.dilation = shape->dilation;
    l.channels_last = shape->channels_last; l.activation = shape->activation;
    l.window = shape->state_window;
    l.slots = slots; l.pool_size = pool_size;
    l.status = word;
    // Four channels per thread: channels last, C % 4 == 0, every pointer 4-element aligned.
    l.vec4 = shape->channels_last && shape->channels % 4 == 0;
    for (const void *ptr : ptrs)
        if (ptr && !aligned(ptr, 4 * es)) l.vec4 = false;
    l.align16 = (!x || aligned(x, 16)) && (!state_in || aligned(state_in, 16));
    cudaError_t e = launch_causal_conv(l, (cudaStream_t)stream);
    if (e != cudaSuccess) return cuda_fail(e, "causal conv launch");
    return GDN_OK;
}

}  // namespace

gdn_status gdn_causal_conv(const gdn_conv_shape *shape, const void *x, const void *weight,
                           const void *bias, const void *state_in, void *y, void *state_out,
                           void *stream) {
    gdn_status st = check_conv(shape, true);
    if (st != GDN_OK) return st;
    return conv_impl(shape, x, weight, bias, state_in, y, state_out, nullptr, 0, stream);
}

gdn_status gdn_causal_conv_slots(const gdn_conv_shape *shape, const void *x, const void *weight,
                                 const void *bias, void *pool, int64_t pool_size,
                                 const int32_t *slots, void *y, void *stream) {
    gdn_status st = check_conv(shape, false);
    if (st != GDN_OK) return st;
    if (!shape->channels_last) return fail(GDN_ERR_INVALID_ARG, "the pool form is channels last");
    if (pool_size < 0) return fail(GDN_ERR_INVALID_ARG, "pool_size must be >= 0");
    if (shape->batch > 0 && (!slots || !aligned(slots, 4)))
        return fail(GDN_ERR_INVALID_ARG, "slots is NULL or misaligned");
    if (shape->batch > 0 && shape->kernel > 1 && !pool)
        return fail(GDN_ERR_INVALID_ARG, "pool is NULL");
    return conv_impl(shape, x, weight, bias, pool, y, pool, slots, pool_size, stream);
}

gdn_status gdn_gated_rmsnorm(int32_t io_dtype, int64_t rows, int32_t width, const void *x,
                             const void *scale, const void *gate, float epsilon,
                             int32_t activation, void *y, void *stream) {
    if (io_dtype != GDN_F32 && io_dtype != GDN_BF16 && io_dtype != GDN_F16)
        return fail(GDN_ERR_INVALID_ARG, "io_dtype %d is not a gdn_dtype", io_dtype);
    if (rows < 0 || width <= 0) return fail(GDN_ERR_INVALID_ARG, "rows >= 0 and width > 0");
    if (activation != GDN_ACT_SILU && activation != GDN_ACT_SIGMOID)
        return fail(GDN_ERR_INVALID_ARG, "the norm's activation is SILU or SIGMOID");
    if (!(epsilon >= 0.0f) || isinf(epsilon))
        return fail(GDN_ERR_INVALID_ARG, "epsilon must be finite and >= 0");
    if (rows == 0) return GDN_OK;
    if (!x || !scale || !gate || !y) return fail(GDN_ERR_INVALID_ARG, "x, scale, gate or y is NULL");
    const size_t es = io_size(io_dtype);
    const void *ptrs[] = {x, scale, gate, y};
    bool vec4 = width % 4 == 0;
    for (const void *ptr : ptrs) {
        if (!aligned(ptr, es)) return fail(GDN_ERR_INVALID_ARG, "pointer is not %zu-byte aligned", es);
        if (!aligned(ptr, 4 * es)) vec4 = false;
    }
    cudaError_t e = launch_gated_rmsnorm((gdn_dtype)io_dtype, rows, width, x, scale, gate, epsilon,
                                         activation, y, vec4, (cudaStream_t)stream);
    if (e != cudaSuccess) return cuda_fail(e, "gated RMS norm launch");
    return GDN_OK;
}

gdn_status gdn_decode_layer(const gdn_shape *shape, const gdn_layer_params *layer, const void *x,
                            const void *conv_weight, const void *conv_bias,
                            const void *conv_state_in, void *conv_state_out, const void *a,
                            const void *b, const float *A_log, const float *dt_bias, float *state,
                            float scale, const void *norm_scale, const void *gate, void *y,
                            void *stream) {
    gdn_status st = check_shape(shape, false);
    if (st != GDN_OK) return st;
    if (shape->seqlen != 1)
        return fail(GDN_ERR_INVALID_ARG, "decode takes seqlen 1 (got %lld)", (long long)shape->seqlen);
    if (shape->d_k != 128) return fail(GDN_ERR_UNSUPPORTED, "the layer step is built for d_k = 128");
    if (shape->d_v % 64 != 0)
        return fail(GDN_ERR_UNSUPPORTED, "the layer step needs d_v a multiple of 64 (got %d)", shape->d_v);
    if (layer == nullptr) return fail(GDN_ERR_INVALID_ARG, "layer is NULL");
    if (layer->conv_kernel < 1 || layer->conv_kernel > 8)
        return fail(GDN_ERR_INVALID_ARG, "conv_kernel %d is not in 1..8", layer->conv_kernel);
    if (layer->conv_activation != GDN_ACT_NONE && layer->conv_activation != GDN_ACT_SILU)
        return fail(GDN_ERR_INVALID_ARG, "the convolution's activation is NONE or SILU");
    if (layer->norm_activation != GDN_ACT_SILU && layer->norm_activation != GDN_ACT_SIGMOID)
        return fail(GDN_ERR_INVALID_ARG, "the norm's activation is SILU or SIGMOID");
    if (!(layer->norm_epsilon >= 0.0f) || isinf(layer->norm_epsilon))
        return fail(GDN_ERR_INVALID_ARG, "norm_epsilon must be finite and >= 0");
    if (!(scale == scale) || isinf(scale)) return fail(GDN_ERR_INVALID_ARG, "scale is not finite");
    if (shape->batch == 0) return GDN_OK;
    const void *need[] = {x, conv_weight, a, b, A_log, dt_bias, state, norm_scale, gate, y};
    const char *names[] = {"x", "conv_weight", "a", "b", "A_log", "dt_bias", "state", "norm_scale",
                           "gate", "y"};
    for (int i = 0; i < 10; ++i)
        if (need[i] == nullptr) return fail(GDN_ERR_INVALID_ARG, "%s is NULL", names[i]);
    const void *al16[] = {x, conv_weight, conv_bias, conv_state_in, conv_state_out, state, norm_scale, gate};
    for (const void *ptr : al16)
        if (ptr != nullptr && !aligned(ptr, 16))
            return fail(GDN_ERR_INVALID_ARG, "x, the conv tensors, state, norm_scale and gate must be 16-byte aligned");
    const size_t es = io_size(shape->io_dtype);
    if (!aligned(a, es) || !aligned(b, es) || !aligned(y, es) || !aligned(A_log, 4) || !aligned(dt_bias, 4))
        return fail(GDN_ERR_INVALID_ARG, "a, b, y, A_log or dt_bias is misaligned");
    const int64_t C = 2LL * shape->h_qk * shape->d_k + (int64_t)shape->h_v * shape->d_v;
    const size_t state_bytes = (size_t)shape->batch * (size_t)(layer->conv_kernel - 1) * (size_t)C * es;
    if (conv_state_in != nullptr && conv_state_out != nullptr && state_bytes > 0) {
        const uintptr_t i0 = reinterpret_cast<uintptr_t>(conv_state_in), o0 = reinterpret_cast<uintptr_t>(conv_state_out);
        if (i0 < o0 + state_bytes && o0 < i0 + state_bytes)
            return fail(GDN_ERR_INVALID_ARG, "conv_state_out overlaps conv_state_in (the update cannot be in place)");
    }
    int *word = nullptr;
    st = status_word(&word);
    if (st != GDN_OK) return st;
    LayerDecodeParams p{};
    p.x = x; p.conv_w = conv_weight; p.conv_b = conv_bias;
    p.conv_state_in = conv_state_in; p.conv_state_out = conv_state_out;
    p.a = a; p.b = b; p.A_log = A_log; p.dt_bias = dt_bias; p.state = state;
    p.norm_scale = norm_scale; p.gate = gate; p.y = y;
    p.batch = shape->batch; p.h_qk = shape->h_qk; p.h_v = shape->h_v; p.d_v = shape->d_v;
    p.conv_k = layer->conv_kernel;
    p.conv_silu = layer->conv_activation == GDN_ACT_SILU;
    p.norm_act = layer->norm_activation;
    p.scale = scale == 0.0f ? 1.0f / sqrtf((float)shape->d_k) : scale;
    p.eps = layer->norm_epsilon;
    cudaError_t e = launch_decode_layer(p, (gdn_dtype)shape->io_dtype, (cudaStream_t)stream);
    if (e != cudaSuccess) return cuda_fail(e, "layer decode launch");
    return GDN_OK;
}

gdn_status gdn_last_device_status(void *stream) {
    cudaError_t e = cudaStreamSynchronize((cudaStream_t)stream);
    if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
    int *word = nullptr;
    gdn_status st = status_word(&word);
    if (st != GDN_OK) return st;
    int value = 0;
    e = cudaMemcpy(&value, word, sizeof(int), cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return cuda_fail(e, "read check word");
    const int zero = 0;
    e = cudaMemcpy(word, &zero, sizeof(int), cudaMemcpyHostToDevice);
    if (e != cudaSuccess) return cuda_fail(e, "clear check word");
    if (value & kDevTimeout) return fail(GDN_ERR_TIMEOUT, "a device-side wait timed out");
    if (value & kDevBadCuSeqlens)
        return fail(GDN_ERR_DEVICE_CHECK, "cu_seqlens is malformed on the device");
    if (value & kDevBadSlot)
        return fail(GDN_ERR_DEVICE_CHECK, "a slot index is outside the state pool");
    return GDN_OK;
}

}  // extern "C"
