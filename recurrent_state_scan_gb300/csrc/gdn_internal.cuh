// gdn_internal.cuh -- definitions shared by libgdn's translation units.
//
// Gate math follows onnx-runtime-ep-cuda 0.1.0-dev.6, src/kernels/linear_attention.rs
// (`la_softplus`, `la_sigmoid`, the fused decay chain g = -exp(A_log) * softplus(a + dt_bias)),
// evaluated in fp32 once per token from widened inputs, with no intermediate
// re-rounding to the I/O dtype (the onnxruntime-ep-mlx ssm.rs gate op computes
// its gates wide and casts once; here g and beta are never stored at all).
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "gdn.h"

namespace gdn {

// Device check word values (OR-ed together by kernels that detect a problem).
enum : int { kDevOk = 0, kDevBadCuSeqlens = 1, kDevTimeout = 2, kDevBadSlot = 4 };

struct ScanParams {
    const void *q, *k, *v, *a, *b;
    const float *A_log, *dt_bias;
    const float *state_in;   // may be null (zeros); may alias state_out
    float *state_out;
    void *o;
    const int32_t *cu_seqlens;   // device, may be null
    int64_t seqlen;              // T per sequence, or packed total with cu_seqlens
    int32_t num_seqs, h_qk, h_v, d_k, d_v;
    float scale;
    int *status;                 // device check word
    const int32_t *slots;        // device, may be null: sequence n's state is pool entry slots[n]
    int64_t pool_size;           // entries of the state pool when slots is set
    float *window;               // may be null: [window_len, N, h_v, d_k, d_v], the states after
    int32_t window_len;          //   the last window_len steps (leading slabs zero when T is shorter)
    // Gate and rule variants (all zero: gated delta rule, one decay and one beta per head).
    int32_t rule;                // gdn_rule: 0 gated_delta, 1 delta, 2 gated, 3 linear
    int32_t decay_per_key;       // a [.., h_v, d_k], A_log / dt_bias [h_v, d_k]
    int32_t beta_shared;         // b [.., 1]: one beta for every head
    // Gated RMS norm of o fused into the tensor-core scan's readout (norm_gate set): o is
    // then written as y = o / rms(o) * norm_scale * act(gate) over each d_v row.
    const void *norm_scale, *norm_gate;
    float norm_eps;
    int32_t norm_silu;           // act = silu (1) or sigmoid (0)
    // The causal convolution of the layer's mixed input before the scan (conv_x set; the
    // tensor-core path only): q, k and v are then convolved inside the chunk prep.
    const void *conv_x, *conv_w, *conv_b, *conv_in;
    void *conv_out;
    int32_t conv_k, conv_silu;
    int32_t conv_fuse;           // 1: in the chunk prep; 0: a streaming pass writes q, k, v first
};

// ------------------------------------------------------------------ I/O types
template <typename T> struct IoType;
template <> struct IoType<float> {
    static __device__ __forceinline__ float ld(const float *p) { return *p; }
    static __device__ __forceinline__ void st(float *p, float x) { *p = x; }
};
template <> struct IoType<__nv_bfloat16> {
    static __device__ __forceinline__ float ld(const __nv_bfloat16 *p) { return __bfloat162float(*p); }
    static __device__ __forceinline__ void st(__nv_bfloat16 *p, float x) { *p = __float2bfloat16_rn(x); }
};
template <> struct IoType<__half> {
    static __device__ __forceinline__ float ld(const __half *p) { return __half2float(*p); }
    static __device__ __forceinline__ void st(__half *p, float x) { *p = __float2half_rn(x); }
};

// ------------------------------------------------------------------ gates
// softplus(x) = log(1 + e^x) written as max(x,0) + log1p(e^-|x|) (no overflow).
__device__ __forceinline__ float softplus_f(float x) {
    return fmaxf(x, 0.0f) + log1pf(expf(-fabsf(x)));
}
// sigmoid(x) = 1/(1+e^-x), split on the sign so the exponential never overflows.
__device__ __forceinline__ float sigmoid_f(float x) {
    if (x >= 0.0f) return 1.0f / (1.0f + expf(-x));
    const float e = expf(x);
    return e / (1.0f + e);
}
// Log-space decay g = -exp(A_log) * softplus(a + dt_bias).
__device__ __forceinline__ float decay_f(float a, float A_log, float dt_bias) {
    return -expf(A_log) * softplus_f(a + dt_bias);
}

// Token range [t0, t1) of sequence n; false (and the check word set) if the
// device-resident cu_seqlens entries for n are malformed.
__device__ __forceinline__ bool seq_range(const int32_t *cu_seqlens, int64_t seqlen,
                                          int32_t num_seqs, int *status, int64_t n, int64_t &t0,
                                          int64_t &t1) {
    if (cu_seqlens == nullptr) {
        t0 = n * seqlen;
        t1 = t0 + seqlen;
        return true;
    }
    t0 = cu_seqlens[n];
    t1 = cu_seqlens[n + 1];
    const bool ok = (t0 >= 0) && (t0 <= t1) && (t1 <= seqlen) && (n != 0 || t0 == 0) &&
                    (n + 1 != num_seqs || t1 == seqlen);
    if (!ok) atomicOr(status, kDevBadCuSeqlens);
    return ok;
}
__device__ __forceinline__ bool seq_range(const ScanParams &p, int64_t n, int64_t &t0,
                                          int64_t &t1) {
    return seq_range(p.cu_seqlens, p.seqlen, p.num_seqs, p.status, n, t0, t1);
}

// Launchers implemented in the kernel translation units.
cudaError_t launch_scan_simt(const ScanParams &p, gdn_dtype io, cudaStream_t stream);

// Causal depthwise convolution with a carried state (validated arguments).
struct ConvLaunch {
    gdn_dtype io;
    const void *x, *w, *bias, *state_in;
    void *y, *state_out;
    int64_t batch, seqlen;
    int32_t channels, kernel, dilation, channels_last, activation, window;
    const int32_t *slots;   // may be null
    int64_t pool_size;
    int *status;            // device check word
    bool vec4;              // channels last, C % 4 == 0 and every pointer 4-element aligned
    bool align16;           // x and state_in 16-byte aligned (shared-memory staging)
};
cudaError_t launch_causal_conv(const ConvLaunch &l, cudaStream_t stream);
cudaError_t launch_gated_rmsnorm(gdn_dtype io, int64_t rows, int32_t width, const void *x,
                                 const void *scale, const void *gate, float eps,
                                 int32_t activation, void *y, bool vec4, cudaStream_t stream);

// One decode step of the whole layer: causal conv -> gated delta-rule step -> gated RMS
// norm (validated arguments; d_k = 128, d_v a multiple of 64 up to 256).
struct LayerDecodeParams {
    const void *x, *conv_w, *conv_b, *conv_state_in;   // conv_b, conv_state_in may be null
    void *conv_state_out;                              // may be null; never overlaps the input
    const void *a, *b;
    const float *A_log, *dt_bias;
    float *state;                                      // [B, h_v, 128, d_v], in place
    const void *norm_scale, *gate;
    void *y;
    int32_t batch, h_qk, h_v, d_v;
    int32_t conv_k, conv_silu, norm_act;
    float scale, eps;
};
cudaError_t launch_decode_layer(const LayerDecodeParams &p, gdn_dtype io, cudaStream_t stream);

// Sets the calling thread's last error message; returns `status`.
gdn_status report_error(gdn_status status, const char *message);

// Chunked tensor-core prefill (bf16/f16 I/O, d_k = d_v = 128): a chunk-prep kernel
// that writes one workspace record per (chunk, value head), then a state-scan kernel.
// prefill_tc_shape_ok: the shape rules alone (host-only).  prefill_tc_workspace: bytes
// of records the call needs (packed sequences: an upper bound from the token total).
// prefill_tc_supported adds the pointer rules and the tensor-map encoder's presence.
bool prefill_tc_shape_ok(gdn_dtype io, int d_k, int d_v, int64_t total_tokens);
size_t prefill_tc_workspace(bool varlen, int64_t seqlen, int64_t batch, int64_t num_seqs, int h_v);
bool prefill_tc_supported(const ScanParams &p, gdn_dtype io, int64_t total_tokens);
// Chunk segments a call of this shape is split into (1: none).  Batched inputs whose scan
// grid leaves most of the GPU idle run the prep of later segments on an internal stream
// beside the scan of earlier ones; each segment costs one prep and one scan launch.
int prefill_tc_segments(bool varlen, int64_t seqlen, int64_t batch, int h_v);
// Bytes of chunk records a prefill of this shape needs on the tensor-core path (0 off it);
// the packed reading when batch is 1.
size_t prefill_records_bytes(const gdn_shape *shape);
// The same for a call that is packed (cu_seqlens given) or batched, as the dispatch reads it.
size_t prefill_records_bytes_for(const gdn_shape *shape, bool varlen);
// Time-parallel scan of batched shapes whose scan grid leaves most of the GPU idle: the
// segments it uses (1: none) and the workspace bytes it needs after the records (0: none).
int prefill_tc_tp_nseg(bool varlen, int64_t seqlen, int64_t batch, int h_v);
size_t prefill_tc_tp_bytes(bool varlen, int64_t seqlen, int64_t batch, int h_v);
// One decay per key dimension on the tensor-core path: the bytes of the Q~ and K~ arrays
// ([tokens][h_v][128] in a 16-bit type, each 1 KiB aligned) that follow the records.
size_t prefill_tc_pk_bytes(int64_t total_tokens, int h_v);
// With the convolution before the scan: the bytes of the convolved q and k arrays
// ([tokens][h_qk][128] in a 16-bit type, each 1 KiB aligned) that follow the records.
size_t prefill_tc_conv_bytes(int64_t total_tokens, int h_qk);
// The convolved v array ([tokens][h_v][128], 16-bit, 1 KiB aligned) that the streaming
// convolution pass adds after those.
size_t prefill_tc_conv_v_bytes(int64_t total_tokens, int h_v);
// workspace_bytes: the caller's workspace size; the time-parallel scan runs only when the
// workspace also holds its buffers (and allow_overlap is set).
cudaError_t launch_prefill_tc(const ScanParams &p, gdn_dtype io, int64_t total_tokens,
                              void *workspace, size_t workspace_bytes, bool allow_overlap,
                              cudaStream_t stream);

// Cycles a bounded wait of the tensor-core prefill kernels may take before the CTA gives
// up (0: about two seconds), set by gdn_set_wait_budget.
extern long long g_wait_budget;

// A TMA tensor map over a 3-D tensor of 16-bit values (dims innermost first, the two outer
// strides in bytes, multiples of 16), no swizzle, out-of-range elements read as zero.
// False when the driver's encoder is missing or rejects the arguments.
bool encode_map_3d(CUtensorMap *m, const void *base, gdn_dtype io, const uint64_t dims[3],
                   const uint64_t strides[2], const uint32_t box[3]);

// The gated RMS norm applied to o after the scan (gdn_prefill_norm).
// The causal convolution before the prefill (gdn_prefill_layer): x [tokens][C], C =
// 2 h_qk d_k + h_v d_v, read as [q | k | v]; weight [C][K], bias [C] or NULL, state in /
// out [sequences][K - 1][C] (in may be NULL: zeros).
struct ConvPrologue {
    const void *x, *weight, *bias, *state_in;
    void *state_out;
    int32_t kernel, silu;
    bool fuse;   // in the chunk prep (else a streaming pass before the prefill)
};

struct NormEpilogue {
    const void *scale;   // [d_v]
    const void *gate;    // like o
    float eps;
    int32_t activation;  // GDN_ACT_SILU or GDN_ACT_SIGMOID
    bool fuse;           // in the tensor-core scan's readout where the path allows
};

// gdn_prefill with the segment overlap allowed or not (no internal stream is created
// when it is not), optionally a gate / rule variant (per-key decay runs on the
// token-sequential kernel, everything else on the path gdn_prefill would take), and
// optionally the gated RMS norm of o (fused into the tensor-core scan's readout; after the
// scan, in place, on the other paths).
gdn_status prefill_impl(const gdn_shape *shape, const void *q, const void *k, const void *v,
                        const void *a, const void *b, const float *A_log, const float *dt_bias,
                        const float *state_in, const int32_t *cu_seqlens, float scale, void *o,
                        float *state_out, void *workspace, size_t workspace_bytes,
                        bool allow_overlap, void *stream, const gdn_variant *variant = nullptr,
                        const NormEpilogue *norm = nullptr, const ConvPrologue *conv = nullptr);

}  // namespace gdn
