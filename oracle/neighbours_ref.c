/*
 * neighbours_ref.c -- CPU oracle for the two layer ops around the scan: the causal
 * depthwise convolution with a carried state that feeds q, k, v, and the gated RMS
 * norm applied to the scan's output.
 *
 * TEST INFRASTRUCTURE ONLY, like gdn_ref.c: plain sequential float64 loops, sharing
 * nothing with the CUDA library.
 *
 * Sources (the pages it restates):
 *  - onnxruntime-ep-mlx 0.31.1, src/ops/ssm.rs, `causal_conv_op` (CausalConvWithState):
 *    the past state (zeros when absent) is prepended to the input along time, giving
 *    carry = (K - 1) * dilation extra positions in front; every channel is convolved on
 *    its own with its K taps spaced `dilation` apart and no flip (a cross-correlation
 *    over the padded sequence, as MLX's conv1d computes it), so output t reads padded
 *    positions t + j * dilation, j = 0..K-1; the bias is added and then, optionally,
 *    silu(y) = y * sigmoid(y).  The present state is the last `carry` padded
 *    positions.  With state_window W > 0 the past state has a leading axis of W slabs
 *    of which only the last is used, and the present state holds, for each of the last
 *    min(L, W) tokens, the `carry` positions that end at that token, preceded by zero
 *    slabs when L < W; for L = 0 it is the past window (or zeros).  Layouts: channels
 *    last x [B, L, C] with state [B, carry, C], or channels first x [B, C, L] with state
 *    [B, C, carry]; the weight is [C, 1, K].
 *  - onnxruntime-ep-mlx 0.31.1, src/ops/ssm.rs, `gated_rms_norm_op` (GatedRMSNorm):
 *    rows of C consecutive values (C = the scale's width), y = x / sqrt(mean(x^2) + eps)
 *    * scale * act(gate) with act(g) = g * sigmoid(g) ("silu"/"swish") or sigmoid(g).
 *
 * Reading where the pages leave it open: everything is evaluated once in float64 from
 * the exact inputs (the pages evaluate in the I/O dtype or float32); the GPU evaluates
 * in float32 and rounds each output once.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

double gdn_ref_sigmoid(double x);   /* gdn_ref.c */

/* Strides of a [B, T, C] (channels last) or [B, C, T] (channels first) array. */
typedef struct {
    int64_t b, c, t;
} strides_t;

static strides_t layout(int32_t channels_last, int64_t C, int64_t T) {
    strides_t s;
    if (channels_last) {
        s.b = T * C; s.t = C; s.c = 1;
    } else {
        s.b = C * T; s.c = T; s.t = 1;
    }
    return s;
}

/*
 * y, state_out = CausalConvWithState(x, weight, bias, state_in).
 * state_in / state_out: [B, carry, C] or [B, C, carry]; with window W > 0 they carry a
 * leading axis of W slabs.  bias and state_in may be NULL.  Returns 0, or -1 on bad
 * arguments.
 */
int gdn_ref_causal_conv(int64_t B, int64_t L, int64_t C, int32_t K, int32_t dilation,
                        int32_t channels_last, int32_t silu, int32_t window, const double *x,
                        const double *w, const double *bias, const double *state_in,
                        double *y, double *state_out) {
    if (B < 0 || L < 0 || C <= 0 || K < 1 || dilation < 1 || window < 0 || window > 8 || !w)
        return -1;
    const int64_t carry = (int64_t)(K - 1) * dilation;
    const strides_t sx = layout(channels_last, C, L);
    const strides_t ss = layout(channels_last, C, carry);
    const int64_t slab = B * C * carry;   /* one state */
    /* The past state: slab W - 1 of a window. */
    const double *past = state_in;
    if (past && window > 0) past += (int64_t)(window - 1) * slab;
    double *xp = malloc(sizeof(double) * (size_t)(carry + L > 0 ? carry + L : 1));
    if (!xp) return -1;   /* the padded sequence of one channel */
    for (int64_t b = 0; b < B; ++b) {
        for (int64_t c = 0; c < C; ++c) {
            for (int64_t p = 0; p < carry; ++p)
                xp[p] = past ? past[b * ss.b + c * ss.c + p * ss.t] : 0.0;
            for (int64_t t = 0; t < L; ++t) xp[carry + t] = x[b * sx.b + c * sx.c + t * sx.t];
            for (int64_t t = 0; t < L; ++t) {
                double acc = 0.0;
                for (int32_t j = 0; j < K; ++j) acc += w[c * K + j] * xp[t + (int64_t)j * dilation];
                if (bias) acc += bias[c];
                if (silu) acc = acc * gdn_ref_sigmoid(acc);
                y[b * sx.b + c * sx.c + t * sx.t] = acc;
            }
            if (!state_out || carry == 0) continue;
            if (window == 0) {
                for (int64_t j = 0; j < carry; ++j)
                    state_out[b * ss.b + c * ss.c + j * ss.t] = xp[L + j];
                continue;
            }
            const int64_t kept = L < window ? L : window;
            for (int64_t s = 0; s < window; ++s) {
                double *dst = state_out + s * slab + b * ss.b + c * ss.c;
                if (L == 0) {
                    /* No token: the present window is the past one (zeros without it). */
                    for (int64_t j = 0; j < carry; ++j)
                        dst[j * ss.t] = state_in ? state_in[s * slab + b * ss.b + c * ss.c + j * ss.t]
                                                 : 0.0;
                } else if (s < window - kept) {
                    for (int64_t j = 0; j < carry; ++j) dst[j * ss.t] = 0.0;
                } else {
                    /* Slab s holds the carry positions that end at token L - window + s. */
                    const int64_t token = L - window + s;
                    for (int64_t j = 0; j < carry; ++j) dst[j * ss.t] = xp[token + 1 + j];
                }
            }
        }
    }
    free(xp);
    return 0;
}

/*
 * y = GatedRMSNorm(x, scale, gate): `rows` rows of `width` values each.
 * activation 1 = silu (g * sigmoid(g)), 2 = sigmoid.  Returns 0, or -1 on bad arguments.
 */
int gdn_ref_gated_rmsnorm(int64_t rows, int64_t width, const double *x, const double *scale,
                          const double *gate, double eps, int32_t activation, double *y) {
    if (rows < 0 || width <= 0 || (activation != 1 && activation != 2)) return -1;
    for (int64_t r = 0; r < rows; ++r) {
        const double *xr = x + r * width, *gr = gate + r * width;
        double ss = 0.0;
        for (int64_t i = 0; i < width; ++i) ss += xr[i] * xr[i];
        const double inv = 1.0 / sqrt(ss / (double)width + eps);
        for (int64_t i = 0; i < width; ++i) {
            const double s = gdn_ref_sigmoid(gr[i]);
            const double act = activation == 1 ? gr[i] * s : s;
            y[r * width + i] = xr[i] * inv * scale[i] * act;
        }
    }
    return 0;
}
