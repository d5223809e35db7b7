// neighbours.cu -- the two layer ops around the scan, as HBM-bound CUDA kernels.
//
// Causal depthwise convolution with a carried state (onnxruntime-ep-mlx 0.31.1,
// src/ops/ssm.rs, `causal_conv_op`, the CausalConvWithState op; and nuvec-core 0.6.1,
// src/fast/imp.rs, `causal_conv1d_slots` for the state pool):
//  - padded position p of a row is the past state for p < carry = (K - 1) * dilation, and
//    input token p - carry after it; output t = act(bias + sum_j w[j] * pad[t + j * dil]),
//    with act = silu or none; the present state is pad[L .. L + carry).
//  - One thread owns VEC channels of one row over a tile of TT >= carry consecutive
//    tokens.  In the channels-last layout neighbouring threads own neighbouring channel
//    groups, so every load and store of a warp is one contiguous run.
//  - K <= 4 with dilation 1 (the shape the layer uses) keeps the last four padded
//    positions in registers and loads each input once; other shapes read their K taps
//    through L1.
//  - Only the tile-0 thread of a channel group reads the past state (TT >= carry), and
//    it writes the present state after all its reads, position by position in ascending
//    order.  So the present state may overwrite the past state in place, and a pool slot
//    is read and written by one thread.
//
// Gated RMS norm (onnxruntime-ep-mlx 0.31.1, src/ops/ssm.rs, `gated_rms_norm_op`): one
// warp per row of `width` values; y = x * rsqrt(mean(x^2) + eps) * scale * act(gate),
// act = silu or sigmoid, all in fp32, rounded once to the I/O dtype.
#include <type_traits>

#include "gdn_internal.cuh"
#include "tc_ptx.cuh"

namespace gdn {
namespace {

// VEC consecutive I/O values widened to fp32 (VEC = 4: one 8- or 16-byte access).
template <typename IO, int VEC> struct Vec {
    float v[VEC];
};

template <typename IO, int VEC>
__device__ __forceinline__ Vec<IO, VEC> ld_vec(const IO *p) {
    Vec<IO, VEC> r;
    if constexpr (VEC == 4 && sizeof(IO) == 2) {
        const uint2 raw = *reinterpret_cast<const uint2 *>(p);
        const IO *h = reinterpret_cast<const IO *>(&raw);
#pragma unroll
        for (int i = 0; i < 4; ++i) r.v[i] = IoType<IO>::ld(h + i);
    } else if constexpr (VEC == 4 && sizeof(IO) == 4) {
        const float4 f = *reinterpret_cast<const float4 *>(p);
        r.v[0] = f.x; r.v[1] = f.y; r.v[2] = f.z; r.v[3] = f.w;
    } else {
#pragma unroll
        for (int i = 0; i < VEC; ++i) r.v[i] = IoType<IO>::ld(p + i);
    }
    return r;
}

template <typename IO, int VEC>
__device__ __forceinline__ void st_vec(IO *p, const float (&x)[VEC]) {
    if constexpr (VEC == 4 && sizeof(IO) == 2) {
        uint2 raw;
        IO *h = reinterpret_cast<IO *>(&raw);
#pragma unroll
        for (int i = 0; i < 4; ++i) IoType<IO>::st(h + i, x[i]);
        *reinterpret_cast<uint2 *>(p) = raw;
    } else if constexpr (VEC == 4 && sizeof(IO) == 4) {
        *reinterpret_cast<float4 *>(p) = make_float4(x[0], x[1], x[2], x[3]);
    } else {
#pragma unroll
        for (int i = 0; i < VEC; ++i) IoType<IO>::st(p + i, x[i]);
    }
}

// Copy VEC raw values (the state is a copy of inputs: no rounding).
template <typename IO, int VEC>
__device__ __forceinline__ void copy_vec(IO *dst, const IO *src) {
    if constexpr (VEC == 4 && sizeof(IO) == 2) {
        *reinterpret_cast<uint2 *>(dst) = *reinterpret_cast<const uint2 *>(src);
    } else if constexpr (VEC == 4 && sizeof(IO) == 4) {
        *reinterpret_cast<float4 *>(dst) = *reinterpret_cast<const float4 *>(src);
    } else {
#pragma unroll
        for (int i = 0; i < VEC; ++i) dst[i] = src[i];
    }
}

template <typename IO, int VEC>
__device__ __forceinline__ void zero_vec(IO *dst) {
    float z[VEC];
#pragma unroll
    for (int i = 0; i < VEC; ++i) z[i] = 0.0f;
    st_vec<IO, VEC>(dst, z);
}

// The bits of VEC consecutive I/O values (one 8- or 16-byte access when VEC = 4).
template <typename IO, int VEC> struct alignas(sizeof(IO) * VEC) Raw {
    IO v[VEC];
};


// sigmoid and silu from the fast exponential and divide intrinsics (a few ulp; for very
// negative x the exponential overflows to inf and the quotient is 0, the right limit).
__device__ __forceinline__ float sigmoid_fast(float x) {
    return __fdividef(1.0f, 1.0f + __expf(-x));
}
__device__ __forceinline__ float silu_fast(float x) { return __fdividef(x, 1.0f + __expf(-x)); }

// Tokens a thread of the register-tiled convolution covers.
constexpr int kShortTile = 8;

struct ConvParams {
    const void *x, *w, *bias, *state_in;
    void *y, *state_out;
    int64_t B, L;
    int32_t C, K, dil, carry;
    int32_t channels_last, silu, window;
    const int32_t *slots;    // may be null: row b's state is pool entry slots[b]
    int64_t pool_size;
    int64_t tt, tiles;       // tokens per thread (>= carry) and tiles per row
    int *status;
};

// Element offsets of (row b, channel c, position t) in an array of T positions.
__device__ __forceinline__ int64_t at(const ConvParams &p, int64_t b, int64_t c, int64_t t,
                                      int64_t T) {
    return p.channels_last ? (b * T + t) * p.C + c : (b * p.C + c) * T + t;
}

// Any kernel size and dilation: each output reads its K taps (the re-reads hit L1).
template <typename IO, int VEC>
__global__ void __launch_bounds__(256) causal_conv_kernel(const ConvParams p) {
    const IO *x = static_cast<const IO *>(p.x);
    const IO *w = static_cast<const IO *>(p.w);
    const IO *bias = static_cast<const IO *>(p.bias);
    const IO *sin = static_cast<const IO *>(p.state_in);
    IO *y = static_cast<IO *>(p.y);
    IO *sout = static_cast<IO *>(p.state_out);
    const int64_t groups = p.C / VEC;
    const int64_t total = p.B * p.tiles * groups;
    const int64_t slab = (p.slots ? p.pool_size : p.B) * (int64_t)p.C * p.carry;

    for (int64_t idx = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; idx < total;
         idx += (int64_t)gridDim.x * blockDim.x) {
        // Channels last: the channel group varies fastest (coalesced along C);
        // channels first: the tile varies fastest.
        int64_t b, tile, g;
        if (p.channels_last) {
            g = idx % groups;
            tile = (idx / groups) % p.tiles;
            b = idx / (groups * p.tiles);
        } else {
            tile = idx % p.tiles;
            g = (idx / p.tiles) % groups;
            b = idx / (p.tiles * groups);
        }
        const int64_t c0 = g * VEC;
        int64_t srow = b;
        if (p.slots != nullptr) {
            srow = p.slots[b];
            if (srow < 0 || srow >= p.pool_size) {
                if (tile == 0 && g == 0) atomicOr(p.status, kDevBadSlot);
                continue;
            }
        }
        // The past state: the last slab of a window.
        const IO *past = sin;
        if (past != nullptr && p.window > 0) past += (int64_t)(p.window - 1) * slab;
        // Padded position q of this thread's channels.
        auto load = [&](int64_t q) -> Vec<IO, VEC> {
            Vec<IO, VEC> r;
            if (q < 0 || (q < p.carry && past == nullptr)) {
#pragma unroll
                for (int i = 0; i < VEC; ++i) r.v[i] = 0.0f;
                return r;
            }
            if (q < p.carry) return ld_vec<IO, VEC>(past + at(p, srow, c0, q, p.carry));
            return ld_vec<IO, VEC>(x + at(p, b, c0, q - p.carry, p.L));
        };

        float bv[VEC];
#pragma unroll
        for (int i = 0; i < VEC; ++i) bv[i] = bias ? IoType<IO>::ld(bias + c0 + i) : 0.0f;
        const int64_t t0 = tile * p.tt;
        const int64_t t1 = p.L < t0 + p.tt ? p.L : t0 + p.tt;

        {
            for (int64_t t = t0; t < t1; ++t) {
                float acc[VEC];
#pragma unroll
                for (int i = 0; i < VEC; ++i) acc[i] = 0.0f;
                for (int j = 0; j < p.K; ++j) {
                    const Vec<IO, VEC> r = load(t + (int64_t)j * p.dil);
#pragma unroll
                    for (int i = 0; i < VEC; ++i)
                        acc[i] = fmaf(IoType<IO>::ld(w + (c0 + i) * p.K + j), r.v[i], acc[i]);
                }
                float out[VEC];
#pragma unroll
                for (int i = 0; i < VEC; ++i) {
                    const float s = acc[i] + bv[i];
                    out[i] = p.silu ? silu_fast(s) : s;
                }
                st_vec<IO, VEC>(y + at(p, b, c0, t, p.L), out);
            }
        }

        // The present state, written by the tile-0 thread after all of its reads.
        if (tile != 0 || sout == nullptr || p.carry == 0) continue;
        // Raw copy of padded position q into dst (zeros before the first position).
        auto put = [&](IO *dst, int64_t q) {
            if (q < p.carry) {
                if (past == nullptr) zero_vec<IO, VEC>(dst);
                else copy_vec<IO, VEC>(dst, past + at(p, srow, c0, q, p.carry));
            } else {
                copy_vec<IO, VEC>(dst, x + at(p, b, c0, q - p.carry, p.L));
            }
        };
        if (p.window == 0) {
            for (int64_t j = 0; j < p.carry; ++j) put(sout + at(p, srow, c0, j, p.carry), p.L + j);
            continue;
        }
        const int64_t kept = p.L < p.window ? p.L : (int64_t)p.window;
        for (int64_t s = 0; s < p.window; ++s) {
            IO *dst = sout + s * slab;
            for (int64_t j = 0; j < p.carry; ++j) {
                IO *d = dst + at(p, srow, c0, j, p.carry);
                if (p.L == 0) {
                    // No token: the present window is the past window (zeros without one).
                    if (sin == nullptr) zero_vec<IO, VEC>(d);
                    else copy_vec<IO, VEC>(d, sin + s * slab + at(p, srow, c0, j, p.carry));
                } else if (s < p.window - kept) {
                    zero_vec<IO, VEC>(d);
                } else {
                    put(d, p.L - p.window + s + 1 + j);
                }
            }
        }
    }
}

// K <= 4 taps at dilation 1 (carry <= 3), the shape the layer uses.  Grid: x over
// blocks of channel groups, y over (row, tile) pairs.  A thread loads the TT + 3 padded
// positions its TT outputs read (widened to fp32 once), its weights (one vector load per
// channel when K = 4), and -- tile 0, no window -- the carry positions of the present
// state, all before it stores anything; then it computes from registers.  A window is
// written slab by slab after the outputs: the only past slab read is the last one, which
// is also written last, and within a slab position j + L is read before position j is
// written, so the window may overwrite the past window in place.
template <typename IO, int VEC, int TT>
__global__ void __launch_bounds__(256, (TT == 1 ? 4 : 3)) causal_conv_short_kernel(const ConvParams p) {
    constexpr int NW = TT + 3;          // padded positions a tile reads: t0 + carry - 3 ..
    using R = Raw<IO, VEC>;
    const IO *x = static_cast<const IO *>(p.x);
    const IO *w = static_cast<const IO *>(p.w);
    const IO *bias = static_cast<const IO *>(p.bias);
    const IO *sin = static_cast<const IO *>(p.state_in);
    IO *y = static_cast<IO *>(p.y);
    IO *sout = static_cast<IO *>(p.state_out);
    const int64_t g = blockIdx.x * (int64_t)blockDim.x + threadIdx.x;   // channel group
    if (g >= p.C / VEC) return;
    const int64_t c0 = g * VEC;
    const int64_t slab = (p.slots ? p.pool_size : p.B) * (int64_t)p.C * p.carry;

    // Weights: w4[3 - m] = w[K - 1 - m] (four taps ending at the newest position), bias.
    float w4[4][VEC], bv[VEC];
#pragma unroll
    for (int i = 0; i < VEC; ++i) {
        if (VEC == 4 && p.K == 4) {   // VEC = 4: the weight is 4-element aligned
            const Vec<IO, 4> v = ld_vec<IO, 4>(w + (c0 + i) * 4);
#pragma unroll
            for (int m = 0; m < 4; ++m) w4[m][i] = v.v[m];
        } else {
#pragma unroll
            for (int m = 0; m < 4; ++m)
                w4[3 - m][i] = m < p.K ? IoType<IO>::ld(w + (c0 + i) * p.K + (p.K - 1 - m)) : 0.0f;
        }
    }
    if (bias != nullptr) {
        const Vec<IO, VEC> v = ld_vec<IO, VEC>(bias + c0);
#pragma unroll
        for (int i = 0; i < VEC; ++i) bv[i] = v.v[i];
    } else {
#pragma unroll
        for (int i = 0; i < VEC; ++i) bv[i] = 0.0f;
    }

    for (int64_t bt = blockIdx.y; bt < p.B * p.tiles; bt += gridDim.y) {
        const int64_t b = bt / p.tiles;
        const int64_t tile = bt - b * p.tiles;
        int64_t srow = b;
        if (p.slots != nullptr) {
            srow = p.slots[b];
            if (srow < 0 || srow >= p.pool_size) {
                if (tile == 0 && g == 0) atomicOr(p.status, kDevBadSlot);
                continue;
            }
        }
        const IO *past = sin;
        if (past != nullptr && p.window > 0) past += (int64_t)(p.window - 1) * slab;
        // Padded position q of this thread's channels (null: zeros).
        auto src = [&](int64_t q) -> const IO * {
            if (q < 0 || q >= p.L + p.carry) return nullptr;
            if (q >= p.carry) return x + (b * p.L + (q - p.carry)) * p.C + c0;
            return past == nullptr ? nullptr : past + (srow * p.carry + q) * p.C + c0;
        };
        const int64_t t0 = tile * TT;
        const int64_t base = t0 + p.carry - 3;           // padded position of win[0]
        float win[NW][VEC];
#pragma unroll
        for (int k = 0; k < NW; ++k) {
            const IO *a = src(base + k);
            Vec<IO, VEC> v;
#pragma unroll
            for (int i = 0; i < VEC; ++i) v.v[i] = 0.0f;
            if (a != nullptr) v = ld_vec<IO, VEC>(a);
#pragma unroll
            for (int i = 0; i < VEC; ++i) win[k][i] = v.v[i];
        }
        // The present state without a window: positions L .. L + carry - 1, read now.
        const bool single = tile == 0 && sout != nullptr && p.window == 0 && p.carry > 0;
        R keep[3];
        if (single) {
#pragma unroll
            for (int j = 0; j < 3; ++j) {
                const IO *a = j < p.carry ? src(p.L + j) : nullptr;
                if (a != nullptr) {
                    keep[j] = *reinterpret_cast<const R *>(a);
                } else {
#pragma unroll
                    for (int i = 0; i < VEC; ++i) IoType<IO>::st(&keep[j].v[i], 0.0f);
                }
            }
        }
#pragma unroll
        for (int k = 0; k < TT; ++k) {
            if (t0 + k >= p.L) break;
            float out[VEC];
#pragma unroll
            for (int i = 0; i < VEC; ++i) {
                // Oldest tap first; positions before the K taps are never touched, so a
                // non-finite value there cannot leak in through a zero weight.
                float acc = 0.0f;
                if (p.K > 3) acc = fmaf(w4[0][i], win[k][i], acc);
                if (p.K > 2) acc = fmaf(w4[1][i], win[k + 1][i], acc);
                if (p.K > 1) acc = fmaf(w4[2][i], win[k + 2][i], acc);
                acc = fmaf(w4[3][i], win[k + 3][i], acc);
                acc += bv[i];
                out[i] = p.silu ? silu_fast(acc) : acc;
            }
            st_vec<IO, VEC>(y + (b * p.L + t0 + k) * p.C + c0, out);
        }
        if (single) {
#pragma unroll
            for (int j = 0; j < 3; ++j)
                if (j < p.carry)
                    *reinterpret_cast<R *>(sout + (srow * p.carry + j) * p.C + c0) = keep[j];
            continue;
        }
        if (tile != 0 || sout == nullptr || p.carry == 0) continue;
        // The window: slab s holds positions L - W + s + 1 + j (j < carry), zero slabs
        // first when L < W, and the past window itself when L = 0.
        const int64_t kept = p.L < p.window ? p.L : (int64_t)p.window;
        for (int64_t s = 0; s < p.window; ++s)
            for (int64_t j = 0; j < p.carry; ++j) {
                IO *d = sout + s * slab + (srow * p.carry + j) * p.C + c0;
                if (p.L == 0) {
                    if (sin == nullptr) zero_vec<IO, VEC>(d);
                    else copy_vec<IO, VEC>(d, sin + s * slab + (srow * p.carry + j) * p.C + c0);
                } else if (s < p.window - kept) {
                    zero_vec<IO, VEC>(d);
                } else {
                    const IO *a = src(p.L - p.window + s + 1 + j);
                    if (a == nullptr) zero_vec<IO, VEC>(d);
                    else copy_vec<IO, VEC>(d, a);
                }
            }
    }
}

// Long rows (L >= kStagedMinTokens), channels last, K <= 4 at dilation 1, no window,
// C % 8 == 0: a CTA owns kStagedWidth channels of one row over kStagedChunk tokens and
// streams them through shared memory in stages of kStagedTokens (+3 halo) rows, three
// stages deep, with 16-byte cp.async copies, so the copies of the next two stages are in
// flight while a stage is computed.  Thread (cg, tg) computes 4 channels x 8 tokens of a
// stage from shared memory and stores them straight to y.  Only the chunk-0 CTA reads the
// past state (its first stage), and it writes the present state after its last stage.
constexpr int kStagedWidth = 256;      // channels per CTA
constexpr int kStagedTokens = 32;      // tokens per stage
constexpr int kStagedChunk = 256;      // tokens per CTA
constexpr int kStagedDepth = 3;        // stages in flight
constexpr int kStagedMinTokens = 64;

__device__ __forceinline__ void stream_commit_conv() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
template <int N> __device__ __forceinline__ void stream_wait_conv() {
    asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory");
}

__device__ __forceinline__ void cp_async16(void *smem, const void *gmem) {
    const unsigned s = static_cast<unsigned>(__cvta_generic_to_shared(smem));
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(s), "l"(gmem) : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
    asm volatile("cp.async.commit_group;\n" ::: "memory");
}
template <int N> __device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory");
}

template <typename IO>
__global__ void __launch_bounds__(256, 3) causal_conv_staged_kernel(const ConvParams p) {
    constexpr int ROWS = kStagedTokens + 3;
    constexpr int ROWB = kStagedWidth * (int)sizeof(IO);     // bytes of a row segment
    constexpr int SEGS = ROWB / 16;                          // 16-byte copies per row
    constexpr int EPS = 16 / (int)sizeof(IO);                // elements per copy
    extern __shared__ __align__(16) unsigned char smem[];    // kStagedDepth x ROWS x ROWB
    const IO *x = static_cast<const IO *>(p.x);
    const IO *w = static_cast<const IO *>(p.w);
    const IO *bias = static_cast<const IO *>(p.bias);
    const IO *past = static_cast<const IO *>(p.state_in);
    IO *y = static_cast<IO *>(p.y);
    IO *sout = static_cast<IO *>(p.state_out);
    const int tid = threadIdx.x;
    const int64_t cbase = (int64_t)blockIdx.x * kStagedWidth;
    const int64_t chunk = blockIdx.y;
    const int64_t b = blockIdx.z;
    int64_t srow = b;
    if (p.slots != nullptr) {
        srow = p.slots[b];
        if (srow < 0 || srow >= p.pool_size) {
            if (chunk == 0 && blockIdx.x == 0 && tid == 0) atomicOr(p.status, kDevBadSlot);
            return;
        }
    }
    const int64_t t_begin = chunk * kStagedChunk;
    const int64_t t_end = t_begin + kStagedChunk < p.L ? t_begin + kStagedChunk : p.L;
    const int nstage = (int)((t_end - t_begin + kStagedTokens - 1) / kStagedTokens);

    // Source of padded position q, channels c .. c + EPS - 1 (null: zeros).
    auto src = [&](int64_t q, int64_t c) -> const IO * {
        if (q < 0 || q >= p.L + p.carry) return nullptr;
        if (q >= p.carry) return x + (b * p.L + (q - p.carry)) * p.C + c;
        return past == nullptr ? nullptr : past + (srow * p.carry + q) * p.C + c;
    };
    auto load_stage = [&](int st) {
        unsigned char *buf = smem + (st % kStagedDepth) * (ROWS * ROWB);
        const int64_t q0 = t_begin + (int64_t)st * kStagedTokens + p.carry - 3;
        for (int i = tid; i < ROWS * SEGS; i += blockDim.x) {
            const int r = i / SEGS, sg = i % SEGS;
            const int64_t c = cbase + (int64_t)sg * EPS;
            if (c >= p.C) continue;
            const IO *a = src(q0 + r, c);
            void *d = buf + r * ROWB + sg * 16;
            if (a != nullptr) cp_async16(d, a);
            else *reinterpret_cast<uint4 *>(d) = make_uint4(0u, 0u, 0u, 0u);
        }
    };

    // Compute role: 4 channels (cg) x 8 tokens (tg) of a stage.
    const int cg = tid % 64, tg = tid / 64;
    const int64_t c0 = cbase + cg * 4;
    const bool live = c0 < p.C;
    float w4[4][4], bv[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        bv[i] = 0.0f;
#pragma unroll
        for (int m = 0; m < 4; ++m) w4[m][i] = 0.0f;
    }
    if (live) {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
#pragma unroll
            for (int m = 0; m < 4; ++m)
                w4[3 - m][i] = m < p.K ? IoType<IO>::ld(w + (c0 + i) * p.K + (p.K - 1 - m)) : 0.0f;
            bv[i] = bias ? IoType<IO>::ld(bias + c0 + i) : 0.0f;
        }
    }

#pragma unroll
    for (int st = 0; st < kStagedDepth - 1; ++st) {
        if (st < nstage) load_stage(st);
        cp_async_commit();
    }
    for (int st = 0; st < nstage; ++st) {
        if (st + kStagedDepth - 1 < nstage) load_stage(st + kStagedDepth - 1);
        cp_async_commit();
        cp_async_wait<kStagedDepth - 1>();
        __syncthreads();
        const unsigned char *buf = smem + (st % kStagedDepth) * (ROWS * ROWB);
        const int64_t ts = t_begin + (int64_t)st * kStagedTokens + tg * 8;   // first token
        if (live) {
            float win[11][4];
#pragma unroll
            for (int k = 0; k < 11; ++k) {
                const Vec<IO, 4> v =
                    ld_vec<IO, 4>(reinterpret_cast<const IO *>(buf + (tg * 8 + k) * ROWB) + cg * 4);
#pragma unroll
                for (int i = 0; i < 4; ++i) win[k][i] = v.v[i];
            }
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                if (ts + k >= t_end) break;
                float out[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    float acc = 0.0f;
                    if (p.K > 3) acc = fmaf(w4[0][i], win[k][i], acc);
                    if (p.K > 2) acc = fmaf(w4[1][i], win[k + 1][i], acc);
                    if (p.K > 1) acc = fmaf(w4[2][i], win[k + 2][i], acc);
                    acc = fmaf(w4[3][i], win[k + 3][i], acc);
                    acc += bv[i];
                    out[i] = p.silu ? silu_fast(acc) : acc;
                }
                st_vec<IO, 4>(y + (b * p.L + ts + k) * p.C + c0, out);
            }
        }
        __syncthreads();   // the buffer is refilled by a later stage's copies
    }
    cp_async_wait<0>();

    // The present state: positions L .. L + carry - 1, one copy per 4 channels.
    if (chunk != 0 || sout == nullptr || !live || tg != 0) return;
    for (int64_t j = 0; j < p.carry; ++j) {
        const IO *a = src(p.L + j, c0);
        IO *d = sout + (srow * p.carry + j) * p.C + c0;
        if (a == nullptr) zero_vec<IO, 4>(d);
        else copy_vec<IO, 4>(d, a);
    }
}

// Long rows of 16-bit values on the staged kernel's shapes, with the copies and the
// arithmetic cut down to what the bytes need.  A CTA owns kStagedWidth channels of one
// row over kStagedChunk tokens, in stages of kStagedTokens + 3 rows (tokens t - 3 ..
// t + 31 of the stage starting at t), kTmaDepth stages deep.
//  - Warp 0 brings a stage in with one TMA tensor copy (a 256-channel x 35-token box of x;
//    tokens past the row read as zero) counted on the stage's `full` barrier.  The first
//    stage of a row's first chunk copies tokens 0 .. 31 and its lanes write the three rows
//    before them from the past state (or zeros) themselves; every lane of warp 0 arrives
//    on `full`, so those stores are seen by whoever waits on it.
//  - Each warp computes from a stage once `full` completes and then arrives on the
//    stage's `empty` barrier; warp 0 refills a buffer once all eight warps have released
//    it.  No CTA-wide barrier runs per stage.
//  - Thread (cg, tg) computes 8 channels x 4 tokens: one 16-byte shared-memory load per
//    window row and one 16-byte store per token, so a warp's store is a whole 512-byte
//    row.  The taps (K = KT) and the activation are compile-time.  The sum is the staged
//    kernel's: fp32, oldest tap first, then the bias, rounded once.
//  - Every wait is bounded; a wait that runs out stops the CTA, whose warp 0 first lets
//    the copies it issued land.
constexpr int kTmaDepth = 4;
constexpr int kTmaRows = kStagedTokens + 3;
// Cycles (about two seconds) a wait may take by default, and always when a CTA that gave
// up lets its own copies land.
constexpr long long kConvDrainBudget = 4000000000LL;

// Wait for phase `parity` of `bar` for at most `budget` cycles (or until `abort` is set),
// polling with a short sleep: a blocking try_wait could hold the thread past the budget.
__device__ __forceinline__ bool conv_wait(uint64_t *bar, uint32_t parity, long long budget,
                                          volatile int *abort) {
    const uint32_t addr = tc::smem_u32(bar);
    const long long t0 = clock64();
    for (;;) {
        uint32_t done;
        asm volatile(
            "{\n\t.reg .pred p;\n\t"
            "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
            "selp.u32 %0, 1, 0, p;\n\t}"
            : "=r"(done)
            : "r"(addr), "r"(parity)
            : "memory");
        if (done) return true;
        if ((abort != nullptr && *abort) || clock64() - t0 > budget) return false;
        __nanosleep(32);
    }
}

struct ConvTmaMaps {
    CUtensorMap stage;   // box 256 channels x 35 tokens x 1 row of x [B][L][C]
    CUtensorMap first;   // box 256 x 32 x 1: a row's first stage, after the past rows
};

template <typename IO, int KT, bool SILU>
__global__ void __launch_bounds__(256, 2)
causal_conv_tma_kernel(const ConvParams p, const __grid_constant__ ConvTmaMaps maps, long long budget) {
    static_assert(sizeof(IO) == 2, "16-bit I/O");
    constexpr int ROWB = kStagedWidth * 2;
    constexpr int BUFB = kTmaRows * ROWB;
    extern __shared__ unsigned char smem_raw[];   // kTmaDepth x kTmaRows x ROWB, + 128
    unsigned char *smem = reinterpret_cast<unsigned char *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 127) & ~static_cast<uintptr_t>(127));
    __shared__ uint64_t full[kTmaDepth], empty[kTmaDepth];
    __shared__ int abort_flag;
    volatile int *abort = &abort_flag;
    const IO *x = static_cast<const IO *>(p.x);
    const IO *w = static_cast<const IO *>(p.w);
    const IO *bias = static_cast<const IO *>(p.bias);
    const IO *past = static_cast<const IO *>(p.state_in);
    IO *y = static_cast<IO *>(p.y);
    IO *sout = static_cast<IO *>(p.state_out);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int64_t cbase = (int64_t)blockIdx.x * kStagedWidth;
    const int64_t chunk = blockIdx.y;
    const int64_t b = blockIdx.z;
    int64_t srow = b;
    if (p.slots != nullptr) {
        srow = p.slots[b];
        if (srow < 0 || srow >= p.pool_size) {
            if (chunk == 0 && blockIdx.x == 0 && tid == 0) atomicOr(p.status, kDevBadSlot);
            return;
        }
    }
    const int64_t t_begin = chunk * kStagedChunk;
    const int64_t t_end = t_begin + kStagedChunk < p.L ? t_begin + kStagedChunk : p.L;
    const int nstage = (int)((t_end - t_begin + kStagedTokens - 1) / kStagedTokens);
    const int width = p.C - cbase < kStagedWidth ? (int)(p.C - cbase) : kStagedWidth;

    if (tid == 0) {
#pragma unroll
        for (int i = 0; i < kTmaDepth; ++i) {
            tc::mbar_init(&full[i], 32);    // every lane of warp 0
            tc::mbar_init(&empty[i], 8);    // one arrival per warp
        }
        tc::fence_mbar_init();
        abort_flag = 0;
    }
    __syncthreads();

    // Warp 0: stage st into its buffer (after its previous use has been released).
    auto issue = [&](int st) -> bool {
        const int i = st % kTmaDepth;
        if (st >= kTmaDepth &&
            !conv_wait(&empty[i], (uint32_t)(st / kTmaDepth - 1) & 1u, budget, abort))
            return false;
        unsigned char *buf = smem + i * BUFB;
        const int64_t ts = t_begin + (int64_t)st * kStagedTokens;   // first token of the stage
        const bool first = ts == 0;
        if (first && lane < 3) {
            // Rows 0..2: tokens -3..-1, i.e. padded positions q = lane + carry - 3.
            const int64_t q = lane + p.carry - 3;
            const IO *src = (q >= 0 && past != nullptr) ? past + (srow * p.carry + q) * p.C + cbase : nullptr;
            for (int o = 0; o < width * 2; o += 16)
                *reinterpret_cast<uint4 *>(buf + lane * ROWB + o) =
                    src ? *reinterpret_cast<const uint4 *>(reinterpret_cast<const unsigned char *>(src) + o)
                        : make_uint4(0u, 0u, 0u, 0u);
            tc::fence_async_smem();   // before later tensor copies into the same rows
        }
        if (lane == 0) {
            tc::mbar_arrive_expect_tx(&full[i], first ? kStagedTokens * ROWB : BUFB);
            if (first)
                tc::tma_load_3d(buf + 3 * ROWB, &maps.first, (int)cbase, 0, (int)b, &full[i]);
            else
                tc::tma_load_3d(buf, &maps.stage, (int)cbase, (int)(ts - 3), (int)b, &full[i]);
        } else {
            tc::mbar_arrive(&full[i]);
        }
        return true;
    };

    const int cg = tid & 31, tg = tid >> 5;
    const int64_t c0 = cbase + cg * 8;
    const bool live = cg * 8 < width;
    float wv[KT][8], bv[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        bv[i] = 0.0f;
#pragma unroll
        for (int m = 0; m < KT; ++m) wv[m][i] = 0.0f;
    }
    if (live) {
#pragma unroll
        for (int i = 0; i < 8; ++i) {
#pragma unroll
            for (int m = 0; m < KT; ++m) wv[m][i] = IoType<IO>::ld(w + (c0 + i) * KT + m);
            if (bias != nullptr) bv[i] = IoType<IO>::ld(bias + c0 + i);
        }
    }

    int issued = 0;   // warp 0: stages issued so far
    bool ok = true;
    if (warp == 0) {
        if (lane == 0) tc::tma_prefetch_desc(&maps.stage);
        for (; issued < kTmaDepth - 1 && issued < nstage; ++issued) issue(issued);
    }
    for (int st = 0; ok && st < nstage; ++st) {
        if (warp == 0 && issued < nstage) {
            if (!issue(issued)) ok = false;
            else ++issued;
        }
        if (ok && !conv_wait(&full[st % kTmaDepth], (uint32_t)(st / kTmaDepth) & 1u, budget, abort))
            ok = false;
        if (!ok) break;
        const unsigned char *buf = smem + (st % kTmaDepth) * BUFB;
        const int j0 = tg * 4;
        const int64_t t0 = t_begin + (int64_t)st * kStagedTokens + j0;
        if (live && t0 < t_end) {
            // Output j0 + k reads rows j0 + k + m + 4 - KT, m < KT.
            float win[KT + 3][8];
#pragma unroll
            for (int r = 0; r < KT + 3; ++r) {
                const uint4 raw =
                    *reinterpret_cast<const uint4 *>(buf + (j0 + r + 4 - KT) * ROWB + cg * 16);
                const IO *h = reinterpret_cast<const IO *>(&raw);
#pragma unroll
                for (int i = 0; i < 8; ++i) win[r][i] = IoType<IO>::ld(h + i);
            }
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                uint4 raw;
                IO *h = reinterpret_cast<IO *>(&raw);
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    float acc = wv[0][i] * win[k][i];
#pragma unroll
                    for (int m = 1; m < KT; ++m) acc = fmaf(wv[m][i], win[k + m][i], acc);
                    acc += bv[i];
                    IoType<IO>::st(h + i, SILU ? silu_fast(acc) : acc);
                }
                if (t0 + k < t_end)
                    *reinterpret_cast<uint4 *>(y + (b * p.L + t0 + k) * p.C + c0) = raw;
            }
        }
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(&empty[st % kTmaDepth]);
    }
    if (!ok) {
        *abort = 1;
        if (tid == 0) atomicOr(p.status, kDevTimeout);
        if (warp == 0) {
            // Let the copies this CTA issued land before it exits: the latest phase of each
            // buffer's `full` barrier.
            for (int s2 = issued - kTmaDepth < 0 ? 0 : issued - kTmaDepth; s2 < issued; ++s2)
                conv_wait(&full[s2 % kTmaDepth], (uint32_t)(s2 / kTmaDepth) & 1u, kConvDrainBudget, nullptr);
        }
        return;
    }

    // The present state: positions L .. L + carry - 1, 8 channels a thread (warp 0 of the
    // row's first chunk, after its own reads of the past state).
    if (chunk != 0 || sout == nullptr || !live || tg != 0) return;
    for (int64_t j = 0; j < p.carry; ++j) {
        const int64_t q = p.L + j;   // padded position
        const IO *a = q >= p.carry ? x + (b * p.L + (q - p.carry)) * p.C + c0
                                   : (past == nullptr ? nullptr : past + (srow * p.carry + q) * p.C + c0);
        uint4 *d = reinterpret_cast<uint4 *>(sout + (srow * p.carry + j) * p.C + c0);
        *d = a == nullptr ? make_uint4(0u, 0u, 0u, 0u) : *reinterpret_cast<const uint4 *>(a);
    }
}

// The decode step (L = 1, K <= 4 at dilation 1, channels last, no window, 16-bit I/O,
// four channels a thread): persistent CTAs walk (row, 1024-channel slab) items.  Each
// thread streams the next item's carry + 1 positions, its taps and its bias into its own
// slots of a double-buffered shared-memory tile with 8-byte cp.async copies, then
// computes the current item from the other buffer, so its copies are always in flight.
// No slot is shared between threads, so cp.async.wait_group alone orders the reads.
// Item i + stride never shares a row and slab with item i (distinct slots), so its early
// reads cannot see this item's state write.
__device__ __forceinline__ void cp_async8(void *smem, const void *gmem) {
    const unsigned s = static_cast<unsigned>(__cvta_generic_to_shared(smem));
    asm volatile("cp.async.ca.shared.global [%0], [%1], 8;\n" ::"r"(s), "l"(gmem) : "memory");
}

template <typename IO>
__global__ void __launch_bounds__(256) causal_conv_decode_stream_kernel(const ConvParams p) {
    static_assert(sizeof(IO) == 2, "16-bit I/O");
    constexpr int kSlots = 9;   // positions 0..3, taps 0..3, bias
    __shared__ __align__(16) uint2 buf[2][kSlots][256];
    const IO *x = static_cast<const IO *>(p.x);
    const IO *w = static_cast<const IO *>(p.w);
    const IO *bias = static_cast<const IO *>(p.bias);
    const IO *past = static_cast<const IO *>(p.state_in);
    IO *y = static_cast<IO *>(p.y);
    IO *sout = static_cast<IO *>(p.state_out);
    const int tid = threadIdx.x;
    const int64_t nslab = (p.C + 1023) / 1024;
    const int64_t items = p.B * nslab;

    auto fetch = [&](int64_t it, int bsel) {
        const int64_t b = it / nslab;
        const int64_t c0 = (it % nslab) * 1024 + 4 * tid;
        if (c0 < p.C) {
            int64_t srow = b;
            bool ok = true;
            if (p.slots != nullptr) {
                srow = p.slots[b];
                ok = srow >= 0 && srow < p.pool_size;
            }
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                if (j < p.carry && ok && past != nullptr)
                    cp_async8(&buf[bsel][j][tid], past + (srow * p.carry + j) * p.C + c0);
                else if (j == p.carry)
                    cp_async8(&buf[bsel][j][tid], x + b * p.C + c0);
                else
                    buf[bsel][j][tid] = make_uint2(0u, 0u);
            }
            // Taps: K consecutive values per channel, 4 channels = 4K values from w + c0 K.
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                if (j < p.K) cp_async8(&buf[bsel][4 + j][tid], w + c0 * p.K + 4 * j);
                else buf[bsel][4 + j][tid] = make_uint2(0u, 0u);
            }
            if (bias != nullptr) cp_async8(&buf[bsel][8][tid], bias + c0);
            else buf[bsel][8][tid] = make_uint2(0u, 0u);
        }
        stream_commit_conv();
    };

    int64_t it = blockIdx.x;
    if (it >= items) return;
    fetch(it, 0);
    for (int k = 0; it < items; it += gridDim.x, ++k) {
        const int cb = k & 1;
        if (it + gridDim.x < items) fetch(it + gridDim.x, cb ^ 1);
        else stream_commit_conv();
        stream_wait_conv<1>();   // this item's copies have landed; the next item's may fly
        const int64_t b = it / nslab;
        const int64_t c0 = (it % nslab) * 1024 + 4 * tid;
        if (c0 >= p.C) continue;
        int64_t srow = b;
        if (p.slots != nullptr) {
            srow = p.slots[b];
            if (srow < 0 || srow >= p.pool_size) {
                if (c0 == 0) atomicOr(p.status, kDevBadSlot);
                continue;
            }
        }
        // Unpack: positions pos[j][i], taps in the weight layout w[c][j] (channel-major).
        float pos[4][4], tap[4][4], bv[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const uint2 u = buf[cb][j][tid];
            const IO *h = reinterpret_cast<const IO *>(&u);
#pragma unroll
            for (int i = 0; i < 4; ++i) pos[j][i] = IoType<IO>::ld(h + i);
        }
        // The 4K tap values of channels c0..c0+3, in order w[c0][0..K-1], w[c0+1][0..K-1]...
        float wflat[16];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const uint2 u = buf[cb][4 + j][tid];
            const IO *h = reinterpret_cast<const IO *>(&u);
#pragma unroll
            for (int e = 0; e < 4; ++e) wflat[4 * j + e] = IoType<IO>::ld(h + e);
        }
        // Static indices for each K (a runtime index would put wflat in local memory).
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                float t = 0.f;
                if (p.K == 4) t = wflat[4 * i + j];
                else if (p.K == 3) t = j < 3 ? wflat[(3 * i + j) % 16] : 0.f;
                else if (p.K == 2) t = j < 2 ? wflat[(2 * i + j) % 16] : 0.f;
                else t = j < 1 ? wflat[i] : 0.f;
                tap[j][i] = t;
            }
        {
            const uint2 u = buf[cb][8][tid];
            const IO *h = reinterpret_cast<const IO *>(&u);
#pragma unroll
            for (int i = 0; i < 4; ++i) bv[i] = IoType<IO>::ld(h + i);
        }
        float out[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            // The output reads padded positions 0 .. K - 1 (carry = K - 1), oldest first.
            float acc = 0.0f;
#pragma unroll
            for (int j = 0; j < 4; ++j)
                if (j < p.K) acc = fmaf(tap[j][i], pos[j][i], acc);
            acc += bv[i];
            out[i] = p.silu ? silu_fast(acc) : acc;
        }
        st_vec<IO, 4>(y + b * p.C + c0, out);
        if (sout != nullptr) {
            // The present state: padded positions 1 .. carry, copied bit for bit.
#pragma unroll
            for (int j = 0; j < 3; ++j)
                if (j < p.carry)
                    *reinterpret_cast<uint2 *>(sout + (srow * p.carry + j) * p.C + c0) = buf[cb][j + 1][tid];
        }
    }
    stream_wait_conv<0>();
}

struct NormParams {
    const void *x, *scale, *gate;
    void *y;
    int64_t rows;
    int32_t width, activation;
    float eps;
};

template <typename IO, int VEC>
__global__ void __launch_bounds__(256) gated_rmsnorm_kernel(const NormParams p) {
    const IO *x = static_cast<const IO *>(p.x);
    const IO *scale = static_cast<const IO *>(p.scale);
    const IO *gate = static_cast<const IO *>(p.gate);
    IO *y = static_cast<IO *>(p.y);
    const int lane = threadIdx.x & 31;
    const int64_t warps = (int64_t)gridDim.x * (blockDim.x >> 5);
    for (int64_t r = blockIdx.x * (int64_t)(blockDim.x >> 5) + (threadIdx.x >> 5); r < p.rows;
         r += warps) {
        const IO *xr = x + r * p.width;
        float ss = 0.0f;
        for (int i = lane * VEC; i < p.width; i += 32 * VEC) {
            const Vec<IO, VEC> v = ld_vec<IO, VEC>(xr + i);
#pragma unroll
            for (int e = 0; e < VEC; ++e) ss = fmaf(v.v[e], v.v[e], ss);
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
        const float inv = rsqrtf(ss / (float)p.width + p.eps);
        for (int i = lane * VEC; i < p.width; i += 32 * VEC) {
            const Vec<IO, VEC> v = ld_vec<IO, VEC>(xr + i);
            const Vec<IO, VEC> g = ld_vec<IO, VEC>(gate + r * p.width + i);
            const Vec<IO, VEC> sc = ld_vec<IO, VEC>(scale + i);
            float out[VEC];
#pragma unroll
            for (int e = 0; e < VEC; ++e) {
                const float sg = sigmoid_fast(g.v[e]);
                const float act = p.activation == GDN_ACT_SILU ? g.v[e] * sg : sg;
                out[e] = v.v[e] * inv * sc.v[e] * act;
            }
            st_vec<IO, VEC>(y + r * p.width + i, out);
        }
    }
}

// Rows of 128 16-bit values: half a warp per row, 8 values (one 16-byte access) a lane,
// and each warp takes 2 x RPW rows at a time, loading x and the gate of all of them before
// the reductions (16 lanes, four shuffle steps).  The math is the other norm kernels'.
template <typename IO, int RPW>
__global__ void __launch_bounds__(256) gated_rmsnorm_w128_kernel(const NormParams p) {
    static_assert(sizeof(IO) == 2, "16-bit I/O");
    const IO *x = static_cast<const IO *>(p.x);
    const IO *gate = static_cast<const IO *>(p.gate);
    IO *y = static_cast<IO *>(p.y);
    const int lane = threadIdx.x & 31, half = lane >> 4, col = (lane & 15) * 8;
    const int64_t warps = (int64_t)gridDim.x * (blockDim.x >> 5);
    float sc[8];
    {
        const uint4 raw = *reinterpret_cast<const uint4 *>(static_cast<const IO *>(p.scale) + col);
        const IO *h = reinterpret_cast<const IO *>(&raw);
#pragma unroll
        for (int e = 0; e < 8; ++e) sc[e] = IoType<IO>::ld(h + e);
    }
    for (int64_t r0 = (blockIdx.x * (int64_t)(blockDim.x >> 5) + (threadIdx.x >> 5)) * (2 * RPW);
         r0 < p.rows; r0 += warps * (2 * RPW)) {
        uint4 xr[RPW], gr[RPW];
#pragma unroll
        for (int k = 0; k < RPW; ++k) {
            const int64_t r = r0 + 2 * k + half;
            xr[k] = gr[k] = make_uint4(0u, 0u, 0u, 0u);
            if (r < p.rows) {
                xr[k] = *reinterpret_cast<const uint4 *>(x + r * 128 + col);
                gr[k] = *reinterpret_cast<const uint4 *>(gate + r * 128 + col);
            }
        }
        float ss[RPW];
#pragma unroll
        for (int k = 0; k < RPW; ++k) {
            const IO *h = reinterpret_cast<const IO *>(&xr[k]);
            ss[k] = 0.0f;
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                const float v = IoType<IO>::ld(h + e);
                ss[k] = fmaf(v, v, ss[k]);
            }
        }
#pragma unroll
        for (int off = 8; off > 0; off >>= 1)
#pragma unroll
            for (int k = 0; k < RPW; ++k) ss[k] += __shfl_xor_sync(0xffffffffu, ss[k], off);
#pragma unroll
        for (int k = 0; k < RPW; ++k) {
            const int64_t r = r0 + 2 * k + half;
            if (r >= p.rows) continue;
            const float inv = rsqrtf(ss[k] / 128.0f + p.eps);
            const IO *hx = reinterpret_cast<const IO *>(&xr[k]);
            const IO *hg = reinterpret_cast<const IO *>(&gr[k]);
            uint4 out;
            IO *ho = reinterpret_cast<IO *>(&out);
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                const float g = IoType<IO>::ld(hg + e);
                const float sg = sigmoid_fast(g);
                const float act = p.activation == GDN_ACT_SILU ? g * sg : sg;
                IoType<IO>::st(ho + e, IoType<IO>::ld(hx + e) * inv * sc[e] * act);
            }
            *reinterpret_cast<uint4 *>(y + r * 128 + col) = out;
        }
    }
}

// Rows of at most 32 * VEC values: a lane holds VEC values of a row, and a warp takes
// RPW consecutive rows at a time, reading x and the gate of all of them before reducing,
// so 2 * RPW loads per lane are in flight.
template <typename IO, int VEC, int RPW>
__global__ void __launch_bounds__(256) gated_rmsnorm_rows_kernel(const NormParams p) {
    const IO *x = static_cast<const IO *>(p.x);
    const IO *scale = static_cast<const IO *>(p.scale);
    const IO *gate = static_cast<const IO *>(p.gate);
    IO *y = static_cast<IO *>(p.y);
    const int lane = threadIdx.x & 31;
    const int i = lane * VEC;
    const bool on = i < p.width;
    const int64_t warps = (int64_t)gridDim.x * (blockDim.x >> 5);
    Vec<IO, VEC> sc;
#pragma unroll
    for (int e = 0; e < VEC; ++e) sc.v[e] = 0.0f;
    if (on) sc = ld_vec<IO, VEC>(scale + i);
    for (int64_t r0 = (blockIdx.x * (int64_t)(blockDim.x >> 5) + (threadIdx.x >> 5)) * RPW;
         r0 < p.rows; r0 += warps * RPW) {
        Vec<IO, VEC> xv[RPW], gv[RPW];
#pragma unroll
        for (int k = 0; k < RPW; ++k) {
#pragma unroll
            for (int e = 0; e < VEC; ++e) xv[k].v[e] = gv[k].v[e] = 0.0f;
            if (on && r0 + k < p.rows) {
                xv[k] = ld_vec<IO, VEC>(x + (r0 + k) * p.width + i);
                gv[k] = ld_vec<IO, VEC>(gate + (r0 + k) * p.width + i);
            }
        }
        float ss[RPW];
#pragma unroll
        for (int k = 0; k < RPW; ++k) {
            ss[k] = 0.0f;
#pragma unroll
            for (int e = 0; e < VEC; ++e) ss[k] = fmaf(xv[k].v[e], xv[k].v[e], ss[k]);
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1)
#pragma unroll
            for (int k = 0; k < RPW; ++k) ss[k] += __shfl_xor_sync(0xffffffffu, ss[k], off);
#pragma unroll
        for (int k = 0; k < RPW; ++k) {
            if (!on || r0 + k >= p.rows) continue;
            const float inv = rsqrtf(ss[k] / (float)p.width + p.eps);
            float out[VEC];
#pragma unroll
            for (int e = 0; e < VEC; ++e) {
                const float g = gv[k].v[e];
                const float sg = sigmoid_fast(g);
                const float act = p.activation == GDN_ACT_SILU ? g * sg : sg;
                out[e] = xv[k].v[e] * inv * sc.v[e] * act;
            }
            st_vec<IO, VEC>(y + (r0 + k) * p.width + i, out);
        }
    }
}

int sm_count_cached() {
    static int count[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 152;
    if (count[dev] == 0) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
            n = 152;
        count[dev] = n;
    }
    return count[dev];
}

// Grid of a grid-stride kernel: enough blocks for every work item, at most 32 per SM.
unsigned grid_for(int64_t items, int threads) {
    const int64_t need = (items + threads - 1) / threads;
    const int64_t cap = (int64_t)sm_count_cached() * 32;
    return (unsigned)(need < 1 ? 1 : (need < cap ? need : cap));
}

// The streaming decode step (16-bit I/O, four channels a thread): as many CTAs as are
// resident at once, each walking its share of the (row, slab) items.
template <typename IO, int VEC>
cudaError_t launch_conv_decode_stream(const ConvParams &p, cudaStream_t stream) {
    if constexpr (VEC == 4 && sizeof(IO) == 2) {
        int per_sm = 0;
        cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(
            &per_sm, causal_conv_decode_stream_kernel<IO>, 256, 0);
        if (e != cudaSuccess) return e;
        const int64_t resident = (int64_t)sm_count_cached() * (per_sm > 0 ? per_sm : 1);
        const int64_t work = p.B * ((p.C + 1023) / 1024);
        causal_conv_decode_stream_kernel<IO>
            <<<(unsigned)(work < resident ? work : resident), 256, 0, stream>>>(p);
        return cudaGetLastError();
    } else {
        return cudaErrorInvalidValue;
    }
}

template <typename IO, int KT, bool SILU>
cudaError_t launch_conv_tma_k(const ConvParams &p, const ConvTmaMaps &maps, cudaStream_t stream) {
    constexpr int smem = kTmaDepth * kTmaRows * kStagedWidth * 2 + 128;
    static bool attr_set[64] = {false};   // the limit is a per-device function attribute
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (!attr_set[dev]) {
        e = cudaFuncSetAttribute(causal_conv_tma_kernel<IO, KT, SILU>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess) return e;
        attr_set[dev] = true;
    }
    const long long set = __atomic_load_n(&g_wait_budget, __ATOMIC_RELAXED);
    dim3 grid((unsigned)((p.C + kStagedWidth - 1) / kStagedWidth),
              (unsigned)((p.L + kStagedChunk - 1) / kStagedChunk), (unsigned)p.B);
    causal_conv_tma_kernel<IO, KT, SILU>
        <<<grid, 256, smem, stream>>>(p, maps, set > 0 ? set : kConvDrainBudget);
    return cudaGetLastError();
}

template <typename IO, bool SILU>
cudaError_t launch_conv_tma_s(const ConvParams &p, const ConvTmaMaps &maps, cudaStream_t stream) {
    switch (p.K) {
        case 1: return launch_conv_tma_k<IO, 1, SILU>(p, maps, stream);
        case 2: return launch_conv_tma_k<IO, 2, SILU>(p, maps, stream);
        case 3: return launch_conv_tma_k<IO, 3, SILU>(p, maps, stream);
        case 4: return launch_conv_tma_k<IO, 4, SILU>(p, maps, stream);
    }
    return cudaErrorInvalidValue;
}

// The two tensor maps of the TMA conv over x [B][L][C] (false: encoder missing or the
// shape out of the encoder's range, and the caller takes another kernel).
template <typename IO>
bool conv_tma_maps(const ConvParams &p, ConvTmaMaps *m) {
    const gdn_dtype io = std::is_same<IO, __nv_bfloat16>::value ? GDN_BF16 : GDN_F16;
    const uint64_t dims[3] = {(uint64_t)p.C, (uint64_t)p.L, (uint64_t)p.B};
    const uint64_t strides[2] = {(uint64_t)p.C * 2, (uint64_t)p.C * 2 * (uint64_t)p.L};
    const uint32_t box[3] = {(uint32_t)kStagedWidth, (uint32_t)kTmaRows, 1};
    const uint32_t box_first[3] = {(uint32_t)kStagedWidth, (uint32_t)kStagedTokens, 1};
    return encode_map_3d(&m->stage, p.x, io, dims, strides, box) &&
           encode_map_3d(&m->first, p.x, io, dims, strides, box_first);
}

template <typename IO, int VEC>
cudaError_t launch_conv_vec(const ConvParams &p, bool align16, cudaStream_t stream) {
    const int64_t items = p.B * p.tiles * (p.C / VEC);
    if (items == 0) return cudaSuccess;
    const int64_t chunks = (p.L + kStagedChunk - 1) / kStagedChunk;
    // 16-bit values on the staged shapes whose output and state are 16-byte aligned too:
    // the TMA kernel.
    if constexpr (VEC == 4 && sizeof(IO) == 2) {
        const bool out16 = reinterpret_cast<uintptr_t>(p.y) % 16 == 0 &&
                           reinterpret_cast<uintptr_t>(p.state_out) % 16 == 0;
        ConvTmaMaps maps;
        if (align16 && out16 && p.tt == kShortTile && p.window == 0 &&
            p.L >= kStagedMinTokens && p.C % 8 == 0 && p.B <= 65535 && chunks <= 65535 &&
            p.L + 3 < 0x7fffffffLL && conv_tma_maps<IO>(p, &maps))
            return p.silu ? launch_conv_tma_s<IO, true>(p, maps, stream)
                          : launch_conv_tma_s<IO, false>(p, maps, stream);
    }
    if (VEC == 4 && align16 && p.tt == kShortTile && p.window == 0 &&
        p.L >= kStagedMinTokens && p.C % 8 == 0 && p.B <= 65535 && chunks <= 65535) {
        const int smem = kStagedDepth * (kStagedTokens + 3) * kStagedWidth * (int)sizeof(IO);
        // The dynamic shared memory limit is a per-device function attribute.
        static bool attr_set[64] = {false};
        int dev = 0;
        cudaError_t e = cudaGetDevice(&dev);
        if (e != cudaSuccess) return e;
        if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
        if (!attr_set[dev]) {
            e = cudaFuncSetAttribute(causal_conv_staged_kernel<IO>,
                                     cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
            if (e != cudaSuccess) return e;
            attr_set[dev] = true;
        }
        dim3 grid((unsigned)((p.C + kStagedWidth - 1) / kStagedWidth), (unsigned)chunks,
                  (unsigned)p.B);
        causal_conv_staged_kernel<IO><<<grid, 256, smem, stream>>>(p);
    } else if (VEC == 4 && sizeof(IO) == 2 && p.tt == 1 && p.L == 1 && p.window == 0) {
        return launch_conv_decode_stream<IO, VEC>(p, stream);
    } else if (p.tt == 1) {
        const int64_t gx = (p.C / VEC + 255) / 256;
        dim3 grid((unsigned)gx, (unsigned)(p.B < 65535 ? p.B : 65535));
        causal_conv_short_kernel<IO, VEC, 1><<<grid, 256, 0, stream>>>(p);
    } else if (p.tt == kShortTile) {
        // x: blocks of 256 channel groups; y: (row, tile) pairs, strided past 65535.
        const int64_t gx = (p.C / VEC + 255) / 256;
        const int64_t pairs = p.B * p.tiles;
        dim3 grid((unsigned)gx, (unsigned)(pairs < 65535 ? pairs : 65535));
        causal_conv_short_kernel<IO, VEC, kShortTile><<<grid, 256, 0, stream>>>(p);
    }
    else
        causal_conv_kernel<IO, VEC><<<grid_for(items, 256), 256, 0, stream>>>(p);
    return cudaGetLastError();
}

template <typename IO>
cudaError_t launch_conv_io(const ConvParams &p, bool vec4, bool align16, cudaStream_t stream) {
    return vec4 ? launch_conv_vec<IO, 4>(p, align16, stream)
                : launch_conv_vec<IO, 1>(p, align16, stream);
}

template <typename IO>
cudaError_t launch_norm_io(const NormParams &p, bool vec4, cudaStream_t stream) {
    const int64_t threads = p.rows * 32;
    if (threads == 0) return cudaSuccess;
    constexpr int RPW = 4;
    if constexpr (sizeof(IO) == 2) {
        // Rows of 128 with every pointer 16-byte aligned: half a warp per row.
        const bool a16 = ((reinterpret_cast<uintptr_t>(p.x) | reinterpret_cast<uintptr_t>(p.gate) |
                           reinterpret_cast<uintptr_t>(p.y) | reinterpret_cast<uintptr_t>(p.scale)) & 15) == 0;
        if (p.width == 128 && a16) {
            gated_rmsnorm_w128_kernel<IO, RPW>
                <<<grid_for((p.rows + 2 * RPW - 1) / (2 * RPW) * 32, 256), 256, 0, stream>>>(p);
            return cudaGetLastError();
        }
    }
    if (vec4 && p.width <= 128)
        gated_rmsnorm_rows_kernel<IO, 4, RPW>
            <<<grid_for((p.rows + RPW - 1) / RPW * 32, 256), 256, 0, stream>>>(p);
    else if (vec4)
        gated_rmsnorm_kernel<IO, 4><<<grid_for(threads, 256), 256, 0, stream>>>(p);
    else if (p.width <= 32)
        gated_rmsnorm_rows_kernel<IO, 1, RPW>
            <<<grid_for((p.rows + RPW - 1) / RPW * 32, 256), 256, 0, stream>>>(p);
    else
        gated_rmsnorm_kernel<IO, 1><<<grid_for(threads, 256), 256, 0, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_causal_conv(const ConvLaunch &l, cudaStream_t stream) {
    ConvParams p{};
    p.x = l.x; p.w = l.w; p.bias = l.bias; p.state_in = l.state_in;
    p.y = l.y; p.state_out = l.state_out;
    p.B = l.batch; p.L = l.seqlen;
    p.C = l.channels; p.K = l.kernel; p.dil = l.dilation;
    p.carry = (l.kernel - 1) * l.dilation;
    p.channels_last = l.channels_last; p.silu = l.activation == GDN_ACT_SILU;
    p.window = l.window;
    p.slots = l.slots; p.pool_size = l.pool_size;
    p.status = l.status;
    // Tiles of at least `carry` tokens, so only tile 0 reads the past state: kShortTile for
    // the register-tiled kernel (K <= 4, dilation 1, channels last), else 16 or carry.
    if (p.channels_last && p.dil == 1 && p.K <= 4)
        p.tt = p.L <= 1 ? 1 : kShortTile;   // one token a thread for a decode step
    else
        p.tt = p.carry > 16 ? p.carry : 16;
    p.tiles = p.L > 0 ? (p.L + p.tt - 1) / p.tt : 1;
    switch (l.io) {
        case GDN_F32: return launch_conv_io<float>(p, l.vec4, l.align16, stream);
        case GDN_BF16: return launch_conv_io<__nv_bfloat16>(p, l.vec4, l.align16, stream);
        case GDN_F16: return launch_conv_io<__half>(p, l.vec4, l.align16, stream);
    }
    return cudaErrorInvalidValue;
}

cudaError_t launch_gated_rmsnorm(gdn_dtype io, int64_t rows, int32_t width, const void *x,
                                 const void *scale, const void *gate, float eps,
                                 int32_t activation, void *y, bool vec4, cudaStream_t stream) {
    NormParams p{x, scale, gate, y, rows, width, activation, eps};
    switch (io) {
        case GDN_F32: return launch_norm_io<float>(p, vec4, stream);
        case GDN_BF16: return launch_norm_io<__nv_bfloat16>(p, vec4, stream);
        case GDN_F16: return launch_norm_io<__half>(p, vec4, stream);
    }
    return cudaErrorInvalidValue;
}

}  // namespace gdn
