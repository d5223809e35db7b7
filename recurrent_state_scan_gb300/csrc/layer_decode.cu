// layer_decode.cu -- one decode step of a gated delta-rule layer in one kernel: the causal
// convolution that produces q, k and v, the recurrence step, and the gated RMS norm of
// its output.
//
// What it computes is the composition of three ops the pages define separately:
//  * onnxruntime-ep-mlx 0.31.1, src/ops/ssm.rs, `causal_conv_op` (CausalConvWithState):
//    every channel c of the layer's mixed input row x_t is convolved with its own K taps
//    over [past state ; x_t], plus a bias, then optionally passed through silu; the
//    present state is the last K - 1 inputs.  The channels are read as q, then k, then v:
//    c = hq * d_k + i for q, h_qk * d_k + hq * d_k + i for k, 2 h_qk d_k + h * d_v + j
//    for v.
//  * onnx-runtime-ep-cuda 0.1.0-dev.6, src/kernels/linear_attention.rs,
//    `linear_attention_core` Steps 1-4 with the fused gate chain, for the one token.
//  * ssm.rs `gated_rms_norm_op` (GatedRMSNorm) over each (sequence, value head) row of
//    d_v outputs: y = o / sqrt(mean(o^2) + eps) * scale * act(gate).
// Each op rounds its output to the I/O type, as the three separate library calls would:
// the convolution's q, k and v and the step's o are rounded before the next op reads
// them.  Nothing of them is written to global memory.
//
// Work unit: one (sequence, value head), whose 64-column state tiles one persistent CTA
// of 128 threads walks in turn (16 rows x 4 columns of the tile a thread, as the decode
// step's streaming kernel does), so that the whole o row is in shared memory for the
// norm.  The next tile's state slots and its convolution inputs stream into shared
// memory with cp.async while the current tile is computed.  The q and k channels of a
// value head's qk head are convolved again by every tile that needs them; their present
// state is written by the first value head of the group at tile 0, so the state must
// come in and go out through different buffers.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "gdn_internal.cuh"

namespace gdn {
namespace {

constexpr int kLdThreads = 128;        // threads of a CTA
constexpr int kLdLpr = 16;             // threads across a tile's 64 columns (4 each)
constexpr int kLdRpp = kLdThreads / kLdLpr;   // row groups
constexpr int kLdRpt = 128 / kLdRpp;   // state rows a thread holds (d_k = 128)
constexpr int kLdTile = 64;            // state columns of a tile
constexpr int kLdCh = 2 * 128 + kLdTile;      // convolved channels a tile needs: q, k, v
constexpr int kLdMaxK = 8;             // taps
constexpr int kLdMaxDv = 256;

__device__ __forceinline__ void ld_cp16(void *smem, const void *gmem) {
    const unsigned a = static_cast<unsigned>(__cvta_generic_to_shared(smem));
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(a), "l"(gmem) : "memory");
}
__device__ __forceinline__ void ld_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
__device__ __forceinline__ void ld_wait_all() { asm volatile("cp.async.wait_group 0;\n" ::: "memory"); }

// sigmoid from the fast exponential and divide (a few ulp; 0 for very negative x), as the
// separate conv and norm kernels evaluate their activations.
__device__ __forceinline__ float sigmoid_fast_ld(float x) { return __fdividef(1.0f, 1.0f + __expf(-x)); }
// act(g) of the norm: g sigmoid(g) (silu) or sigmoid(g).
__device__ __forceinline__ float norm_act(float g, int act) {
    const float s = sigmoid_fast_ld(g);
    return act == GDN_ACT_SILU ? g * s : s;
}

// Staged inputs of one tile, in I/O elements: the three channel blocks (q 128, k 128,
// v 64) of x, of each of the K - 1 state rows and of the bias, the taps of those
// channels (K per channel, channel-major), then the tile's gate and norm scale.
struct StageLayout {
    int x, st, w, bias, gate, nscale, total;
    __device__ __forceinline__ StageLayout(int K) {
        x = 0;
        st = kLdCh;
        w = st + (K - 1) * kLdCh;
        bias = w + K * kLdCh;
        gate = bias + kLdCh;
        nscale = gate + kLdTile;
        total = nscale + kLdTile;
    }
};

// The same layout on the host (sizes the dynamic shared memory).
struct StageLayoutHost {
    int K;
    int total_elems() const { return kLdCh + (K - 1) * kLdCh + K * kLdCh + kLdCh + 2 * kLdTile; }
};

// x rounded to the I/O type and widened again: the value a separate op would store.
template <typename IO> __device__ __forceinline__ float round_io(float x);
template <> __device__ __forceinline__ float round_io<float>(float x) { return x; }
template <> __device__ __forceinline__ float round_io<__nv_bfloat16>(float x) {
    return __bfloat162float(__float2bfloat16_rn(x));
}
template <> __device__ __forceinline__ float round_io<__half>(float x) { return __half2float(__float2half_rn(x)); }

template <typename IO>
__global__ void __launch_bounds__(kLdThreads, 4) decode_layer_kernel(const LayerDecodeParams p) {
    constexpr int ES = (int)sizeof(IO);
    extern __shared__ __align__(16) unsigned char ld_stage[];      // staged inputs, StageLayout
    __shared__ __align__(16) float4 pre[kLdRpt][kLdThreads];       // the next tile's state slots
    __shared__ float sq[128], sk[128], sv[kLdTile], sdelta[kLdTile];
    __shared__ __align__(16) float red_k[kLdRpp * kLdTile];
    __shared__ __align__(16) float red_q[kLdRpp * kLdTile];
    __shared__ float so[kLdMaxDv], sgate[kLdMaxDv], sns[kLdMaxDv];   // the head's o row, gate, scale
    __shared__ float s_alpha, s_beta, s_qk, s_rms, s_part[kLdThreads / 32];

    const int tid = threadIdx.x, lr = tid % kLdLpr, rg = tid / kLdLpr;
    const int K = p.conv_k, tiles = p.d_v / kLdTile, group = p.h_v / p.h_qk;
    const int64_t C = 2LL * p.h_qk * 128 + (int64_t)p.h_v * p.d_v;
    const int64_t heads = (int64_t)p.batch * p.h_v;
    const StageLayout L(K);
    IO *stage = reinterpret_cast<IO *>(ld_stage);
    const IO *x = static_cast<const IO *>(p.x);
    const IO *w = static_cast<const IO *>(p.conv_w);
    const IO *cb = static_cast<const IO *>(p.conv_b);
    const IO *csi = static_cast<const IO *>(p.conv_state_in);
    IO *cso = static_cast<IO *>(p.conv_state_out);
    const IO *ga = static_cast<const IO *>(p.a);
    const IO *gb = static_cast<const IO *>(p.b);
    const IO *gate = static_cast<const IO *>(p.gate);
    const IO *ns = static_cast<const IO *>(p.norm_scale);
    IO *y = static_cast<IO *>(p.y);

    struct Unit {
        int64_t n;
        int h, hq, tile;
    };
    auto unit_at = [&](int64_t hu, int tile) {
        Unit u;
        u.n = hu / p.h_v;
        u.h = (int)(hu % p.h_v);
        u.hq = u.h / group;
        u.tile = tile;
        return u;
    };
    // First global channel of block b3 (q, k, v) of unit u.
    auto chan0 = [&](const Unit &u, int b3) -> int64_t {
        if (b3 == 0) return (int64_t)u.hq * 128;
        if (b3 == 1) return (int64_t)(p.h_qk + u.hq) * 128;
        return 2LL * p.h_qk * 128 + (int64_t)u.h * p.d_v + (int64_t)u.tile * kLdTile;
    };
    float ra = 0.f, rb = 0.f, rA = 0.f, rD = 0.f;   // the next tile's gate inputs
    // Issue the copies of tile u: its state slots and its staged inputs (16-byte cp.async
    // granules; absent state rows and bias are zero-filled).
    // The state slots this thread will hold: issued as soon as the thread has moved the
    // current tile's slots to registers (no other thread touches them).
    auto prefetch_state = [&](const Unit &u) {
        const int col0 = u.tile * kLdTile + 4 * lr;
        const size_t sbase = ((size_t)u.n * p.h_v + u.h) * (size_t)128 * p.d_v;
#pragma unroll
        for (int m = 0; m < kLdRpt; ++m)
            ld_cp16(&pre[m][tid], p.state + sbase + (size_t)(rg + kLdRpp * m) * p.d_v + col0);
    };
    // The staged inputs, once every thread has read the current ones.
    auto prefetch_stage = [&](const Unit &u) {
        auto seg = [&](int dst, const IO *src, int count) {
            unsigned char *d = reinterpret_cast<unsigned char *>(stage + dst);
            const unsigned char *s8 = reinterpret_cast<const unsigned char *>(src);
            for (int g = tid; g < count * ES / 16; g += kLdThreads) ld_cp16(d + 16 * g, s8 + 16 * g);
        };
        auto zero = [&](int dst, int count) {
            for (int e = tid; e < count; e += kLdThreads) stage[dst + e] = IO(0.0f);
        };
        const int base[3] = {0, 128, 256}, cnt[3] = {128, 128, kLdTile};
        // q and k are the same for every tile of the head: they are convolved at tile 0.
        for (int b3 = u.tile == 0 ? 0 : 2; b3 < 3; ++b3) {
            const int64_t c0 = chan0(u, b3);
            seg(L.x + base[b3], x + u.n * C + c0, cnt[b3]);
            for (int j = 0; j < K - 1; ++j) {
                if (csi) seg(L.st + j * kLdCh + base[b3], csi + (u.n * (K - 1) + j) * C + c0, cnt[b3]);
                else zero(L.st + j * kLdCh + base[b3], cnt[b3]);
            }
            seg(L.w + base[b3] * K, w + c0 * K, cnt[b3] * K);
            if (cb) seg(L.bias + base[b3], cb + c0, cnt[b3]);
            else zero(L.bias + base[b3], cnt[b3]);
        }
        seg(L.gate, gate + ((size_t)u.n * p.h_v + u.h) * p.d_v + (size_t)u.tile * kLdTile, kLdTile);
        seg(L.nscale, ns + (size_t)u.tile * kLdTile, kLdTile);
        ld_commit();
        const size_t gi = (size_t)u.n * p.h_v + u.h;
        if (tid == 0) {
            ra = IoType<IO>::ld(ga + gi);
            rA = p.A_log[u.h];
            rD = p.dt_bias[u.h];
        }
        if (tid == 32) rb = IoType<IO>::ld(gb + gi);
    };

    int64_t hu = blockIdx.x;
    if (hu >= heads) return;
    Unit cur = unit_at(hu, 0);
    prefetch_state(cur);
    prefetch_stage(cur);
    for (;;) {
        ld_wait_all();              // this thread's copies of the tile have landed
        __syncthreads();            // everyone's copies and zero fills have landed
        const Unit u = cur;
        float4 S[kLdRpt];
#pragma unroll
        for (int m = 0; m < kLdRpt; ++m) S[m] = pre[m][tid];
        // The next tile: its state starts streaming now.
        bool more = true;
        if (u.tile + 1 < tiles) {
            cur = unit_at(hu, u.tile + 1);
        } else {
            hu += gridDim.x;
            more = hu < heads;
            if (more) cur = unit_at(hu, 0);
        }
        if (more) prefetch_state(cur);
        // The convolution of the tile's channels, rounded to the I/O type: q, k, this
        // tile's 64 values of v; and the present state pad[1 .. K - 1] of the channels
        // this tile owns.
        for (int c = (u.tile == 0 ? 0 : 256) + tid; c < kLdCh; c += kLdThreads) {
            float pad[kLdMaxK];
#pragma unroll
            for (int j = 0; j < kLdMaxK; ++j) {
                if (j < K - 1) pad[j] = IoType<IO>::ld(stage + L.st + j * kLdCh + c);
                else if (j == K - 1) pad[j] = IoType<IO>::ld(stage + L.x + c);
            }
            float acc = IoType<IO>::ld(stage + L.bias + c);
#pragma unroll
            for (int j = 0; j < kLdMaxK; ++j)
                if (j < K) acc = fmaf(IoType<IO>::ld(stage + L.w + c * K + j), pad[j], acc);
            if (p.conv_silu) acc *= sigmoid_fast_ld(acc);
            const float val = round_io<IO>(acc);
            if (c < 128) sq[c] = val;
            else if (c < 256) sk[c - 128] = val;
            else sv[c - 256] = val;
            const int b3 = c < 128 ? 0 : (c < 256 ? 1 : 2);
            const bool owner = b3 == 2 || (u.h % group == 0 && u.tile == 0);
            if (cso != nullptr && owner) {
                const int64_t gc = chan0(u, b3) + (c - (b3 == 0 ? 0 : (b3 == 1 ? 128 : 256)));
#pragma unroll
                for (int j = 0; j < kLdMaxK - 1; ++j)
                    if (j < K - 1) IoType<IO>::st(cso + (u.n * (K - 1) + j) * C + gc, pad[j + 1]);
            }
        }
        if (tid < kLdTile) {
            sgate[u.tile * kLdTile + tid] = IoType<IO>::ld(stage + L.gate + tid);
            sns[u.tile * kLdTile + tid] = IoType<IO>::ld(stage + L.nscale + tid);
        }
        if (tid == 0) s_alpha = expf(decay_f(ra, rA, rD));
        if (tid == 32) s_beta = sigmoid_f(rb);
        __syncthreads();            // the staging tile is read

        if (more) prefetch_stage(cur);   // the next tile's staged inputs

        // Partial retrieval S^T k and readout S^T q over this thread's rows.
        float4 pk = make_float4(0.f, 0.f, 0.f, 0.f), pq = pk;
#pragma unroll
        for (int m = 0; m < kLdRpt; ++m) {
            const int i = rg + kLdRpp * m;
            const float kk = sk[i], qq = sq[i];
            pk.x = fmaf(S[m].x, kk, pk.x); pk.y = fmaf(S[m].y, kk, pk.y);
            pk.z = fmaf(S[m].z, kk, pk.z); pk.w = fmaf(S[m].w, kk, pk.w);
            pq.x = fmaf(S[m].x, qq, pq.x); pq.y = fmaf(S[m].y, qq, pq.y);
            pq.z = fmaf(S[m].z, qq, pq.z); pq.w = fmaf(S[m].w, qq, pq.w);
        }
        *reinterpret_cast<float4 *>(&red_k[rg * kLdTile + 4 * lr]) = pk;
        *reinterpret_cast<float4 *>(&red_q[rg * kLdTile + 4 * lr]) = pq;
        if (tid < 32) {
            float acc = 0.f;
            for (int i = tid; i < 128; i += 32) acc = fmaf(sq[i], sk[i], acc);
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
            if (tid == 0) s_qk = acc;
        }
        __syncthreads();            // the partial sums are in shared memory

        const float alpha = s_alpha;
        if (tid < kLdTile) {
            float rk = 0.f, rq = 0.f;
#pragma unroll
            for (int r = 0; r < kLdRpp; ++r) {
                rk += red_k[r * kLdTile + tid];
                rq += red_q[r * kLdTile + tid];
            }
            // r = (alpha S)^T k; delta = beta (v - r); o = scale (alpha S + k delta^T)^T q
            const float delta = s_beta * (sv[tid] - alpha * rk);
            sdelta[tid] = delta;
            so[u.tile * kLdTile + tid] = round_io<IO>(p.scale * fmaf(s_qk, delta, alpha * rq));
        }
        __syncthreads();

        const float4 d4 = *reinterpret_cast<const float4 *>(&sdelta[4 * lr]);
        const int col0 = u.tile * kLdTile + 4 * lr;
        const size_t sbase = ((size_t)u.n * p.h_v + u.h) * (size_t)128 * p.d_v;
#pragma unroll
        for (int m = 0; m < kLdRpt; ++m) {
            const float kk = sk[rg + kLdRpp * m];
            S[m].x = fmaf(alpha, S[m].x, kk * d4.x);
            S[m].y = fmaf(alpha, S[m].y, kk * d4.y);
            S[m].z = fmaf(alpha, S[m].z, kk * d4.z);
            S[m].w = fmaf(alpha, S[m].w, kk * d4.w);
            __stcs(reinterpret_cast<float4 *>(p.state + sbase + (size_t)(rg + kLdRpp * m) * p.d_v + col0), S[m]);
        }

        if (u.tile == tiles - 1) {
            // The gated RMS norm of the head's o row.
            float ss = 0.f;
            for (int j = tid; j < p.d_v; j += kLdThreads) ss = fmaf(so[j], so[j], ss);
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
            if ((tid & 31) == 0) s_part[tid >> 5] = ss;
            __syncthreads();
            if (tid == 0) {
                float t = 0.f;
#pragma unroll
                for (int i = 0; i < kLdThreads / 32; ++i) t += s_part[i];
                s_rms = 1.0f / sqrtf(t / (float)p.d_v + p.eps);
            }
            __syncthreads();
            const float r = s_rms;
            IO *yr = y + ((size_t)u.n * p.h_v + u.h) * p.d_v;
            for (int j = tid; j < p.d_v; j += kLdThreads)
                IoType<IO>::st(yr + j, so[j] * r * sns[j] * norm_act(sgate[j], p.norm_act));
        }
        if (!more) break;
    }
}

template <typename IO>
cudaError_t launch_layer_io(const LayerDecodeParams &p, cudaStream_t stream) {
    const int64_t heads = (int64_t)p.batch * p.h_v;
    if (heads <= 0) return cudaSuccess;
    StageLayoutHost L{p.conv_k};
    const size_t dyn = (size_t)L.total_elems() * sizeof(IO);
    struct DevInfo {
        int sms, smem_sm, reserved, static_smem;
    };
    static DevInfo info[64] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    e = cudaFuncSetAttribute(decode_layer_kernel<IO>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)dyn);
    if (e != cudaSuccess) return e;
    DevInfo &d = info[dev];
    if (d.sms == 0) {
        cudaFuncAttributes fa;
        e = cudaDeviceGetAttribute(&d.smem_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev);
        if (e == cudaSuccess) e = cudaDeviceGetAttribute(&d.reserved, cudaDevAttrReservedSharedMemoryPerBlock, dev);
        if (e == cudaSuccess) e = cudaFuncGetAttributes(&fa, decode_layer_kernel<IO>);
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(decode_layer_kernel<IO>, cudaFuncAttributePreferredSharedMemoryCarveout,
                                     (int)cudaSharedmemCarveoutMaxShared);
        if (e == cudaSuccess) e = cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) {
            d.sms = 0;
            return e;
        }
        d.static_smem = (int)fa.sharedSizeBytes;
    }
    // As many CTAs as the SMs' shared memory holds at this stage size, at most the four
    // the launch bounds size the registers for.
    int per_sm = (int)(d.smem_sm / (size_t)(d.static_smem + dyn + d.reserved));
    if (per_sm > 4) per_sm = 4;
    if (d.sms <= 0 || per_sm <= 0) return cudaErrorInvalidConfiguration;
    const int64_t slots = (int64_t)d.sms * per_sm;
    const int64_t ctas = heads < slots ? heads : slots;
    decode_layer_kernel<IO><<<(unsigned)ctas, kLdThreads, dyn, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_decode_layer(const LayerDecodeParams &p, gdn_dtype io, cudaStream_t stream) {
    switch (io) {
        case GDN_F32: return launch_layer_io<float>(p, stream);
        case GDN_BF16: return launch_layer_io<__nv_bfloat16>(p, stream);
        case GDN_F16: return launch_layer_io<__half>(p, stream);
    }
    return cudaErrorInvalidValue;
}

}  // namespace gdn
