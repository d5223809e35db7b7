// prefill_tc.cu -- chunked gated delta-rule prefill on the tcgen05 tensor cores.
//
// What it computes is the recurrence of onnx-runtime-ep-cuda 0.1.0-dev.6,
// src/kernels/linear_attention.rs (`linear_attention_core`, Steps 1-4), re-associated
// over chunks of C = 64 tokens so that the work becomes dense contractions.  With
// S0 the state entering a chunk, G_i = g_1 + ... + g_i and gamma_i = e^{G_i}:
//   A_ij = beta_i e^{G_i-G_j} k_i.k_j (j < i),  T = (I + A)^-1
//   W = T diag(beta gamma) K,   U = T diag(beta) V,   Delta = U - W S0
//   o_i = scale gamma_i q_i^T S0 + sum_{j<=i} scale e^{G_i-G_j} (q_i.k_j) Delta_j
//   S  = gamma_C S0 + (diag(e^{G_C-G}) K)^T Delta
// Every product above runs on tcgen05 (bf16/f16 operands, fp32 accumulation in
// TMEM); T is formed in fp32 on the SIMT cores; the state S stays in TMEM in fp32
// for the whole sequence.  The pages run the recurrence one token at a time; this
// chunked form is a re-association, exact up to rounding.
//
// One CTA (256 threads) owns one (sequence, value head, slice of NV state columns).
// Columns of S evolve independently (the page's "Parallelization" note), so a slice
// needs only its columns of V, U, Delta and o; the q/k-only chunk work (k.k, q.k, T,
// W) is recomputed by each slice.
//
// All MMAs use M = 128 so every accumulator row lives in TMEM lane = row:
//   D1  = [K ; Q] K^T       (K-major A and B)      lanes 0-63 K K^T, 64-127 Q K^T
//   D2  = [T'; T''] K       (B = K tile MN-major)  lanes 0-63 W
//   D3  = [T'; T''] V       (B = V tile MN-major)  lanes 64-127 U
//   D4  = [Q ; W] S         (B = S bf16 MN-major)  lanes 0-63 Q S, 64-127 W S
//   D5  = [P ; 0] Delta     (B = Delta MN-major)   lanes 0-63 P Delta
//   DS += Ktil^T Delta      (A = Ktil MN-major)    lanes = d_k rows of S
// with T' = T diag(beta gamma), T'' = T diag(beta), P_ij = scale e^{G_i-G_j} q_i.k_j.
// Rows past the end of a sequence get g = 0 and beta = 0, which makes their T row the
// unit row and their W, U and Delta rows exactly zero, so they change nothing.
#include <cudaTypedefs.h>

#include "gdn_internal.cuh"
#include "tc_ptx.cuh"

namespace gdn {
namespace {

using namespace tc;

constexpr int kC = 64;             // tokens per chunk
constexpr int kDK = 128;           // d_k (and full d_v) of this path
constexpr int kThreads = 256;
constexpr long long kWaitBudget = 4000000000LL;   // cycles (~2 s) before a wait gives up

struct TcParams {
    CUtensorMap tm_q, tm_k, tm_v;
    const void *a, *b;
    const float *A_log, *dt_bias;
    const float *state_in;
    float *state_out;
    void *o;
    const int32_t *cu_seqlens;
    int64_t seqlen;
    int32_t num_seqs, h_qk, h_v;
    float scale;
    int *status;
};

// Shared-memory plan (byte offsets from a 1024-aligned base).
template <int NV>
struct Plan {
    static constexpr int kRegion = 24576;                    // 192 rows x 128 B: K | Q | W
    static constexpr int KQW = 0;                            // 2 regions (d_k 0-63, 64-127)
    static constexpr int V = KQW + 2 * kRegion;              // NV/64 regions of 64 x 128 B
    static constexpr int KT = V + (NV / 64) * 8192;          // Ktil, 2 regions 64 x 128 B
    static constexpr int TT = KT + 2 * 8192;                 // [T'; T''] 128 x 128 B
    static constexpr int PZ = TT + 16384;                    // [P; 0]    128 x 128 B
    static constexpr int SB = PZ + 16384;                    // S bf16, NV/64 regions 128 x 128 B
    static constexpr int DB = SB + (NV / 64) * 16384;        // Delta,  NV/64 regions 64 x 128 B
    static constexpr int AS = DB + (NV / 64) * 8192;         // A fp32 [64][65]
    static constexpr int TS = AS + 17408;                    // T fp32 [64][65]
    static constexpr int kBytes = TS + 17408;
    static constexpr int kAlloc = kBytes + 1024;             // slack for the 1024 alignment
    // TMEM columns
    static constexpr uint32_t tD1 = 0, tD24 = 64, tD35 = 192, tDS = 192 + NV;
};

template <typename IO> struct Pack;
template <> struct Pack<__nv_bfloat16> {
    static __device__ __forceinline__ uint32_t two(float a, float b) {
        __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
        return *reinterpret_cast<uint32_t *>(&v);
    }
    static __device__ __forceinline__ float2 unpack(uint32_t u) {
        return __bfloat1622float2(*reinterpret_cast<__nv_bfloat162 *>(&u));
    }
};
template <> struct Pack<__half> {
    static __device__ __forceinline__ uint32_t two(float a, float b) {
        __half2 v = __floats2half2_rn(a, b);
        return *reinterpret_cast<uint32_t *>(&v);
    }
    static __device__ __forceinline__ float2 unpack(uint32_t u) {
        return __half22float2(*reinterpret_cast<__half2 *>(&u));
    }
};

template <typename IO>
__device__ __forceinline__ uint4 pack8(const float *x) {
    return make_uint4(Pack<IO>::two(x[0], x[1]), Pack<IO>::two(x[2], x[3]),
                      Pack<IO>::two(x[4], x[5]), Pack<IO>::two(x[6], x[7]));
}

// T = (I + A)^-1 for a 64 x 64 strictly-lower A (row stride 65 floats), in fp32.
// Diagonal 16x16 blocks by forward substitution, then block forward substitution
// T_ij = -T_ii sum_{k=j}^{i-1} A_ik T_kj for the blocks below the diagonal.
// Entries above the diagonal of T are left unwritten.
__device__ void invert_unit_lower_64(const float *As, float *Ts, float (*sX)[16][17], int tid) {
    if (tid < 64) {
        const int blk = tid >> 4, j = tid & 15, o = blk * 16;
        float x[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            if (i < j) {
                x[i] = 0.f;
            } else if (i == j) {
                x[i] = 1.f;
            } else {
                float acc = 0.f;
#pragma unroll
                for (int l = 0; l < i; ++l)
                    if (l >= j) acc = fmaf(As[(o + i) * 65 + o + l], x[l], acc);
                x[i] = -acc;
            }
        }
#pragma unroll
        for (int i = 0; i < 16; ++i)
            if (i >= j) Ts[(o + i) * 65 + o + j] = x[i];
    }
    __syncthreads();
    for (int bi = 1; bi < 4; ++bi) {
        for (int e = tid; e < bi * 256; e += kThreads) {
            const int bj = e >> 8, r = (e >> 4) & 15, cc = e & 15;
            float acc = 0.f;
            for (int k = bj; k < bi; ++k) {
#pragma unroll
                for (int l = 0; l < 16; ++l)
                    acc = fmaf(As[(bi * 16 + r) * 65 + k * 16 + l], Ts[(k * 16 + l) * 65 + bj * 16 + cc],
                               acc);
            }
            sX[bj][r][cc] = acc;
        }
        __syncthreads();
        for (int e = tid; e < bi * 256; e += kThreads) {
            const int bj = e >> 8, r = (e >> 4) & 15, cc = e & 15;
            float acc = 0.f;
#pragma unroll
            for (int l = 0; l < 16; ++l)
                if (l <= r) acc = fmaf(Ts[(bi * 16 + r) * 65 + bi * 16 + l], sX[bj][l][cc], acc);
            Ts[(bi * 16 + r) * 65 + bj * 16 + cc] = -acc;
        }
        __syncthreads();
    }
}

template <typename IO, int NV>
__global__ void __launch_bounds__(kThreads, 1) prefill_tc_kernel(const __grid_constant__ TcParams p) {
    using PL = Plan<NV>;
    constexpr bool kBf16 = std::is_same<IO, __nv_bfloat16>::value;
    constexpr int NSL = kDK / NV;                 // column slices per head
    constexpr int HALF = NV / 2;                  // columns per thread in 2-warp splits
    constexpr uint32_t kIdD1 = idesc_f16(kBf16, 128, 64, false, false);
    constexpr uint32_t kIdD2 = idesc_f16(kBf16, 128, 128, false, true);
    constexpr uint32_t kIdNV = idesc_f16(kBf16, 128, NV, false, true);
    constexpr uint32_t kIdDS = idesc_f16(kBf16, 128, NV, true, true);

    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                              ~static_cast<uintptr_t>(1023));
    __shared__ uint64_t bar_load, bar_mma;
    __shared__ uint32_t s_tmem;
    __shared__ float sG[kC], sBeta[kC], sGam[kC], sKf[kC];
    __shared__ float s_wsum[2];
    __shared__ float sX[3][16][17];

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int quarter = warp & 3, half = warp >> 2;
    const int slice = blockIdx.x % NSL;
    const int h = (blockIdx.x / NSL) % p.h_v;
    const int64_t n = (int64_t)(blockIdx.x / NSL) / p.h_v;
    const int hq = h / (p.h_v / p.h_qk);
    const int v0 = slice * NV;

    int64_t t0, t1;
    if (!seq_range(p.cu_seqlens, p.seqlen, p.num_seqs, p.status, n, t0, t1)) return;

    uint8_t *const sKQW = sm + PL::KQW, *const sV = sm + PL::V, *const sKT = sm + PL::KT;
    uint8_t *const sTT = sm + PL::TT, *const sPZ = sm + PL::PZ, *const sSB = sm + PL::SB;
    uint8_t *const sDB = sm + PL::DB;
    float *const As = reinterpret_cast<float *>(sm + PL::AS);
    float *const Ts = reinterpret_cast<float *>(sm + PL::TS);

    if (warp == 0) {
        tmem_alloc(&s_tmem, 512);
        tmem_relinquish();
    }
    if (tid == 0) {
        mbar_init(&bar_load, 1);
        mbar_init(&bar_mma, 1);
        fence_mbar_init();
        tma_prefetch_desc(&p.tm_q);
        tma_prefetch_desc(&p.tm_k);
        tma_prefetch_desc(&p.tm_v);
    }
    // Zero rows 64-127 of [P; 0] once.
    for (int e = tid; e < 8192 / 16; e += kThreads)
        *reinterpret_cast<uint4 *>(sPZ + 8192 + 16 * e) = make_uint4(0, 0, 0, 0);
    fence_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();

    const uint32_t tmem = s_tmem;
    const uint32_t lane_base = static_cast<uint32_t>(32 * quarter) << 16;
    const int row = 32 * quarter + lane;           // this thread's TMEM lane
    const IO *ga = static_cast<const IO *>(p.a);
    const IO *gb = static_cast<const IO *>(p.b);
    IO *go = static_cast<IO *>(p.o);
    const float A_log = p.A_log[h], dt_bias = p.dt_bias[h];
    const size_t sbase = ((size_t)n * p.h_v + h) * kDK * kDK;

    // Initial state -> DS (thread: row `row`, columns [half*HALF, +HALF)).
#pragma unroll
    for (int c0 = 0; c0 < HALF; c0 += 32) {
        const int col = half * HALF + c0;
        uint32_t r[32];
        if (p.state_in != nullptr) {
            const float4 *src =
                reinterpret_cast<const float4 *>(p.state_in + sbase + (size_t)row * kDK + v0 + col);
#pragma unroll
            for (int q4 = 0; q4 < 8; ++q4) {
                const float4 f = src[q4];
                r[4 * q4 + 0] = __float_as_uint(f.x);
                r[4 * q4 + 1] = __float_as_uint(f.y);
                r[4 * q4 + 2] = __float_as_uint(f.z);
                r[4 * q4 + 3] = __float_as_uint(f.w);
            }
        } else {
#pragma unroll
            for (int j = 0; j < 32; ++j) r[j] = 0u;
        }
        tmem_st32(tmem + lane_base + PL::tDS + col, r);
    }
    tmem_st_wait();

    uint32_t ph_load = 0, ph_mma = 0;
    bool failed = false;
    const int64_t L = t1 - t0;
    const int64_t nchunks = (L + kC - 1) / kC;
    const uint32_t aKQW = smem_u32(sKQW), aV = smem_u32(sV), aKT = smem_u32(sKT);
    const uint32_t aTT = smem_u32(sTT), aPZ = smem_u32(sPZ), aSB = smem_u32(sSB);
    const uint32_t aDB = smem_u32(sDB);

    for (int64_t c = 0; c < nchunks && !failed; ++c) {
        const int64_t tc0 = t0 + c * kC;
        const int Lc = (int)((L - c * kC) < kC ? (L - c * kC) : kC);

        // (1) TMA: K and Q of the q/k head, V columns of this slice.
        if (tid == 0) {
            mbar_arrive_expect_tx(&bar_load, 2 * 2 * 8192 + (NV / 64) * 8192);
#pragma unroll
            for (int r = 0; r < 2; ++r) {
                tma_load_3d(sKQW + r * PL::kRegion, &p.tm_k, r * 64, hq, (int)tc0, &bar_load);
                tma_load_3d(sKQW + r * PL::kRegion + 8192, &p.tm_q, r * 64, hq, (int)tc0, &bar_load);
            }
#pragma unroll
            for (int r = 0; r < NV / 64; ++r)
                tma_load_3d(sV + r * 8192, &p.tm_v, v0 + r * 64, h, (int)tc0, &bar_load);
        }
        // (2) Gates and their within-chunk prefix sum (threads 0-63 = tokens).
        float gsum = 0.f;
        if (tid < kC) {
            float g = 0.f, be = 0.f;
            if (tid < Lc) {
                const size_t gi = (size_t)(tc0 + tid) * p.h_v + h;
                g = decay_f(IoType<IO>::ld(ga + gi), A_log, dt_bias);
                be = sigmoid_f(IoType<IO>::ld(gb + gi));
            }
            gsum = g;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const float y = __shfl_up_sync(0xffffffffu, gsum, off);
                if (lane >= off) gsum += y;
            }
            if (lane == 31) s_wsum[warp] = gsum;
            sBeta[tid] = be;
        }
        __syncthreads();
        if (tid < kC) sG[tid] = gsum + (warp == 1 ? s_wsum[0] : 0.f);
        __syncthreads();
        const float GC = sG[kC - 1];
        if (tid < kC) {
            sGam[tid] = expf(sG[tid]);
            sKf[tid] = expf(GC - sG[tid]);
        }
        const bool ok_load = mbar_wait(&bar_load, ph_load, kWaitBudget);
        ph_load ^= 1;
        if (__syncthreads_or(!ok_load)) { failed = true; break; }

        // (3) D1 = [K; Q] K^T.
        if (tid == 0) {
            tc_fence_after();
#pragma unroll
            for (int s = 0; s < 8; ++s) {
                const uint32_t off = (s >> 2) * PL::kRegion + (s & 3) * 32;
                mma_f16(tmem + PL::tD1, sw128_desc(aKQW + off, 16, 1024),
                        sw128_desc(aKQW + off, 16, 1024), kIdD1, s > 0);
            }
            mma_commit(&bar_mma);
        }
        // Meanwhile: Ktil = diag(e^{G_C - G_j}) K, same swizzled layout as the K tile.
        for (int e = tid; e < 1024; e += kThreads) {
            const int r = e >> 9, j = (e >> 3) & 63, ch = e & 7;
            const uint32_t off = sw128_offset(j, ch);
            const uint4 u = *reinterpret_cast<const uint4 *>(sKQW + r * PL::kRegion + off);
            const float f = sKf[j];
            float x[8];
            const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const float2 t = Pack<IO>::unpack(w[q]);
                x[2 * q] = t.x * f;
                x[2 * q + 1] = t.y * f;
            }
            *reinterpret_cast<uint4 *>(sKT + r * 8192 + off) = pack8<IO>(x);
        }
        fence_async_smem();
        bool ok = mbar_wait(&bar_mma, ph_mma, kWaitBudget);
        ph_mma ^= 1;
        tc_fence_after();

        // (4) A from k.k (lanes 0-63), P from q.k (lanes 64-127); each half-warp group
        //     takes 32 of the 64 columns.
        {
            uint32_t r[32];
            tmem_ld32(tmem + lane_base + PL::tD1 + 32 * half, r);
            tmem_ld_wait();
            if (quarter < 2) {
                const int i = row;
                const float Gi = sG[i], bi = sBeta[i];
#pragma unroll
                for (int jj = 0; jj < 32; ++jj) {
                    const int j = 32 * half + jj;
                    As[i * 65 + j] = (j < i) ? bi * __expf(Gi - sG[j]) * __uint_as_float(r[jj]) : 0.f;
                }
            } else {
                const int i = row - 64;
                const float Gi = sG[i];
#pragma unroll
                for (int q8 = 0; q8 < 4; ++q8) {
                    float x[8];
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        const int j = 32 * half + 8 * q8 + e;
                        x[e] = (j <= i) ? p.scale * __expf(Gi - sG[j]) * __uint_as_float(r[8 * q8 + e])
                                        : 0.f;
                    }
                    *reinterpret_cast<uint4 *>(sPZ + sw128_offset(i, 4 * half + q8)) = pack8<IO>(x);
                }
            }
        }
        fence_async_smem();
        if (__syncthreads_or(!ok)) { failed = true; break; }

        // (5) T = (I + A)^-1, then [T'; T''] in the I/O type, K-major.
        invert_unit_lower_64(As, Ts, sX, tid);
        for (int e = tid; e < 128 * 8; e += kThreads) {
            const int R = e >> 3, ch = e & 7, i = R & 63;
            float x[8];
#pragma unroll
            for (int q = 0; q < 8; ++q) {
                const int j = 8 * ch + q;
                const float f = (R < 64) ? sBeta[j] * sGam[j] : sBeta[j];
                x[q] = (j <= i) ? Ts[i * 65 + j] * f : 0.f;
            }
            *reinterpret_cast<uint4 *>(sTT + sw128_offset(R, ch)) = pack8<IO>(x);
        }
        fence_async_smem();
        tc_fence_before();
        __syncthreads();

        // (6) D2 = [T'; T''] K, D3 = [T'; T''] V (B operands MN-major from the TMA tiles).
        if (tid == 0) {
            tc_fence_after();
#pragma unroll
            for (int s = 0; s < 4; ++s) {
                const uint64_t da = sw128_desc(aTT + s * 32, 16, 1024);
                mma_f16(tmem + PL::tD24, da, sw128_desc(aKQW + s * 2048, PL::kRegion, 1024), kIdD2,
                        s > 0);
                mma_f16(tmem + PL::tD35, da, sw128_desc(aV + s * 2048, 8192, 1024), kIdNV, s > 0);
            }
            mma_commit(&bar_mma);
        }
        // Meanwhile: S0 (TMEM) -> bf16 B operand (MN-major: row = d_k index), then
        // DS <- gamma_C * S0, to which the chunk's K^T Delta is added below.
        {
            const float gC = expf(GC);
#pragma unroll
            for (int c0 = 0; c0 < HALF; c0 += 32) {
                const int col = half * HALF + c0;           // within the slice
                uint32_t r[32];
                tmem_ld32(tmem + lane_base + PL::tDS + col, r);
                tmem_ld_wait();
                float x[32];
#pragma unroll
                for (int j = 0; j < 32; ++j) x[j] = __uint_as_float(r[j]);
                uint8_t *dst = sSB + (col >> 6) * 16384;
#pragma unroll
                for (int q8 = 0; q8 < 4; ++q8)
                    *reinterpret_cast<uint4 *>(dst + sw128_offset(row, ((col & 63) >> 3) + q8)) =
                        pack8<IO>(x + 8 * q8);
#pragma unroll
                for (int j = 0; j < 32; ++j) r[j] = __float_as_uint(x[j] * gC);
                tmem_st32(tmem + lane_base + PL::tDS + col, r);
            }
            tmem_st_wait();
        }
        fence_async_smem();
        ok = mbar_wait(&bar_mma, ph_mma, kWaitBudget);
        ph_mma ^= 1;
        tc_fence_after();

        // (7) W (lanes 0-63 of D2) -> rows 128-191 of the K|Q|W regions.
        if (quarter < 2) {
#pragma unroll
            for (int c0 = 0; c0 < 64; c0 += 32) {
                uint32_t r[32];
                tmem_ld32(tmem + lane_base + PL::tD24 + 64 * half + c0, r);
                tmem_ld_wait();
                float x[32];
#pragma unroll
                for (int j = 0; j < 32; ++j) x[j] = __uint_as_float(r[j]);
#pragma unroll
                for (int q8 = 0; q8 < 4; ++q8)
                    *reinterpret_cast<uint4 *>(sKQW + half * PL::kRegion +
                                               sw128_offset(128 + row, (c0 >> 3) + q8)) =
                        pack8<IO>(x + 8 * q8);
            }
        }
        fence_async_smem();
        tc_fence_before();
        if (__syncthreads_or(!ok)) { failed = true; break; }

        // (8) D4 = [Q; W] S0.
        if (tid == 0) {
            tc_fence_after();
#pragma unroll
            for (int s = 0; s < 8; ++s) {
                const uint32_t off = (s >> 2) * PL::kRegion + 8192 + (s & 3) * 32;
                mma_f16(tmem + PL::tD24, sw128_desc(aKQW + off, 16, 1024),
                        sw128_desc(aSB + s * 2048, 16384, 1024), kIdNV, s > 0);
            }
            mma_commit(&bar_mma);
        }
        ok = mbar_wait(&bar_mma, ph_mma, kWaitBudget);
        ph_mma ^= 1;
        tc_fence_after();

        // (9) Delta = U - W S0 (lanes 64-127), written MN-major (row = token).
        if (quarter >= 2) {
            const int j = row - 64;
#pragma unroll
            for (int c0 = 0; c0 < HALF; c0 += 32) {
                const int col = half * HALF + c0;
                uint32_t ws[32], u[32];
                tmem_ld32(tmem + lane_base + PL::tD24 + col, ws);
                tmem_ld32(tmem + lane_base + PL::tD35 + col, u);
                tmem_ld_wait();
                float x[32];
#pragma unroll
                for (int e = 0; e < 32; ++e) x[e] = __uint_as_float(u[e]) - __uint_as_float(ws[e]);
                uint8_t *dst = sDB + (col >> 6) * 8192;
#pragma unroll
                for (int q8 = 0; q8 < 4; ++q8)
                    *reinterpret_cast<uint4 *>(dst + sw128_offset(j, ((col & 63) >> 3) + q8)) =
                        pack8<IO>(x + 8 * q8);
            }
        }
        fence_async_smem();
        tc_fence_before();
        if (__syncthreads_or(!ok)) { failed = true; break; }

        // (10) D5 = [P; 0] Delta;  DS += Ktil^T Delta.
        if (tid == 0) {
            tc_fence_after();
#pragma unroll
            for (int s = 0; s < 4; ++s) {
                const uint64_t db = sw128_desc(aDB + s * 2048, 8192, 1024);
                mma_f16(tmem + PL::tD35, sw128_desc(aPZ + s * 32, 16, 1024), db, kIdNV, s > 0);
                mma_f16(tmem + PL::tDS, sw128_desc(aKT + s * 2048, 8192, 1024), db, kIdDS, 1u);
            }
            mma_commit(&bar_mma);
        }
        ok = mbar_wait(&bar_mma, ph_mma, kWaitBudget);
        ph_mma ^= 1;
        tc_fence_after();

        // (11) o_i = scale gamma_i (Q S0)_i + (P Delta)_i for the chunk's valid rows.
        if (quarter < 2) {
            const int i = row;
            const float f = p.scale * sGam[i];
#pragma unroll
            for (int c0 = 0; c0 < HALF; c0 += 32) {
                const int col = half * HALF + c0;
                uint32_t qs[32], pd[32];
                tmem_ld32(tmem + lane_base + PL::tD24 + col, qs);
                tmem_ld32(tmem + lane_base + PL::tD35 + col, pd);
                tmem_ld_wait();
                if (i < Lc) {
                    float x[32];
#pragma unroll
                    for (int e = 0; e < 32; ++e)
                        x[e] = fmaf(f, __uint_as_float(qs[e]), __uint_as_float(pd[e]));
                    uint4 *dst = reinterpret_cast<uint4 *>(
                        go + ((size_t)(tc0 + i) * p.h_v + h) * kDK + v0 + col);
#pragma unroll
                    for (int q8 = 0; q8 < 4; ++q8) dst[q8] = pack8<IO>(x + 8 * q8);
                }
            }
        }
        tc_fence_before();
        if (__syncthreads_or(!ok)) { failed = true; break; }
    }

    if (failed) {
        if (tid == 0) atomicOr(p.status, kDevTimeout);
        // Let any MMA still in flight drain (bounded) before TMEM is released.
        mbar_wait(&bar_mma, ph_mma, kWaitBudget);
    } else {
        // Final state: DS -> state_out (fp32).
#pragma unroll
        for (int c0 = 0; c0 < HALF; c0 += 32) {
            const int col = half * HALF + c0;
            uint32_t r[32];
            tmem_ld32(tmem + lane_base + PL::tDS + col, r);
            tmem_ld_wait();
            float4 *dst = reinterpret_cast<float4 *>(p.state_out + sbase + (size_t)row * kDK + v0 + col);
#pragma unroll
            for (int q4 = 0; q4 < 8; ++q4)
                dst[q4] = make_float4(__uint_as_float(r[4 * q4]), __uint_as_float(r[4 * q4 + 1]),
                                      __uint_as_float(r[4 * q4 + 2]), __uint_as_float(r[4 * q4 + 3]));
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

// ------------------------------------------------------------------ host side

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static bool tried = false;
    if (!tried) {
        tried = true;
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
    }
    return fn;
}

// 3-D map over a [tokens][heads][128] tensor with 64 x 1 x 64 boxes, 128-byte swizzle.
bool make_map(CUtensorMap *m, const void *base, gdn_dtype io, int heads, int64_t tokens) {
    auto fn = encode_fn();
    if (fn == nullptr) return false;
    const cuuint64_t dims[3] = {(cuuint64_t)kDK, (cuuint64_t)heads, (cuuint64_t)tokens};
    const cuuint64_t strides[2] = {(cuuint64_t)kDK * 2, (cuuint64_t)kDK * 2 * heads};
    const cuuint32_t box[3] = {64, 1, (cuuint32_t)kC};
    const cuuint32_t estr[3] = {1, 1, 1};
    const CUresult r = fn(m, io == GDN_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16,
                          3, const_cast<void *>(base), dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

template <typename IO, int NV>
cudaError_t launch_typed(const TcParams &tp, int64_t units, cudaStream_t stream) {
    static bool configured = false;
    if (!configured) {
        cudaError_t e = cudaFuncSetAttribute(prefill_tc_kernel<IO, NV>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             Plan<NV>::kAlloc);
        if (e != cudaSuccess) return e;
        configured = true;
    }
    const int64_t blocks = units * (kDK / NV);
    prefill_tc_kernel<IO, NV><<<(unsigned)blocks, kThreads, Plan<NV>::kAlloc, stream>>>(tp);
    return cudaGetLastError();
}

}  // namespace

bool prefill_tc_supported(const ScanParams &p, gdn_dtype io, int64_t total_tokens) {
    if (io != GDN_BF16 && io != GDN_F16) return false;
    if (p.d_k != kDK || p.d_v != kDK) return false;
    if (total_tokens <= 0 || total_tokens > 0x7fffff00LL) return false;
    const void *ptrs[] = {p.q, p.k, p.v, p.o};
    for (const void *ptr : ptrs)
        if (reinterpret_cast<uintptr_t>(ptr) % 16 != 0) return false;
    if ((int64_t)p.num_seqs * p.h_v * 2 > 0x7fffffffLL) return false;
    return encode_fn() != nullptr;
}

int prefill_tc_columns(const ScanParams &p) {
    // Few (sequence, head) units: split the columns to put more CTAs on the SMs.
    return ((int64_t)p.num_seqs * p.h_v >= 120) ? 128 : 64;
}

cudaError_t launch_prefill_tc(const ScanParams &p, gdn_dtype io, int64_t total_tokens, int nv,
                              cudaStream_t stream) {
    TcParams tp;
    memset(&tp, 0, sizeof(tp));
    if (!make_map(&tp.tm_q, p.q, io, p.h_qk, total_tokens) ||
        !make_map(&tp.tm_k, p.k, io, p.h_qk, total_tokens) ||
        !make_map(&tp.tm_v, p.v, io, p.h_v, total_tokens))
        return cudaErrorInvalidValue;
    tp.a = p.a; tp.b = p.b; tp.A_log = p.A_log; tp.dt_bias = p.dt_bias;
    tp.state_in = p.state_in; tp.state_out = p.state_out; tp.o = p.o;
    tp.cu_seqlens = p.cu_seqlens; tp.seqlen = p.seqlen; tp.num_seqs = p.num_seqs;
    tp.h_qk = p.h_qk; tp.h_v = p.h_v; tp.scale = p.scale; tp.status = p.status;
    const int64_t units = (int64_t)p.num_seqs * p.h_v;
    if (io == GDN_BF16)
        return nv == 64 ? launch_typed<__nv_bfloat16, 64>(tp, units, stream)
                        : launch_typed<__nv_bfloat16, 128>(tp, units, stream);
    return nv == 64 ? launch_typed<__half, 64>(tp, units, stream)
                    : launch_typed<__half, 128>(tp, units, stream);
}

}  // namespace gdn
