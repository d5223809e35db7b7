// prefill_tc.cu -- chunked gated delta-rule prefill on the tcgen05 tensor cores.
//
// What it computes is the recurrence of onnx-runtime-ep-cuda 0.1.0-dev.6,
// src/kernels/linear_attention.rs (`linear_attention_core`, Steps 1-4), re-associated
// over chunks of C = 64 tokens so that the work becomes dense contractions.  With
// S0 the state entering a chunk, G_i = g_1 + ... + g_i and gamma_i = e^{G_i}:
//   A_ij = beta_i e^{G_i-G_j} k_i.k_j (j < i),  T = (I + A)^-1
//   W = T diag(beta gamma) K,   U = T diag(beta) V,   Delta = U - W S0
//   o_i = scale gamma_i q_i^T S0 + sum_{j<=i} scale e^{G_i-G_j} (q_i.k_j) Delta_j
//   S  = gamma_C S0 + K^T diag(e^{G_C-G}) Delta
// The pages run the recurrence one token at a time; this chunked form is a
// re-association of the same sums, exact up to rounding.
//
// One CTA owns one (sequence, value head, half of the 128 state columns) and walks the
// sequence's chunks in order.  Columns of S evolve independently (the page's
// "Parallelization" note), so a half needs only its columns of V, U, Delta and o.
// Its 12 warps split into two roles that run one chunk apart:
//   prep  (warps 0-7)  chunk c+1: gates and their prefix sums, D1 = [K; Q] K^T (tcgen05),
//                      A and P, T = (I + A)^-1 (fp32 diagonal blocks + tf32 warp-MMA
//                      merges), [T'; T''] = [T diag(beta gamma); T diag(beta)],
//                      D2 = [T'; T''] K -> W,  D3 = [T'; T''] V -> U (tcgen05).
//   chain (warps 8-11) chunk c: D4 = [Q; W] S0 (tcgen05), Delta = U - W S0,
//                      D5 = [P; 0] Delta, DS = K^T diag(e^{G_C-G}) Delta (tcgen05),
//                      S = gamma_C S0 + DS with S in fp32 registers, o to HBM.
// K, Q and V arrive by TMA into two stages; the chain refills a stage as soon as its
// last reader is done.  All MMAs use M = 128, so accumulator row r is TMEM lane r:
//   D1 lanes 0-63 K K^T, 64-127 Q K^T;  D2 lanes 0-63 W;  D3 lanes 64-127 U;
//   D4 lanes 0-63 Q S0, 64-127 W S0;  D5 lanes 0-63 P Delta;  DS lanes = d_k rows.
// Rows past the end of a sequence get g = 0 and beta = 0, which makes their T row the
// unit row and their W, U and Delta rows exactly zero, so they change nothing.
#include <cudaTypedefs.h>

#include <type_traits>

#include "gdn_internal.cuh"
#include "tc_ptx.cuh"

namespace gdn {
namespace {

using namespace tc;

constexpr int kC = 64;                 // tokens per chunk
constexpr int kDK = 128;               // d_k = d_v of this path
constexpr int kNV = 64;                // state columns per CTA
constexpr int kPrepThreads = 256, kChainThreads = 128;
constexpr int kThreads = kPrepThreads + kChainThreads;
constexpr uint32_t kBarPrep = 1, kBarChain = 2;
constexpr long long kWaitBudget = 4000000000LL;   // cycles (~2 s) before a wait gives up

struct TcParams {
    CUtensorMap tm_q, tm_k, tm_v, tm_o;
    CUtensorMap tm_a, tm_b;        // gate logits [tokens][h_v], used when gate_tma != 0
    int32_t gate_tma;
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
constexpr int kRegion = 24576;                 // 192 rows x 128 B: K | Q | W for 64 d_k
constexpr int kGates = 2 * kRegion + 8192;     // gate logit tiles a, b: 64 tokens x 8 heads
constexpr int kStage = kGates + 2048;          // + V (64 tokens x 64 columns) + gate tiles
constexpr int OFF_STAGE = 0;                   // two stages
constexpr int OFF_PZ = 2 * kStage;             // two P tiles, 64 x 128 B each
constexpr int OFF_TT = OFF_PZ + 2 * 8192;      // [T'; T''], 128 x 128 B
constexpr int OFF_TTR = OFF_TT + 16384;        // [0; T''] received from the peer CTA
constexpr int OFF_SB = OFF_TTR + 16384;        // S0 in the I/O type, MN-major (d_k rows)
constexpr int OFF_DB0 = OFF_SB + 16384;        // Delta, MN-major (token rows)
constexpr int OFF_DB1 = OFF_DB0 + 8192;        // diag(e^{G_C - G}) Delta
constexpr int OFF_AS = OFF_DB1 + 8192;         // A, then T, fp32 [64][68]
constexpr int kAs = 68;                        // row stride (floats) of A / T
constexpr int kSmemBytes = OFF_AS + 64 * kAs * 4;
constexpr int kSmemAlloc = kSmemBytes + 1024;  // slack for the 1024-byte alignment

// TMEM columns.
constexpr uint32_t TM_D1 = 0, TM_D2 = 64, TM_D3 = 192, TM_D4 = 320, TM_DS = 384;

// Per-chunk gate values the chain needs; sent whole to the peer CTA (16-byte multiple).
struct __align__(16) GateBuf {
    float gam[kC];      // e^{G_i}
    float kf[kC];       // e^{G_C - G_i}
    float gC, pad[3];   // e^{G_C}
};

struct Ctl {
    uint64_t full[2], prep_done[2], chain_done[2], d1, d23, d4, d5;
    uint64_t recv[2], recvd[2], peer_free[2];  // cluster hand-off of the shared chunk prep
    uint32_t tmem;
    int abort;
    float G[kC], beta[kC], E[kC], F[kC], wsum[2];
    GateBuf gb[2];
    float X[4][16][20];                        // warp scratch of the T merges
};
constexpr uint32_t kPeerBytes = 2 * 8192 + 8192 + 8192 + sizeof(GateBuf);

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

// OR-reduction of `pred` over the `count` threads of named barrier `id`.
__device__ __forceinline__ bool bar_any(uint32_t id, uint32_t count, bool pred) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 p, %1, 0;\n\t"
        "bar.red.or.pred q, %2, %3, p;\n\t"
        "selp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"(pred ? 1u : 0u), "r"(id), "r"(count)
        : "memory");
    return r != 0;
}

// Store T[r][c] (scaled by f1 and f2) into [T diag(beta gamma); T diag(beta)].
template <typename IO>
__device__ __forceinline__ void tt_put(uint8_t *tt, int r, int c, float x, float f1, float f2) {
    const uint32_t off = sw128_offset(r, c >> 3) + (c & 7) * 2;
    IoType<IO>::st(reinterpret_cast<IO *>(tt + off), x * f1);
    IoType<IO>::st(reinterpret_cast<IO *>(tt + 8192 + off), x * f2);   // row r + 64
}
template <typename IO>
__device__ __forceinline__ void tt_put2(uint8_t *tt, int r, int c, float x0, float x1,
                                        const float *beta, const float *gam) {
    const uint32_t off = sw128_offset(r, c >> 3) + (c & 7) * 2;
    const float b0 = beta[c], b1 = beta[c + 1];
    *reinterpret_cast<uint32_t *>(tt + off) = Pack<IO>::two(x0 * b0 * gam[c], x1 * b1 * gam[c + 1]);
    *reinterpret_cast<uint32_t *>(tt + 8192 + off) = Pack<IO>::two(x0 * b0, x1 * b1);
}

// A 16x16 block of a matrix in shared memory: element (r, c) at p[r * rs + c * cs].
struct Blk {
    float *p;
    int rs, cs;
    __device__ __forceinline__ float at(int r, int c) const { return p[r * rs + c * cs]; }
};

// acc (16x16 fp32, as two 16x8 halves) += X * Y for 16x16 blocks, with tf32 warp MMAs.
__device__ __forceinline__ void block_mma(float (&acc)[2][4], const Blk &x, const Blk &y, int g,
                                          int t) {
#pragma unroll
    for (int kh = 0; kh < 2; ++kh) {
        const uint32_t a[4] = {to_tf32(x.at(g, 8 * kh + t)), to_tf32(x.at(g + 8, 8 * kh + t)),
                               to_tf32(x.at(g, 8 * kh + t + 4)), to_tf32(x.at(g + 8, 8 * kh + t + 4))};
#pragma unroll
        for (int nh = 0; nh < 2; ++nh) {
            const uint32_t bb[2] = {to_tf32(y.at(8 * kh + t, 8 * nh + g)),
                                    to_tf32(y.at(8 * kh + t + 4, 8 * nh + g))};
            mma_tf32_16x8x8(acc[nh], a, bb);
        }
    }
}

__device__ __forceinline__ void block_store(const Blk &d, const float (&acc)[2][4], float sgn, int g,
                                            int t) {
#pragma unroll
    for (int nh = 0; nh < 2; ++nh) {
        const int c = 8 * nh + 2 * t;
        d.p[g * d.rs + c * d.cs] = sgn * acc[nh][0];
        d.p[g * d.rs + (c + 1) * d.cs] = sgn * acc[nh][1];
        d.p[(g + 8) * d.rs + c * d.cs] = sgn * acc[nh][2];
        d.p[(g + 8) * d.rs + (c + 1) * d.cs] = sgn * acc[nh][3];
    }
}

// T = (I + A)^-1 for the strictly-lower 64 x 64 A in As (prep threads only), written
// straight into the K-major operand tile [T diag(beta gamma); T diag(beta)].
//  1. The diagonal 16x16 blocks T_bb = (I + A_bb)^-1 by forward substitution in fp32,
//     one thread per column, kept in place in As.
//  2. 16 -> 32: T_10 = -T_11 A_10 T_00 and T_32 = -T_33 A_32 T_22 (one warp each).
//  3. 32 -> 64: Y = A_[23][01] T_[01][01], then T_[23][01] = -T_[23][23] Y, one 16x16
//     block per warp.
// Blocks below the diagonal use tf32 warp MMAs; each is also kept transposed in the
// unused upper block of As (T_ij at As[16 j + c][16 i + r]), so A below the diagonal
// is never overwritten while it is still read.
template <typename IO>
__device__ void invert_chunk(float *As, float (*X)[16][20], uint8_t *tt, const float *beta,
                             const float *gam, int pt) {
    if (pt < 64) {
        const int o = (pt >> 4) * 16, j = pt & 15, cj = o + j;
        float x[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            float acc = 0.f;
#pragma unroll
            for (int l = 0; l < i; ++l) acc = fmaf(As[(o + i) * kAs + o + l], x[l], acc);
            x[i] = (i < j) ? 0.f : ((i == j) ? 1.f : -acc);
        }
        __syncwarp();
        const float f2 = beta[cj], f1 = f2 * gam[cj];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            As[(o + i) * kAs + cj] = x[i];
            tt_put<IO>(tt, o + i, cj, x[i], f1, f2);
        }
    }
    named_bar(kBarPrep, kPrepThreads);
    const int w = pt >> 5, lane = pt & 31, g = lane >> 2, t = lane & 3;
    auto diag = [&](int b) { return Blk{As + 16 * b * kAs + 16 * b, kAs, 1}; };
    auto low = [&](int i, int j) { return Blk{As + 16 * i * kAs + 16 * j, kAs, 1}; };  // A_ij
    auto tlo = [&](int i, int j) { return Blk{As + 16 * j * kAs + 16 * i, 1, kAs}; };  // T_ij
    auto scratch = [&](int k) { return Blk{&X[k][0][0], 20, 1}; };
    auto emit = [&](int i, int j, const float (&acc)[2][4]) {   // T_ij = -acc
        block_store(tlo(i, j), acc, -1.f, g, t);
#pragma unroll
        for (int nh = 0; nh < 2; ++nh) {
            const int c = 16 * j + 8 * nh + 2 * t, r = 16 * i + g;
            tt_put2<IO>(tt, r, c, -acc[nh][0], -acc[nh][1], beta, gam);
            tt_put2<IO>(tt, r + 8, c, -acc[nh][2], -acc[nh][3], beta, gam);
        }
    };
    if (w < 2) {                                    // 16 -> 32
        const int hi = 2 * w + 1, lo = 2 * w;       // (1, 0) or (3, 2)
        float acc[2][4] = {};
        block_mma(acc, low(hi, lo), diag(lo), g, t);
        block_store(scratch(w), acc, 1.f, g, t);
        __syncwarp();
        float res[2][4] = {};
        block_mma(res, diag(hi), scratch(w), g, t);
        emit(hi, lo, res);
    }
    named_bar(kBarPrep, kPrepThreads);
    const int bi = 2 + (w >> 1), bj = w & 1;        // this warp's block of T_[23][01]
    if (w < 4) {                                    // Y = A_[23][01] T_[01][01]
        float acc[2][4] = {};
        if (bj == 0) {
            block_mma(acc, low(bi, 0), diag(0), g, t);
            block_mma(acc, low(bi, 1), tlo(1, 0), g, t);
        } else {
            block_mma(acc, low(bi, 1), diag(1), g, t);
        }
        block_store(scratch(w), acc, 1.f, g, t);
    }
    named_bar(kBarPrep, kPrepThreads);
    if (w < 4) {                                    // T_[23][01] = -T_[23][23] Y
        float res[2][4] = {};
        if (bi == 2) {
            block_mma(res, diag(2), scratch(bj), g, t);
        } else {
            block_mma(res, tlo(3, 2), scratch(bj), g, t);
            block_mma(res, diag(3), scratch(2 + bj), g, t);
        }
        emit(bi, bj, res);
    }
}

template <typename IO>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    prefill_tc_kernel(const __grid_constant__ TcParams p) {
    constexpr bool kBf16 = std::is_same<IO, __nv_bfloat16>::value;
    constexpr uint32_t kIdD1 = idesc_f16(kBf16, 128, 64, false, false);
    constexpr uint32_t kIdD2 = idesc_f16(kBf16, 128, 128, false, true);
    constexpr uint32_t kIdNV = idesc_f16(kBf16, 128, kNV, false, true);
    constexpr uint32_t kIdDS = idesc_f16(kBf16, 128, kNV, true, true);

    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                              ~static_cast<uintptr_t>(1023));
    __shared__ Ctl ctl;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const uint32_t rank = cluster_ctarank(), peer = rank ^ 1u;   // rank = column half
    const int h = (blockIdx.x >> 1) % p.h_v;
    const int64_t n = (int64_t)(blockIdx.x >> 1) / p.h_v;
    const int hq = h / (p.h_v / p.h_qk);
    const int v0 = (int)rank * kNV;

    // Both CTAs of a cluster share (n, h), so they leave here together.
    int64_t t0, t1;
    if (!seq_range(p.cu_seqlens, p.seqlen, p.num_seqs, p.status, n, t0, t1)) return;
    const int64_t L = t1 - t0;
    const int nchunks = (int)((L + kC - 1) / kC);

    float *const As = reinterpret_cast<float *>(sm + OFF_AS);
    const uint32_t aStage = smem_u32(sm + OFF_STAGE), aPZ = smem_u32(sm + OFF_PZ);
    const uint32_t aTT = smem_u32(sm + OFF_TT), aTTR = smem_u32(sm + OFF_TTR);
    const uint32_t aSB = smem_u32(sm + OFF_SB);
    const uint32_t aDB0 = smem_u32(sm + OFF_DB0), aDB1 = smem_u32(sm + OFF_DB1);

    if (warp == 0) {
        tmem_alloc(&ctl.tmem, 512);
        tmem_relinquish();
    }
    if (tid == 0) {
        for (int i = 0; i < 2; ++i) {
            mbar_init(&ctl.full[i], 1);
            mbar_init(&ctl.prep_done[i], 1);
            mbar_init(&ctl.chain_done[i], 1);
            mbar_init(&ctl.recv[i], 1);
            mbar_init(&ctl.recvd[i], 1);
            mbar_init(&ctl.peer_free[i], 1);
        }
        mbar_init(&ctl.d1, 1);
        mbar_init(&ctl.d23, 1);
        mbar_init(&ctl.d4, 1);
        mbar_init(&ctl.d5, 1);
        ctl.abort = 0;
        fence_mbar_init();
        tma_prefetch_desc(&p.tm_q);
        tma_prefetch_desc(&p.tm_k);
        tma_prefetch_desc(&p.tm_v);
    }
    // Zero the P tiles, [T'; T''] (its blocks above the diagonal stay zero) and the
    // receive tile [0; T''], so every operand row an MMA reads is finite.
    for (int e = tid; e < (2 * 8192 + 2 * 16384) / 16; e += kThreads)
        *reinterpret_cast<uint4 *>(sm + OFF_PZ + 16 * e) = make_uint4(0, 0, 0, 0);
    fence_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    cluster_sync();   // the peer's barriers exist before any remote arrive or copy
    const uint32_t tmem = ctl.tmem;
    const uint32_t lane_base = static_cast<uint32_t>(32 * (warp & 3)) << 16;
    const size_t sbase = ((size_t)n * p.h_v + h) * kDK * kDK;
    auto owns = [&](int c) { return (uint32_t)(c & 1) == rank; };

    // TMA of chunk c into stage c & 1: K, Q and V always; the gate logits only for the
    // chunks this CTA preps.
    auto issue_stage = [&](int c) {
        const int s = c & 1;
        const bool own = owns(c);
        uint8_t *st = sm + OFF_STAGE + s * kStage;
        const int tok = (int)(t0 + (int64_t)c * kC);
        const uint32_t tx = 2 * 2 * 8192 + 8192 + ((own && p.gate_tma) ? 2048 : 0);
        mbar_arrive_expect_tx(&ctl.full[s], tx);
#pragma unroll
        for (int r = 0; r < 2; ++r) {
            tma_load_3d(st + r * kRegion, &p.tm_k, r * 64, hq, tok, &ctl.full[s]);
            tma_load_3d(st + r * kRegion + 8192, &p.tm_q, r * 64, hq, tok, &ctl.full[s]);
        }
        tma_load_3d(st + 2 * kRegion, &p.tm_v, v0, h, tok, &ctl.full[s]);
        if (own && p.gate_tma) {
            tma_load_2d(st + kGates, &p.tm_a, h & ~7, tok, &ctl.full[s]);
            tma_load_2d(st + kGates + 1024, &p.tm_b, h & ~7, tok, &ctl.full[s]);
        }
    };

    if (tid < kPrepThreads) {
        // ============================================================== prep role
        // Preps the chunks c with c % 2 == rank, for this CTA's chain and the peer's.
        const int pt = tid;
        const int q = warp & 3, hf = warp >> 2;    // TMEM lane quarter, column half
        const IO *ga = static_cast<const IO *>(p.a);
        const IO *gb = static_cast<const IO *>(p.b);
        const float A_log = p.A_log[h], dt_bias = p.dt_bias[h];
        bool failed = false;
        for (int c = (int)rank; c < nchunks; c += 2) {
            const int b = c & 1, s = c & 1;
            const int64_t tc0 = t0 + (int64_t)c * kC;
            const int Lc = (int)((L - (int64_t)c * kC) < kC ? (L - (int64_t)c * kC) : kC);
            GateBuf &gbuf = ctl.gb[b];
            bool ok = true;
            if (c >= 2) {
                ok = mbar_wait(&ctl.chain_done[b], ((c >> 1) - 1) & 1, kWaitBudget);
                if (ok) ok = mbar_wait(&ctl.recvd[b], ((c >> 1) - 1) & 1, kWaitBudget);
            }
            if (ok) ok = mbar_wait(&ctl.full[s], (c >> 1) & 1, kWaitBudget);
            if (bar_any(kBarPrep, kPrepThreads, !ok || *(volatile int *)&ctl.abort)) { failed = true; break; }

            // D1 = [K; Q] K^T (the stage has landed); the gates are computed meanwhile.
            if (pt == 0) {
                tc_fence_after();
                const uint32_t st = aStage + s * kStage;
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                    const uint32_t off = (k >> 2) * kRegion + (k & 3) * 32;
                    mma_f16(tmem + TM_D1, sw128_desc(st + off, 16, 1024),
                            sw128_desc(st + off, 16, 1024), kIdD1, k > 0);
                }
                mma_commit(&ctl.d1);
            }

            // Gates and prefix sums (threads 0-63 = tokens of the chunk).
            float gsum = 0.f, be = 0.f;
            if (pt < kC) {
                float ra = 0.f, rb = 0.f;
                if (p.gate_tma) {
                    const IO *gt = reinterpret_cast<const IO *>(sm + OFF_STAGE + s * kStage + kGates);
                    ra = IoType<IO>::ld(gt + pt * 8 + (h & 7));
                    rb = IoType<IO>::ld(gt + 512 + pt * 8 + (h & 7));
                } else if (pt < Lc) {
                    ra = IoType<IO>::ld(ga + (size_t)(tc0 + pt) * p.h_v + h);
                    rb = IoType<IO>::ld(gb + (size_t)(tc0 + pt) * p.h_v + h);
                }
                if (pt < Lc) {
                    gsum = decay_f(ra, A_log, dt_bias);
                    be = sigmoid_f(rb);
                }
#pragma unroll
                for (int off = 1; off < 32; off <<= 1) {
                    const float y = __shfl_up_sync(0xffffffffu, gsum, off);
                    if (lane >= off) gsum += y;
                }
                if (lane == 31) ctl.wsum[warp] = gsum;
            }
            named_bar(kBarPrep, kPrepThreads);
            if (pt < kC) {
                ctl.G[pt] = gsum + (warp == 1 ? ctl.wsum[0] : 0.f);
                ctl.beta[pt] = be;
            }
            named_bar(kBarPrep, kPrepThreads);
            const float GC = ctl.G[kC - 1], Gm = ctl.G[31];
            const bool safe = (ctl.G[0] - GC) <= 80.f;   // e^{G_i - G_m} e^{G_m - G_j} cannot overflow
            if (pt < kC) {
                const float G = ctl.G[pt];
                gbuf.gam[pt] = __expf(G);
                gbuf.kf[pt] = __expf(GC - G);
                ctl.E[pt] = __expf(G - Gm);
                ctl.F[pt] = __expf(Gm - G);
                if (pt == 0) gbuf.gC = __expf(GC);
            }
            named_bar(kBarPrep, kPrepThreads);   // E, F, gamma visible to every prep warp
            ok = mbar_wait(&ctl.d1, (c >> 1) & 1, kWaitBudget);
            tc_fence_after();

            // A rows (lanes 0-63, fp32) and P rows (lanes 64-127, I/O type); each column
            // half of the prep warps takes 32 of the 64 columns.
            {
                uint32_t r[32];
                tmem_ld32(tmem + lane_base + TM_D1 + 32 * hf, r);
                tmem_ld_wait();
                const int i = (32 * q + lane) & 63;
                const float Ei = ctl.E[i], Gi = ctl.G[i];
                if (q < 2) {
                    const float bi = ctl.beta[i];
#pragma unroll
                    for (int j4 = 0; j4 < 8; ++j4) {
                        float x[4];
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const int j = 32 * hf + 4 * j4 + e;
                            const float d = safe ? Ei * ctl.F[j] : __expf(Gi - ctl.G[j]);
                            x[e] = (j < i) ? bi * d * __uint_as_float(r[4 * j4 + e]) : 0.f;
                        }
                        *reinterpret_cast<float4 *>(As + i * kAs + 32 * hf + 4 * j4) =
                            make_float4(x[0], x[1], x[2], x[3]);
                    }
                } else {
                    uint8_t *pz = sm + OFF_PZ + b * 8192;
#pragma unroll
                    for (int q8 = 0; q8 < 4; ++q8) {
                        float x[8];
#pragma unroll
                        for (int e = 0; e < 8; ++e) {
                            const int j = 32 * hf + 8 * q8 + e;
                            const float d = safe ? Ei * ctl.F[j] : __expf(Gi - ctl.G[j]);
                            x[e] = (j <= i) ? p.scale * d * __uint_as_float(r[8 * q8 + e]) : 0.f;
                        }
                        *reinterpret_cast<uint4 *>(pz + sw128_offset(i, 4 * hf + q8)) = pack8<IO>(x);
                    }
                }
            }
            // D1 has read Q: scale the stage's Q rows in place, Q~ = diag(scale gamma) Q,
            // so that [Q~; W] S0 yields the inter-chunk output term directly.
            for (int e = pt; e < 1024; e += kPrepThreads) {
                const int r = e >> 9, row = (e >> 3) & 63, ch = e & 7;
                uint8_t *ptr = sm + OFF_STAGE + s * kStage + r * kRegion + 8192 + sw128_offset(row, ch);
                const uint4 u = *reinterpret_cast<const uint4 *>(ptr);
                const float f = p.scale * gbuf.gam[row];
                const uint32_t w[4] = {u.x, u.y, u.z, u.w};
                float x[8];
#pragma unroll
                for (int k2 = 0; k2 < 4; ++k2) {
                    const float2 t2 = Pack<IO>::unpack(w[k2]);
                    x[2 * k2] = t2.x * f;
                    x[2 * k2 + 1] = t2.y * f;
                }
                *reinterpret_cast<uint4 *>(ptr) = pack8<IO>(x);
            }
            fence_async_smem();
            if (bar_any(kBarPrep, kPrepThreads, !ok)) { failed = true; break; }

            // T = (I + A)^-1, written as [T diag(beta gamma); T diag(beta)] (K-major).
            invert_chunk<IO>(As, ctl.X, sm + OFF_TT, ctl.beta, gbuf.gam, pt);
            fence_async_smem();
            tc_fence_before();
            named_bar(kBarPrep, kPrepThreads);

            // D2 = [T'; T''] K and D3 = [T'; T''] V (B operands MN-major from the stage).
            if (pt == 0) {
                tc_fence_after();
                const uint32_t st = aStage + s * kStage;
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const uint64_t da = sw128_desc(aTT + k * 32, 16, 1024);
                    mma_f16(tmem + TM_D2, da, sw128_desc(st + k * 2048, kRegion, 1024), kIdD2, k > 0);
                    mma_f16(tmem + TM_D3 + 64 * b, da, sw128_desc(st + 2 * kRegion + k * 2048, 8192, 1024),
                            kIdNV, k > 0);
                }
                mma_commit(&ctl.d23);
            }
            ok = mbar_wait(&ctl.d23, (c >> 1) & 1, kWaitBudget);
            tc_fence_after();

            // W (lanes 0-63 of D2) -> rows 128-191 of the stage's K|Q|W regions.
            if (q < 2) {
                const int i = 32 * q + lane;
                uint8_t *reg = sm + OFF_STAGE + s * kStage + hf * kRegion;
#pragma unroll
                for (int c0 = 0; c0 < 64; c0 += 32) {
                    uint32_t r[32];
                    tmem_ld32(tmem + lane_base + TM_D2 + 64 * hf + c0, r);
                    tmem_ld_wait();
                    float x[32];
#pragma unroll
                    for (int e = 0; e < 32; ++e) x[e] = __uint_as_float(r[e]);
#pragma unroll
                    for (int q8 = 0; q8 < 4; ++q8)
                        *reinterpret_cast<uint4 *>(reg + sw128_offset(128 + i, (c0 >> 3) + q8)) =
                            pack8<IO>(x + 8 * q8);
                }
            }
            fence_async_smem();
            tc_fence_before();
            if (bar_any(kBarPrep, kPrepThreads, !ok)) { failed = true; break; }
            if (pt == 0) {
                mbar_arrive(&ctl.prep_done[b]);
                // Hand the chunk to the peer once it has released the previous one:
                // the W rows of both d_k halves, P, T'' and the gate values.
                ok = (c < 2) || mbar_wait(&ctl.peer_free[b], ((c >> 1) - 1) & 1, kWaitBudget);
                if (ok) {
                    const uint32_t rb = mapa_shared(smem_u32(&ctl.recv[b]), peer);
                    uint8_t *st = sm + OFF_STAGE + s * kStage;
#pragma unroll
                    for (int r = 0; r < 2; ++r)
                        bulk_copy_to_cluster(mapa_shared(smem_u32(st + r * kRegion + 16384), peer),
                                             st + r * kRegion + 16384, 8192, rb);
                    bulk_copy_to_cluster(mapa_shared(aPZ + b * 8192, peer), sm + OFF_PZ + b * 8192, 8192, rb);
                    bulk_copy_to_cluster(mapa_shared(aTTR + 8192, peer), sm + OFF_TT + 8192, 8192, rb);
                    bulk_copy_to_cluster(mapa_shared(smem_u32(&gbuf), peer), &gbuf, sizeof(GateBuf), rb);
                }
            }
            if (bar_any(kBarPrep, kPrepThreads, !ok)) { failed = true; break; }
        }
        if (failed && pt == 0) {
            ctl.abort = 1;
            atomicOr(p.status, kDevTimeout);
        }
    } else {
        // ============================================================== chain role
        const int ct = tid - kPrepThreads;         // = TMEM lane = d_k row of S
        const int cw = ct >> 5;
        IO *go = static_cast<IO *>(p.o);
        float S[kNV];
        {
            const float4 *src = reinterpret_cast<const float4 *>(p.state_in + sbase +
                                                                 (size_t)ct * kDK + v0);
#pragma unroll
            for (int q4 = 0; q4 < kNV / 4; ++q4) {
                const float4 f = p.state_in ? src[q4] : make_float4(0.f, 0.f, 0.f, 0.f);
                S[4 * q4] = f.x; S[4 * q4 + 1] = f.y; S[4 * q4 + 2] = f.z; S[4 * q4 + 3] = f.w;
            }
        }
        auto write_sb = [&]() {   // S (fp32 registers) -> MN-major operand tile, row = ct
#pragma unroll
            for (int q8 = 0; q8 < 8; ++q8)
                *reinterpret_cast<uint4 *>(sm + OFF_SB + sw128_offset(ct, q8)) = pack8<IO>(S + 8 * q8);
        };
        write_sb();
        fence_async_smem();
        if (ct == 0) {
            if (nchunks > 0) issue_stage(0);
            if (nchunks > 1) issue_stage(1);
        }
        named_bar(kBarChain, kChainThreads);
        bool failed = false;
        for (int c = 0; c < nchunks; ++c) {
            const int b = c & 1, s = c & 1;
            const bool own = owns(c);
            const int64_t tc0 = t0 + (int64_t)c * kC;
            const int Lc = (int)((L - (int64_t)c * kC) < kC ? (L - (int64_t)c * kC) : kC);
            bool ok;
            if (own) {
                ok = mbar_wait(&ctl.prep_done[b], (c >> 1) & 1, kWaitBudget);
            } else {
                if (ct == 0) mbar_arrive_expect_tx(&ctl.recv[b], kPeerBytes);
                ok = mbar_wait(&ctl.recv[b], (c >> 1) & 1, kWaitBudget);
                if (ok) ok = mbar_wait(&ctl.full[s], (c >> 1) & 1, kWaitBudget);
                if (ok && ct == 0) mbar_arrive_cluster(mapa_shared(smem_u32(&ctl.recvd[b]), peer));
                if (ok) {   // Q~ = diag(scale gamma) Q in place, as the owner did for its copy
                    for (int e = ct; e < 1024; e += kChainThreads) {
                        const int r = e >> 9, row = (e >> 3) & 63, ch = e & 7;
                        uint8_t *ptr = sm + OFF_STAGE + s * kStage + r * kRegion + 8192 +
                                       sw128_offset(row, ch);
                        const uint4 u = *reinterpret_cast<const uint4 *>(ptr);
                        const float f = p.scale * ctl.gb[b].gam[row];
                        const uint32_t w[4] = {u.x, u.y, u.z, u.w};
                        float x[8];
#pragma unroll
                        for (int k2 = 0; k2 < 4; ++k2) {
                            const float2 t2 = Pack<IO>::unpack(w[k2]);
                            x[2 * k2] = t2.x * f;
                            x[2 * k2 + 1] = t2.y * f;
                        }
                        *reinterpret_cast<uint4 *>(ptr) = pack8<IO>(x);
                    }
                    fence_async_smem();
                }
            }
            if (ct == 0) bulk_wait_read();   // the previous output tile (in DB0) has been read
            if (bar_any(kBarChain, kChainThreads, !ok || *(volatile int *)&ctl.abort)) { failed = true; break; }
            tc_fence_after();
            const uint32_t st = aStage + s * kStage;

            // (Received chunks: U = T'' V of this half.)  D4 = [Q~; W] S0.
            if (ct == 0) {
                if (!own) {
#pragma unroll
                    for (int k = 0; k < 4; ++k)
                        mma_f16(tmem + TM_D3 + 64 * b, sw128_desc(aTTR + k * 32, 16, 1024),
                                sw128_desc(st + 2 * kRegion + k * 2048, 8192, 1024), kIdNV, k > 0);
                }
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                    const uint32_t off = (k >> 2) * kRegion + 8192 + (k & 3) * 32;
                    mma_f16(tmem + TM_D4, sw128_desc(st + off, 16, 1024),
                            sw128_desc(aSB + k * 2048, 16384, 1024), kIdNV, k > 0);
                }
                mma_commit(&ctl.d4);
            }
            ok = mbar_wait(&ctl.d4, c & 1, kWaitBudget);
            tc_fence_after();

            // Delta = U - W S0 on lanes 64-127 (token rows), in two versions.
            if (cw >= 2) {
                const int j = ct - 64;
                const float kfj = ctl.gb[b].kf[j];
#pragma unroll
                for (int c0 = 0; c0 < kNV; c0 += 32) {
                    uint32_t ws[32], u[32];
                    tmem_ld32(tmem + lane_base + TM_D4 + c0, ws);
                    tmem_ld32(tmem + lane_base + TM_D3 + 64 * b + c0, u);
                    tmem_ld_wait();
                    float x[32], y[32];
#pragma unroll
                    for (int e = 0; e < 32; ++e) {
                        x[e] = __uint_as_float(u[e]) - __uint_as_float(ws[e]);
                        y[e] = kfj * x[e];
                    }
#pragma unroll
                    for (int q8 = 0; q8 < 4; ++q8) {
                        const uint32_t off = sw128_offset(j, (c0 >> 3) + q8);
                        *reinterpret_cast<uint4 *>(sm + OFF_DB0 + off) = pack8<IO>(x + 8 * q8);
                        *reinterpret_cast<uint4 *>(sm + OFF_DB1 + off) = pack8<IO>(y + 8 * q8);
                    }
                }
            }
            fence_async_smem();
            tc_fence_before();
            if (bar_any(kBarChain, kChainThreads, !ok)) { failed = true; break; }

            // D4[0:64] += P Delta (the A rows past P land in the spent W S0 lanes);
            // DS = K^T diag(e^{G_C - G}) Delta.
            if (ct == 0) {
                tc_fence_after();
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    mma_f16(tmem + TM_D4, sw128_desc(aPZ + b * 8192 + k * 32, 16, 1024),
                            sw128_desc(aDB0 + k * 2048, 8192, 1024), kIdNV, 1u);
                    mma_f16(tmem + TM_DS, sw128_desc(st + k * 2048, kRegion, 1024),
                            sw128_desc(aDB1 + k * 2048, 8192, 1024), kIdDS, k > 0);
                }
                mma_commit(&ctl.d5);
            }
            ok = mbar_wait(&ctl.d5, c & 1, kWaitBudget);
            tc_fence_after();
            // The stage's last readers are done: refill it with chunk c + 2.
            if (ct == 0 && ok && c + 2 < nchunks) issue_stage(c + 2);

            // S = gamma_C S0 + DS (fp32 registers), then the next chunk's operand tile.
            {
                const float gC = ctl.gb[b].gC;
#pragma unroll
                for (int c0 = 0; c0 < kNV; c0 += 32) {
                    uint32_t r[32];
                    tmem_ld32(tmem + lane_base + TM_DS + c0, r);
                    tmem_ld_wait();
#pragma unroll
                    for (int e = 0; e < 32; ++e) S[c0 + e] = fmaf(gC, S[c0 + e], __uint_as_float(r[e]));
                }
                write_sb();
            }
            // o_i = (Q~ S0 + P Delta)_i on lanes 0-63.  A full chunk goes out as one TMA
            // store of a 64 x 64 tile staged in DB0 (free once D4 and DS have read it); a
            // sequence's ragged last chunk is stored row by row so that no row of the next
            // sequence is touched.
            const bool tile_store = (Lc == kC);
            if (cw < 2) {
                const int i = ct;
#pragma unroll
                for (int c0 = 0; c0 < kNV; c0 += 32) {
                    uint32_t r[32];
                    tmem_ld32(tmem + lane_base + TM_D4 + c0, r);
                    tmem_ld_wait();
                    float x[32];
#pragma unroll
                    for (int e = 0; e < 32; ++e) x[e] = __uint_as_float(r[e]);
                    if (tile_store) {
#pragma unroll
                        for (int q8 = 0; q8 < 4; ++q8)
                            *reinterpret_cast<uint4 *>(sm + OFF_DB0 + sw128_offset(i, (c0 >> 3) + q8)) =
                                pack8<IO>(x + 8 * q8);
                    } else if (i < Lc) {
                        uint4 *dst = reinterpret_cast<uint4 *>(
                            go + ((size_t)(tc0 + i) * p.h_v + h) * kDK + v0 + c0);
#pragma unroll
                        for (int q8 = 0; q8 < 4; ++q8) dst[q8] = pack8<IO>(x + 8 * q8);
                    }
                }
            }
            fence_async_smem();
            tc_fence_before();
            if (bar_any(kBarChain, kChainThreads, !ok)) { failed = true; break; }
            if (ct == 0 && tile_store) {
                tma_store_3d(&p.tm_o, sm + OFF_DB0, v0, h, (int)tc0);
                bulk_commit();
            }
            if (ct == 0) {
                if (own) mbar_arrive(&ctl.chain_done[b]);
                else mbar_arrive_cluster(mapa_shared(smem_u32(&ctl.peer_free[b]), peer));
            }
        }
        if (ct == 0) bulk_wait_all();   // the output tiles have reached global memory
        if (failed) {
            if (ct == 0) {
                ctl.abort = 1;
                atomicOr(p.status, kDevTimeout);
            }
        } else {
            float4 *dst = reinterpret_cast<float4 *>(p.state_out + sbase + (size_t)ct * kDK + v0);
#pragma unroll
            for (int q4 = 0; q4 < kNV / 4; ++q4)
                dst[q4] = make_float4(S[4 * q4], S[4 * q4 + 1], S[4 * q4 + 2], S[4 * q4 + 3]);
        }
    }

    tc_fence_before();
    __syncthreads();
    cluster_sync();   // no remote copy or arrive may target a CTA that has exited
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

// 2-D map over the [tokens][h_v] gate logits with 8-head x 64-token boxes.
bool make_gate_map(CUtensorMap *m, const void *base, gdn_dtype io, int h_v, int64_t tokens) {
    auto fn = encode_fn();
    if (fn == nullptr) return false;
    const cuuint64_t dims[2] = {(cuuint64_t)h_v, (cuuint64_t)tokens};
    const cuuint64_t strides[1] = {(cuuint64_t)h_v * 2};
    const cuuint32_t box[2] = {8, (cuuint32_t)kC};
    const cuuint32_t estr[2] = {1, 1};
    const CUresult r = fn(m, io == GDN_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16,
                          2, const_cast<void *>(base), dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                          CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

template <typename IO>
cudaError_t launch_typed(const TcParams &tp, int64_t units, cudaStream_t stream) {
    static bool configured = false;
    if (!configured) {
        cudaError_t e = cudaFuncSetAttribute(prefill_tc_kernel<IO>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemAlloc);
        if (e != cudaSuccess) return e;
        configured = true;
    }
    const int64_t blocks = units * (kDK / kNV);
    prefill_tc_kernel<IO><<<(unsigned)blocks, kThreads, kSmemAlloc, stream>>>(tp);
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

int prefill_tc_columns(const ScanParams &) { return kNV; }

cudaError_t launch_prefill_tc(const ScanParams &p, gdn_dtype io, int64_t total_tokens, int nv,
                              cudaStream_t stream) {
    if (nv != kNV) return cudaErrorInvalidValue;
    TcParams tp;
    memset(&tp, 0, sizeof(tp));
    if (!make_map(&tp.tm_q, p.q, io, p.h_qk, total_tokens) ||
        !make_map(&tp.tm_k, p.k, io, p.h_qk, total_tokens) ||
        !make_map(&tp.tm_v, p.v, io, p.h_v, total_tokens) ||
        !make_map(&tp.tm_o, p.o, io, p.h_v, total_tokens))
        return cudaErrorInvalidValue;
    // Gate logits ride along with each stage's TMA when their rows are 16-byte multiples.
    tp.gate_tma = (p.h_v % 8 == 0 && reinterpret_cast<uintptr_t>(p.a) % 16 == 0 &&
                   reinterpret_cast<uintptr_t>(p.b) % 16 == 0 &&
                   make_gate_map(&tp.tm_a, p.a, io, p.h_v, total_tokens) &&
                   make_gate_map(&tp.tm_b, p.b, io, p.h_v, total_tokens))
                      ? 1 : 0;
    tp.a = p.a; tp.b = p.b; tp.A_log = p.A_log; tp.dt_bias = p.dt_bias;
    tp.state_in = p.state_in; tp.state_out = p.state_out; tp.o = p.o;
    tp.cu_seqlens = p.cu_seqlens; tp.seqlen = p.seqlen; tp.num_seqs = p.num_seqs;
    tp.h_qk = p.h_qk; tp.h_v = p.h_v; tp.scale = p.scale; tp.status = p.status;
    const int64_t units = (int64_t)p.num_seqs * p.h_v;
    if (io == GDN_BF16) return launch_typed<__nv_bfloat16>(tp, units, stream);
    return launch_typed<__half>(tp, units, stream);
}

}  // namespace gdn
