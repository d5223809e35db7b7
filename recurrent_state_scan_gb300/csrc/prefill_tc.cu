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
// Two kernels, stream-ordered:
//  * gdn_chunk_prep -- persistent CTAs, three to an SM, walk the (chunk, value head)
//    items: everything that does not depend on the state.  Gates and their prefix sums,
//    D1 = [K; Q] K^T (tcgen05), A and P, T = (I + A)^-1 (fp32 diagonal blocks, tf32
//    warp-MMA merges), D2 = [T'; T''] K -> W and D3 = [T'; T''] V -> U (tcgen05), and
//    for the scan's lookahead M = W K_prev^T diag(e^{G_C - G}) against the previous
//    chunk's keys.  It writes one workspace record per (chunk, head): images of W, [P; M],
//    U and the gate values, laid out exactly as the scan loads them (the scan applies
//    gamma_C of the previous chunk to the W S rows in fp32).
//  * gdn_chunk_scan -- one CTA per (sequence, value head, half of the 128 state columns),
//    walking the sequence's chunks in order: D4 = [Q; W] S0 (tcgen05),
//    Delta = U - W S0, DS = K^T diag(e^{G_C-G}) Delta and X = [P; M] Delta (tcgen05),
//    S = gamma_C S0 + DS with S in fp32 registers, o = scale gamma (Q S0) + P Delta by
//    TMA store.  Records, Q and K arrive by bulk copy / TMA into two stages, one chunk
//    ahead.
// Columns of S evolve independently (the page's "Parallelization" note), so a column
// half needs only its half of U and Delta.  All MMAs use M = 128, so accumulator row r
// is TMEM lane r.  Rows past the end of a sequence get g = 0 and beta = 0, which makes
// their T row the unit row and their W, U and Delta rows exactly zero.
#include <cudaTypedefs.h>

#include <mutex>
#include <type_traits>

#include "gdn_internal.cuh"
#include "tc_ptx.cuh"

namespace gdn {
namespace {

using namespace tc;

constexpr int kC = 64;                 // tokens per chunk
constexpr int kDK = 128;               // d_k = d_v of this path
constexpr int kNV = 64;                // state columns per scan CTA
constexpr int kPrepThreads = 256;
constexpr uint32_t kBarPrep = 1;
constexpr long long kWaitBudget = 4000000000LL;   // cycles (~2 s) before a wait gives up
constexpr int kAs = 68;                // row stride (floats) of the fp32 A / T tile

// Workspace record of one (chunk c, value head): shared-memory images for the scan.
// Rows marked (c + 1) are written by the prep of the next chunk of the same sequence.
constexpr int REC_W = 0;               // W_{c+1}: 2 d_k halves x 64 rows x 128 B
constexpr int REC_PM = 16384;          // [P_c rows | M_{c+1} rows], 128 x 128 B
constexpr int REC_U = 32768;           // U_c: 2 column halves x 64 token rows x 128 B
constexpr int REC_W0 = 49152;          // W_c, 2 d_k halves x 64 rows (first chunk of a segment only)
constexpr int REC_G = 65536;           // GateRec
constexpr int kRecord = 66560;

struct __align__(16) GateRec {
    float gam[kC];      // e^{G_i}
    float kf[kC];       // e^{G_C - G_i}
    float gC, pad[3];   // e^{G_C}
};

struct TcParams {
    CUtensorMap tm_q, tm_k, tm_v, tm_o;
    const void *a, *b;
    const float *A_log, *dt_bias;
    const float *state_in;
    float *state_out;
    void *o;
    const int32_t *cu_seqlens;
    int64_t seqlen;
    int32_t num_seqs, h_qk, h_v;
    int32_t chunks_per_seq;         // batched input: chunks of every sequence
    // Chunk range [seg_begin, seg_end) of every sequence that this launch covers.  A
    // segment's first chunk starts from W S (like a sequence's first chunk); the state
    // crosses segments through state_in / state_out.  seg_direct: the prep grid holds
    // exactly (sequence, chunk of the range, head) instead of every workspace slot.
    int32_t seg_begin, seg_end, seg_direct;
    float scale;
    int *status;
    uint8_t *ws;                    // workspace records
    long long wait_budget;          // cycles a bounded wait may take (0: kWaitBudget)
    int64_t prep_items;             // (chunk slot, value head) items of this prep launch
    // Update rule (the CUDA page's UpdateRule list): without decay g = 0; without the
    // delta term A = 0, beta = 1 and W = 0 (the T diag(beta gamma) half of the operand
    // tile is zero), so Delta = U = V.  beta_shared: b is [tokens], one beta for all heads.
    int32_t has_decay, has_delta, beta_shared;
    // Time-parallel scan (tp_seg > 0): every sequence is cut into tp_nseg segments of
    // tp_seg chunks, all scanned at once.  Segment k > 0 runs twice: from a zero state
    // (outputs to o, end state to tp_psi[k]) and as the operator pass, from the identity
    // with U = 0 (outputs R to tm_r, end state Phi_k to tp_phi[k]).  Segment 0 runs once
    // from state_in (end state to tp_psi[0]).  A combine and a correction GEMM follow.
    int32_t tp_seg, tp_nseg;
    float *tp_phi, *tp_psi;         // [tp_nseg][N][h_v][128][128] fp32
    CUtensorMap tm_r;               // R: [tokens][h_v][128] in the I/O type
    void *tp_r;
    // Gated RMS norm in the scan's readout (norm_gate set; never with the time-parallel
    // scan): each d_v row of o becomes o / rms(o) * norm_scale * act(gate), written in o's
    // place, with o rounded to the I/O type first as a separate norm would read it.
    const void *norm_scale;         // [128] I/O type
    const void *norm_gate;          // [tokens][h_v][128] I/O type, 16-byte aligned
    float norm_eps;
    int32_t norm_silu;              // act = silu (1) or sigmoid (0)
    // One decay per key dimension (gdn_chunk_prep_pk): the prep writes Q o e^G and
    // K o e^{G_C - G} to qt and kt ([tokens][h_v][128], I/O type), and the scan reads its
    // Q and K through tm_qt and tm_kt instead of tm_q and tm_k.
    int32_t per_key;
    void *qt, *kt;
    CUtensorMap tm_qt, tm_kt;
    CUtensorMap tm_a;               // the gate logits a [tokens][h_v][128]
    // The causal convolution before the scan (gdn_chunk_prep<IO, false, true>): q, k and v
    // are channels of the layer's mixed input x [tokens][conv_C] ([q | k | v], heads
    // outer), each convolved with its conv_k taps (conv_w [conv_C][conv_k], conv_b
    // [conv_C] or NULL) over the conv state (conv_in [sequences][conv_k - 1][conv_C] or
    // NULL: zeros) and the sequence's inputs, then silu when conv_silu.  The prep writes the
    // convolved q and k to cq and ck ([tokens][h_qk][128]; the scan reads them through
    // tm_q and tm_k) and each sequence's last conv_k - 1 inputs to conv_out.
    const void *cx, *conv_w, *conv_b, *conv_in;
    void *conv_out, *cq, *ck, *cv;   // cv: the convolved v, written by the streaming pass only
    int32_t conv_k, conv_silu, conv_C;
};

// First workspace slot of sequence n.  Batched: n * chunks_per_seq.  Packed: slot
// floor(cu[n] / C) + n; consecutive sequences never overlap because a sequence of L
// tokens starting at cu[n] ends before slot floor((cu[n] + L) / C) + n + 1.
__device__ __forceinline__ int64_t slot_base(const TcParams &p, int64_t n) {
    if (p.cu_seqlens == nullptr) return n * p.chunks_per_seq;
    return (int64_t)(p.cu_seqlens[n] / kC) + n;
}

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
// The eight values of a packed 16-byte group, widened to fp32.
template <typename IO>
__device__ __forceinline__ void unpack8(const uint4 &u, float *x) {
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float2 t = Pack<IO>::unpack(w[i]);
        x[2 * i] = t.x;
        x[2 * i + 1] = t.y;
    }
}
// 16-byte global -> shared copy (cp.async) and its group bookkeeping.
__device__ __forceinline__ void cp_async16(void *smem, const void *gmem) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(smem)), "l"(gmem) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N> __device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}
// Store one fp32 value into shared memory of a CTA of this cluster (shared::cluster address).
__device__ __forceinline__ void st_cluster_f32(uint32_t addr, float v) {
    asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(addr), "f"(v) : "memory");
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
// t1 scales the T diag(beta gamma) half (0 for rules without the delta term: W = 0).
template <typename IO>
__device__ __forceinline__ void tt_put2(uint8_t *tt, int r, int c, float x0, float x1,
                                        const float *beta, const float *gam, float t1) {
    const uint32_t off = sw128_offset(r, c >> 3) + (c & 7) * 2;
    const float b0 = beta[c], b1 = beta[c + 1];
    *reinterpret_cast<uint32_t *>(tt + off) =
        Pack<IO>::two(x0 * b0 * gam[c] * t1, x1 * b1 * gam[c + 1] * t1);
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
// Blocks below the diagonal use tf32 warp MMAs.  A is strictly lower, so the blocks of
// As above the diagonal are free: step 2 keeps T_10 and T_32 there transposed (T_ij at
// As[16 j + c][16 i + r]), so A below the diagonal is never overwritten while it is still
// read, and the four other upper blocks hold the intermediate products.  Step 3's blocks
// go only to the operand tile: nothing reads them in fp32 again.
// `side(t)` runs on the other 192 threads (t = 0 .. 191) during step 1.
template <typename IO, typename Side>
__device__ void invert_chunk(float *As, uint8_t *tt, const float *beta, const float *gam, float t1,
                             int pt, Side &&side) {
    if (pt < 64) {
        // Column-oriented: once x_l is known it updates every later row's sum, so the
        // serial chain is one FMA per row instead of a whole dot product.
        const int o = (pt >> 4) * 16, j = pt & 15, cj = o + j;
        float x[16], acc[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) acc[i] = 0.f;
#pragma unroll
        for (int l = 0; l < 16; ++l) {
            x[l] = (l < j) ? 0.f : ((l == j) ? 1.f : -acc[l]);
#pragma unroll
            for (int i = l + 1; i < 16; ++i) acc[i] = fmaf(As[(o + i) * kAs + o + l], x[l], acc[i]);
        }
        __syncwarp();
        const float f2 = beta[cj], f1 = f2 * gam[cj] * t1;
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            As[(o + i) * kAs + cj] = x[i];
            tt_put<IO>(tt, o + i, cj, x[i], f1, f2);
        }
    } else {
        side(pt - 64);
    }
    named_bar(kBarPrep, kPrepThreads);
    const int w = pt >> 5, lane = pt & 31, g = lane >> 2, t = lane & 3;
    auto diag = [&](int b) { return Blk{As + 16 * b * kAs + 16 * b, kAs, 1}; };
    auto low = [&](int i, int j) { return Blk{As + 16 * i * kAs + 16 * j, kAs, 1}; };  // A_ij
    auto tlo = [&](int i, int j) { return Blk{As + 16 * j * kAs + 16 * i, 1, kAs}; };  // T_ij
    // Intermediate k in upper block (0, 2), (1, 3), (0, 3) or (1, 2).
    auto scratch = [&](int k) {
        const int rb = (k == 1 || k == 3) ? 1 : 0, cb = (k == 0 || k == 3) ? 2 : 3;
        return Blk{As + 16 * rb * kAs + 16 * cb, kAs, 1};
    };
    auto emit = [&](int i, int j, const float (&acc)[2][4], bool keep) {   // T_ij = -acc
        if (keep) block_store(tlo(i, j), acc, -1.f, g, t);
#pragma unroll
        for (int nh = 0; nh < 2; ++nh) {
            const int c = 16 * j + 8 * nh + 2 * t, r = 16 * i + g;
            tt_put2<IO>(tt, r, c, -acc[nh][0], -acc[nh][1], beta, gam, t1);
            tt_put2<IO>(tt, r + 8, c, -acc[nh][2], -acc[nh][3], beta, gam, t1);
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
        emit(hi, lo, res, true);
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
        emit(bi, bj, res, false);
    }
}

// ===================================================================== chunk prep
// Shared memory (from a 1024-aligned base): 66 KB, so that three CTAs share an SM.  The
// record's pieces go to global memory straight from registers.
constexpr int kRegP = 16384;                   // 128 rows x 128 B for 64 d_k: [K; Q]
constexpr int PP_KQ = 0;                       // two regions; V lands over Q, W over K
constexpr int PP_TT = 2 * kRegP;               // [T'; T''], 128 x 128 B
constexpr int PP_AS = PP_TT + 16384;           // A, then T, fp32 [64][68]; later K_{c-1}
constexpr int kPrepSmem = PP_AS + 64 * kAs * 4 + 1024;
constexpr uint32_t kPrepCols = 128;            // TMEM columns of a prep CTA

// One (chunk slot, value head) item of the prep.  Idle slots (past a sequence's last
// chunk, outside the launch's chunk range, or of a sequence whose device cu_seqlens
// entries are malformed) are not valid.
struct PrepItem {
    int64_t slot, tc0;
    int64_t n, ts, te;                 // sequence, its token range [ts, te)
    int32_t h, hq, Lc, first, valid, pad;
};

__device__ PrepItem prep_item(const TcParams &p, int64_t item) {
    PrepItem it;
    it.valid = 0;
    if (item >= p.prep_items) return it;
    it.h = (int32_t)(item % p.h_v);
    it.hq = it.h / (p.h_v / p.h_qk);
    int64_t slot = item / p.h_v, n;
    if (p.seg_direct) {
        const int64_t per = p.seg_end - p.seg_begin;
        n = slot / per;
        if (n >= p.num_seqs) return it;
        slot = n * p.chunks_per_seq + p.seg_begin + slot % per;
    } else if (p.cu_seqlens == nullptr) {
        n = slot / p.chunks_per_seq;
        if (n >= p.num_seqs) return it;
    } else {
        int64_t lo = 0, hi = p.num_seqs - 1;       // last n with slot_base(n) <= slot
        if (slot_base(p, 0) > slot) return it;
        while (lo < hi) {
            const int64_t mid = (lo + hi + 1) >> 1;
            if (slot_base(p, mid) <= slot) lo = mid; else hi = mid - 1;
        }
        n = lo;
    }
    int64_t t0, t1;
    if (!seq_range(p.cu_seqlens, p.seqlen, p.num_seqs, p.status, n, t0, t1)) return it;
    const int64_t c = slot - slot_base(p, n);
    if (c * kC >= t1 - t0 || c < p.seg_begin || c >= p.seg_end) return it;
    it.slot = slot;
    it.n = n;
    it.ts = t0;
    it.te = t1;
    it.tc0 = t0 + c * kC;
    it.Lc = (int32_t)((t1 - it.tc0) < kC ? (t1 - it.tc0) : kC);
    // A segment's first chunk writes W for the scan to start from; every other chunk
    // writes W and M into its predecessor's record.
    it.first = (c == p.seg_begin) || (p.tp_seg > 0 && c % p.tp_seg == 0);
    it.valid = 1;
    return it;
}

struct PrepCtl {
    uint64_t full, vfull, d1, d2, d3, kprev, dm;
    PrepItem nxt;                      // the CTA's next item
    uint32_t tmem;
    float G[kC], beta[kC], gam[kC], E[kC], F[kC], wsum[2];
    float kfp[kC], wsum_p[2];          // previous chunk: e^{G_C - G_j}
};

// ------------------------------------------------------------------ convolution prologue
// The causal convolution of eight consecutive channels c0 .. c0 + 7 (one 16-byte group) of
// the mixed input x, for `count` consecutive tokens from `tok` of the sequence that starts
// at ts (sequence n), each written by put(j, packed outputs of token tok + j).  Output
// token t is act(w[c][0] x[t - K + 1][c] + ... + w[c][K - 1] x[t][c] + bias[c]) in fp32,
// oldest tap first, rounded once, as gdn_causal_conv computes it; positions before ts
// come from the conv state.  A sliding window of K rows is loaded once per position.
// Tokens at or past the sequence's end te (a ragged chunk's padded rows) are written as
// zeros and nothing past te is read: the chunk algebra masks those rows with beta = 0,
// which needs finite values in them.
template <typename IO, typename Put>
__device__ __forceinline__ void conv_group(const TcParams &p, int64_t n, int64_t ts, int64_t te,
                                           int64_t tok, int count, int c0, Put &&put) {
    const int K = p.conv_k;
    const IO *x = static_cast<const IO *>(p.cx);
    const IO *w = static_cast<const IO *>(p.conv_w);
    // Window slot j holds position t - 3 + j; tap m (oldest first) sits in slot 4 - K + m,
    // and the slots before it carry a zero weight (and a zero input), which leaves the
    // first real product exact, so the sum runs in the convolution kernel's order.  The
    // taps, the bias and the window stay packed in the I/O type (exact) to spare registers.
    uint4 wp[4], bp, win[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        float t[8];
#pragma unroll
        for (int i = 0; i < 8; ++i)
            t[i] = j >= 4 - K ? IoType<IO>::ld(w + (size_t)(c0 + i) * K + (j - (4 - K))) : 0.f;
        wp[j] = pack8<IO>(t);
    }
    bp = p.conv_b != nullptr ? *reinterpret_cast<const uint4 *>(static_cast<const IO *>(p.conv_b) + c0)
                             : make_uint4(0, 0, 0, 0);
    auto row = [&](int64_t pos) {   // x[pos][c0 ..], or the state before ts
        uint4 u = make_uint4(0, 0, 0, 0);
        if (pos >= te) {
        } else if (pos >= ts) {
            u = *reinterpret_cast<const uint4 *>(x + (size_t)pos * p.conv_C + c0);
        } else if (p.conv_in != nullptr) {
            const int64_t r = (K - 1) + (pos - ts);   // >= 0 for the taps that reach here
            u = *reinterpret_cast<const uint4 *>(static_cast<const IO *>(p.conv_in) +
                                                  ((size_t)n * (K - 1) + r) * p.conv_C + c0);
        }
        return u;
    };
#pragma unroll
    for (int j = 0; j < 3; ++j) win[j] = j >= 4 - K ? row(tok - 3 + j) : make_uint4(0, 0, 0, 0);
    auto word = [](const uint4 &u, int k) { return k == 0 ? u.x : k == 1 ? u.y : k == 2 ? u.z : u.w; };
#pragma unroll 1
    for (int e = 0; e < count; ++e) {
        if (tok + e >= te) {
            put(e, make_uint4(0, 0, 0, 0));
            continue;
        }
        win[3] = row(tok + e);
        float out[8];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            float2 acc;
            {
                const float2 wv = Pack<IO>::unpack(word(wp[0], k)), xv = Pack<IO>::unpack(word(win[0], k));
                acc = make_float2(wv.x * xv.x, wv.y * xv.y);
            }
#pragma unroll
            for (int j = 1; j < 4; ++j) {
                const float2 wv = Pack<IO>::unpack(word(wp[j], k)), xv = Pack<IO>::unpack(word(win[j], k));
                acc.x = fmaf(wv.x, xv.x, acc.x);
                acc.y = fmaf(wv.y, xv.y, acc.y);
            }
            const float2 bv = Pack<IO>::unpack(word(bp, k));
            acc.x += bv.x;
            acc.y += bv.y;
            out[2 * k] = p.conv_silu ? __fdividef(acc.x, 1.0f + __expf(-acc.x)) : acc.x;
            out[2 * k + 1] = p.conv_silu ? __fdividef(acc.y, 1.0f + __expf(-acc.y)) : acc.y;
        }
        put(e, pack8<IO>(out));
        win[0] = win[1];
        win[1] = win[2];
        win[2] = win[3];
    }
}

// The same convolution for the streaming pass (conv_pass), four tokens at a time: the
// taps are loaded once per thread, and the seven window rows of a call all at once.
struct ConvTaps {
    float w[4][8], b[8];   // slot-aligned taps and the bias, widened once
};

template <typename IO>
__device__ __forceinline__ ConvTaps conv_taps(const TcParams &p, int c0) {
    const int K = p.conv_k;
    const IO *w = static_cast<const IO *>(p.conv_w);
    ConvTaps t;
#pragma unroll
    for (int j = 0; j < 4; ++j)
#pragma unroll
        for (int i = 0; i < 8; ++i)
            t.w[j][i] = j >= 4 - K ? IoType<IO>::ld(w + (size_t)(c0 + i) * K + (j - (4 - K))) : 0.f;
#pragma unroll
    for (int i = 0; i < 8; ++i)
        t.b[i] = p.conv_b != nullptr ? IoType<IO>::ld(static_cast<const IO *>(p.conv_b) + c0 + i) : 0.f;
    return t;
}

// Tokens tok .. tok + 3 from the seven window rows row(tok - 3) .. row(tok + 3), widened
// once: each output is formed oldest tap first, then the bias, rounded once, and handed
// to put(e, packed).
template <typename IO, typename Row, typename Put>
__device__ __forceinline__ void conv4(const TcParams &p, const ConvTaps &tp, int64_t tok, Row &&row, Put &&put) {
    float win[7][8];
#pragma unroll
    for (int j = 0; j < 7; ++j) unpack8<IO>(row(tok - 3 + j), win[j]);
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        float out[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            float acc = tp.w[0][i] * win[e][i];
#pragma unroll
            for (int j = 1; j < 4; ++j) acc = fmaf(tp.w[j][i], win[e + j][i], acc);
            acc += tp.b[i];
            out[i] = p.conv_silu ? __fdividef(acc, 1.0f + __expf(-acc)) : acc;
        }
        put(e, pack8<IO>(out));
    }
}

// One token tok from the four rows row(tok - 3) .. row(tok), in the same order.
template <typename IO, typename Row>
__device__ __forceinline__ uint4 conv1(const TcParams &p, const ConvTaps &tp, int64_t tok, Row &&row) {
    float win[4][8];
#pragma unroll
    for (int j = 0; j < 4; ++j) unpack8<IO>(row(tok - 3 + j), win[j]);
    float out[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        float acc = tp.w[0][i] * win[0][i];
#pragma unroll
        for (int j = 1; j < 4; ++j) acc = fmaf(tp.w[j][i], win[j][i], acc);
        acc += tp.b[i];
        out[i] = p.conv_silu ? __fdividef(acc, 1.0f + __expf(-acc)) : acc;
    }
    return pack8<IO>(out);
}

// The present conv state of sequence n for channels c0 .. c0 + 7: its last K - 1 inputs
// (state rows first when the sequence is shorter than that).
template <typename IO>
__device__ __forceinline__ void conv_state_group(const TcParams &p, int64_t n, int64_t ts, int64_t te,
                                                 int c0) {
    const int K = p.conv_k;
    for (int r = 0; r < K - 1; ++r) {
        const int64_t pos = te - (K - 1) + r;
        uint4 u = make_uint4(0, 0, 0, 0);
        if (pos >= ts) {
            u = *reinterpret_cast<const uint4 *>(static_cast<const IO *>(p.cx) + (size_t)pos * p.conv_C + c0);
        } else if (p.conv_in != nullptr) {
            u = *reinterpret_cast<const uint4 *>(static_cast<const IO *>(p.conv_in) +
                                                  ((size_t)n * (K - 1) + (K - 1) + (pos - ts)) * p.conv_C + c0);
        }
        *reinterpret_cast<uint4 *>(static_cast<IO *>(p.conv_out) + ((size_t)n * (K - 1) + r) * p.conv_C + c0) = u;
    }
}

// Persistent CTAs, three to an SM, walk the (chunk slot, value head) items with the
// grid's stride.  TMEM (128 columns) holds one product at a time: D1 = [K; Q] K^T, then
// D2 = [T'; T''] K (W on lanes 0-63), D3 = [T'; T''] V (U on lanes 64-127) and
// M = W K_{c-1}^T, each read out before the next is issued.  While an item's diagonal
// blocks are inverted, one thread looks up the CTA's next item.  (Prefetching the next
// item's tiles into L2 there was measured slower.)
// kVariant: the update-rule switches and the shared beta are read from the parameters;
// without it the gated delta rule with one beta per head is compiled in (the switches
// cost the default rule about 5% when they were runtime values).
// kConv (with the default rule): q, k and v are not loaded but convolved from the layer's
// mixed input (conv_group) straight into the operand tiles -- K and Q at the item's
// start, V by the threads the inversion's first step leaves idle, the previous chunk's K
// while D2 runs -- and thread 0 arrives on the barriers the copies would have completed.
// The first value head of each q/k head writes the convolved q and k for the scan, and the
// items of a sequence's last chunk write its present conv state.
template <typename IO, bool kVariant, bool kConv = false>
__global__ void __launch_bounds__(kPrepThreads, 3) gdn_chunk_prep(const __grid_constant__ TcParams p) {
    constexpr bool kBf16 = std::is_same<IO, __nv_bfloat16>::value;
    const bool has_decay = !kVariant || p.has_decay != 0;
    const bool has_delta = !kVariant || p.has_delta != 0;
    const bool beta_shared = kVariant && p.beta_shared != 0;
    constexpr uint32_t kIdD1 = idesc_f16(kBf16, 128, 64, false, false);
    constexpr uint32_t kIdD2 = idesc_f16(kBf16, 128, 128, false, true);

    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                              ~static_cast<uintptr_t>(1023));
    __shared__ PrepCtl ctl;
    const int pt = threadIdx.x, warp = pt >> 5, lane = pt & 31;
    const long long budget = p.wait_budget > 0 ? p.wait_budget : kWaitBudget;
    const int q = warp & 3, hf = warp >> 2;        // TMEM lane quarter, column half
    float *const As = reinterpret_cast<float *>(sm + PP_AS);
    const uint32_t aKQ = smem_u32(sm + PP_KQ), aTT = smem_u32(sm + PP_TT);
    if (warp == 0) {
        tmem_alloc(&ctl.tmem, kPrepCols);
        tmem_relinquish();
    }
    if (pt == 0) {
        mbar_init(&ctl.full, 1);
        mbar_init(&ctl.vfull, 1);
        mbar_init(&ctl.d1, 1);
        mbar_init(&ctl.d2, 1);
        mbar_init(&ctl.d3, 1);
        mbar_init(&ctl.kprev, 1);
        mbar_init(&ctl.dm, 1);
        fence_mbar_init();
        ctl.nxt = prep_item(p, blockIdx.x);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = ctl.tmem;
    const uint32_t lane_base = static_cast<uint32_t>(32 * q) << 16;
    const int row = 32 * q + lane;
    // mbarrier parities: full, vfull, d1, d2 and d3 complete once per item, kprev and dm
    // once per item that is not a segment's first chunk.
    uint32_t ph = 0, phk = 0;
    // thread 0: 1 = V load, 2 = D1, 4 = D2, 8 = K_{c-1} load, 16 = M, 32 = D3
    uint32_t issued = 0;
    bool ok = true, failed = false;
    for (int64_t item = blockIdx.x; item < p.prep_items; item += gridDim.x) {
    const PrepItem it = ctl.nxt;
    if (!it.valid) {
        __syncthreads();   // every thread has read ctl.nxt
        if (pt == 0) ctl.nxt = prep_item(p, item + gridDim.x);
        __syncthreads();
        continue;
    }
    const int h = it.h, hq = it.hq, Lc = it.Lc;
    const bool first = it.first != 0;
    const int64_t tc0 = it.tc0;
    uint8_t *rec = p.ws + ((size_t)it.slot * p.h_v + h) * kRecord;
    uint8_t *const rec_prev = rec - (size_t)p.h_v * kRecord;   // chunk c - 1, same head
    issued = 0;

    // [T'; T''] blocks above the diagonal are never written: keep them zero (the previous
    // item's U staging has been read out of this tile).
    for (int e = pt; e < 16384 / 16; e += kPrepThreads)
        *reinterpret_cast<uint4 *>(sm + PP_TT + 16 * e) = make_uint4(0, 0, 0, 0);
    fence_async_smem();
    const int tok = (int)tc0;
    // With the convolution: the channel group of q or k (head hq) this thread convolves,
    // and whether this item writes them out (the first value head of the q/k head) and the
    // present conv state (a sequence's last chunk).
    const bool cv_qk_out = kConv && (h % (p.h_v / p.h_qk)) == 0;
    const bool cv_last = kConv && tc0 + Lc == it.te;
    if constexpr (kConv) {
        // K and Q of this chunk: thread (group 0-31 of [q | k] head hq, tokens 8 tb ..).
        const int grp = pt & 31, tb = pt >> 5;
        const bool isk = grp >= 16;
        const int i0 = 8 * (grp & 15);                         // channel within the head
        const int c0 = (isk ? p.h_qk * kDK : 0) + hq * kDK + i0;
        uint8_t *dst = sm + PP_KQ + (i0 >> 6) * kRegP + (isk ? 0 : 8192);
        IO *gout = static_cast<IO *>(isk ? p.ck : p.cq) + (size_t)hq * kDK + i0;
        conv_group<IO>(p, it.n, it.ts, it.te, tc0 + 8 * tb, 8, c0, [&](int e, const uint4 &u) {
            const int t = 8 * tb + e;
            *reinterpret_cast<uint4 *>(dst + sw128_offset(t, (i0 & 63) >> 3)) = u;
            if (cv_qk_out && t < Lc) *reinterpret_cast<uint4 *>(gout + (size_t)(tc0 + t) * p.h_qk * kDK) = u;
        });
        if (cv_qk_out && cv_last && tb == 0) conv_state_group<IO>(p, it.n, it.ts, it.te, c0);
        fence_async_smem();
        named_bar(kBarPrep, kPrepThreads);
        if (pt == 0) mbar_arrive(&ctl.full);
    } else if (pt == 0) {
        mbar_arrive_expect_tx(&ctl.full, 4 * 8192);
#pragma unroll
        for (int r = 0; r < 2; ++r) {
            tma_load_3d(sm + PP_KQ + r * kRegP, &p.tm_k, r * 64, hq, tok, &ctl.full);
            tma_load_3d(sm + PP_KQ + r * kRegP + 8192, &p.tm_q, r * 64, hq, tok, &ctl.full);
        }
    }
    // The gates (this chunk's and, for W' and M, the previous chunk's decay) are computed
    // from plain loads of the logits while K and Q are in flight.
    float ra = 0.f, rb = 0.f, rap = 0.f;
    if (pt < Lc) {
        if (has_decay) ra = IoType<IO>::ld(static_cast<const IO *>(p.a) + (size_t)(tc0 + pt) * p.h_v + h);
        if (has_delta)
            rb = IoType<IO>::ld(static_cast<const IO *>(p.b) +
                                (beta_shared ? (size_t)(tc0 + pt) : (size_t)(tc0 + pt) * p.h_v + h));
    }
    if (!first && pt < kC && has_decay)
        rap = IoType<IO>::ld(static_cast<const IO *>(p.a) + (size_t)(tc0 - kC + pt) * p.h_v + h);
    bool ok = true, failed = false;
    {
        float gsum = 0.f, be = 0.f, gsum_p = 0.f;
        if (pt < kC) {
            if (pt < Lc) {
                gsum = has_decay ? decay_f(ra, p.A_log[h], p.dt_bias[h]) : 0.f;
                be = has_delta ? sigmoid_f(rb) : 1.f;
            }
            if (!first && has_decay) gsum_p = decay_f(rap, p.A_log[h], p.dt_bias[h]);
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const float y = __shfl_up_sync(0xffffffffu, gsum, off);
                const float yp = __shfl_up_sync(0xffffffffu, gsum_p, off);
                if (lane >= off) {
                    gsum += y;
                    gsum_p += yp;
                }
            }
            if (lane == 31) {
                ctl.wsum[warp] = gsum;
                ctl.wsum_p[warp] = gsum_p;
            }
        }
        named_bar(kBarPrep, kPrepThreads);
        if (pt < kC) {
            ctl.G[pt] = gsum + (warp == 1 ? ctl.wsum[0] : 0.f);
            ctl.beta[pt] = be;
            // Previous chunk: e^{G_C - G_j} = e^{(sum of its g) - G_j}.
            const float gp = gsum_p + (warp == 1 ? ctl.wsum_p[0] : 0.f);
            ctl.kfp[pt] = __expf(ctl.wsum_p[0] + ctl.wsum_p[1] - gp);
        }
        named_bar(kBarPrep, kPrepThreads);
        const float GC = ctl.G[kC - 1], Gm = ctl.G[31];
        if (pt < kC) {
            const float G = ctl.G[pt];
            const float gm = __expf(G);
            GateRec *grec = reinterpret_cast<GateRec *>(rec + REC_G);
            ctl.gam[pt] = gm;
            grec->gam[pt] = gm;
            grec->kf[pt] = __expf(GC - G);
            ctl.E[pt] = __expf(G - Gm);
            ctl.F[pt] = __expf(Gm - G);
            if (pt == 0) grec->gC = __expf(GC);
        }
    }
    // D1 = [K; Q] K^T once K and Q have landed; then V over the Q rows, which D1 has read.
    if (pt == 0) {
        ok = mbar_wait(&ctl.full, ph, budget);
        if (ok) {
            tc_fence_after();
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                const uint32_t off = (k >> 2) * kRegP + (k & 3) * 32;
                mma_f16(tmem, sw128_desc(aKQ + off, 16, 1024), sw128_desc(aKQ + off, 16, 1024), kIdD1,
                        k > 0);
            }
            mma_commit(&ctl.d1);
            issued |= 2;
            ok = mbar_wait(&ctl.d1, ph, budget);
        }
        if (ok && !kConv) {
            mbar_arrive_expect_tx(&ctl.vfull, 2 * 8192);
#pragma unroll
            for (int r = 0; r < 2; ++r)
                tma_load_3d(sm + PP_KQ + r * kRegP + 8192, &p.tm_v, r * 64, h, tok, &ctl.vfull);
            issued |= 1;
        }
    }
    failed = bar_any(kBarPrep, kPrepThreads, !ok);   // also publishes E, F, gamma
    if (!failed) ok = mbar_wait(&ctl.full, ph, budget);   // K, written by TMA, is rewritten below
    if (!failed) {
        tc_fence_after();
        // A rows (lanes 0-63, fp32, to As) and P rows (lanes 64-127, I/O type, to the
        // record); each column half of the warps takes 32 of the 64 columns.
        {
            uint32_t r[32];
            tmem_ld32(tmem + lane_base + 32 * hf, r);
            tmem_ld_wait();
            const int i = (32 * q + lane) & 63;
            const float Ei = ctl.E[i], Gi = ctl.G[i];
            // e^{G_i - G_m} e^{G_m - G_j} cannot overflow while G spans at most 80.
            const bool safe = (ctl.G[0] - ctl.G[kC - 1]) <= 80.f;
            if (q < 2) {
                const float bi = ctl.beta[i];
#pragma unroll
                for (int j4 = 0; j4 < 8; ++j4) {
                    float x[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const int j = 32 * hf + 4 * j4 + e;
                        const float d = safe ? Ei * ctl.F[j] : __expf(Gi - ctl.G[j]);
                        x[e] = (j < i && has_delta) ? bi * d * __uint_as_float(r[4 * j4 + e]) : 0.f;
                    }
                    *reinterpret_cast<float4 *>(As + i * kAs + 32 * hf + 4 * j4) =
                        make_float4(x[0], x[1], x[2], x[3]);
                }
            } else {
                // Two 16-byte chunks of a row at a time: logical chunks 2m and 2m + 1 sit
                // side by side in the 128-byte swizzle, swapped on odd rows.
#pragma unroll
                for (int m = 0; m < 2; ++m) {
                    uint4 u[2];
#pragma unroll
                    for (int h2 = 0; h2 < 2; ++h2) {
                        const int q8 = 2 * m + h2;
                        float x[8];
#pragma unroll
                        for (int e = 0; e < 8; ++e) {
                            const int j = 32 * hf + 8 * q8 + e;
                            const float d = safe ? Ei * ctl.F[j] : __expf(Gi - ctl.G[j]);
                            x[e] = (j <= i) ? p.scale * d * __uint_as_float(r[8 * q8 + e]) : 0.f;
                        }
                        u[h2] = pack8<IO>(x);
                    }
                    uint8_t *dst = rec + REC_PM + sw128_offset(i, (4 * hf + 2 * m) & ~1);
                    if (i & 1) st_global_v8(dst - 16, u[1], u[0]);   // chunk pair starts at the odd slot - 1
                    else st_global_v8(dst, u[0], u[1]);
                }
            }
        }
        tc_fence_before();
        named_bar(kBarPrep, kPrepThreads);

        // T = (I + A)^-1, written as [T diag(beta gamma); T diag(beta)] (K-major).
        // Meanwhile one thread of warp 2 looks up the CTA's next item, and with the
        // convolution 128 of the other threads convolve V over the spent Q rows (D1 has
        // read them): thread (group of 8 v channels, 8 tokens).
        auto next_item = [&](int t) {
            if (t == 0) ctl.nxt = prep_item(p, item + gridDim.x);
            if constexpr (kConv) {
                if (t < 128) {
                    const int grp = t & 15, tb = t >> 4, i0 = 8 * grp;
                    const int c0 = 2 * p.h_qk * kDK + h * kDK + i0;
                    uint8_t *dst = sm + PP_KQ + (i0 >> 6) * kRegP + 8192;
                    conv_group<IO>(p, it.n, it.ts, it.te, tc0 + 8 * tb, 8, c0, [&](int e, const uint4 &u) {
                        *reinterpret_cast<uint4 *>(dst + sw128_offset(8 * tb + e, (i0 & 63) >> 3)) = u;
                    });
                    if (cv_last && tb == 0) conv_state_group<IO>(p, it.n, it.ts, it.te, c0);
                }
            }
        };
        invert_chunk<IO>(As, sm + PP_TT, ctl.beta, ctl.gam, has_delta ? 1.f : 0.f, pt, next_item);
        fence_async_smem();
        tc_fence_before();
        named_bar(kBarPrep, kPrepThreads);
        if (kConv && pt == 0) mbar_arrive(&ctl.vfull);
        if (pt == 0) {
            // The previous chunk's keys (for M) into the spent A/T tile.
            if (!first && !kConv) {
                mbar_arrive_expect_tx(&ctl.kprev, 2 * 8192);
#pragma unroll
                for (int r = 0; r < 2; ++r)
                    tma_load_3d(sm + PP_AS + r * 8192, &p.tm_k, r * 64, hq, tok - kC, &ctl.kprev);
                issued |= 8;
            }
            // D2 = [T'; T''] K: W on lanes 0-63.
            tc_fence_after();
#pragma unroll
            for (int k = 0; k < 4; ++k)
                mma_f16(tmem, sw128_desc(aTT + k * 32, 16, 1024), sw128_desc(aKQ + k * 2048, kRegP, 1024),
                        kIdD2, k > 0);
            mma_commit(&ctl.d2);
            issued |= 4;
        }
        if constexpr (kConv) {
            // The previous chunk's keys, convolved while D2 runs: thread (group of 8 k
            // channels, 4 tokens).
            if (!first) {
                const int grp = pt & 15, tb = pt >> 4, i0 = 8 * grp;
                const int c0 = p.h_qk * kDK + hq * kDK + i0;
                uint8_t *dst = sm + PP_AS + (i0 >> 6) * 8192;
                conv_group<IO>(p, it.n, it.ts, it.te, tc0 - kC + 4 * tb, 4, c0, [&](int e, const uint4 &u) {
                    *reinterpret_cast<uint4 *>(dst + sw128_offset(4 * tb + e, (i0 & 63) >> 3)) = u;
                });
                fence_async_smem();
                named_bar(kBarPrep, kPrepThreads);
                if (pt == 0) mbar_arrive(&ctl.kprev);
            }
        }
        if (pt == 0) ok = mbar_wait(&ctl.d2, ph, budget);
        failed = bar_any(kBarPrep, kPrepThreads, !ok);
    }
    const int row = 32 * q + lane;
    if (!failed) {
        // W (fp32, lanes 0-63) in the I/O type over the spent K rows: the A operand of M and
        // the image of the record's W (the previous chunk's W_{c+1}, or W_0 for a segment's
        // first chunk).
        tc_fence_after();
        if (q < 2) {
#pragma unroll
            for (int c0 = 0; c0 < 64; c0 += 32) {
                uint32_t r[32];
                tmem_ld32(tmem + lane_base + 64 * hf + c0, r);
                tmem_ld_wait();
                float x[32];
#pragma unroll
                for (int e = 0; e < 32; ++e) x[e] = __uint_as_float(r[e]);
#pragma unroll
                for (int q8 = 0; q8 < 4; ++q8)
                    *reinterpret_cast<uint4 *>(sm + PP_KQ + hf * kRegP + sw128_offset(row, (c0 >> 3) + q8)) =
                        pack8<IO>(x + 8 * q8);
            }
        }
        fence_async_smem();
        tc_fence_before();
        named_bar(kBarPrep, kPrepThreads);
        // D3 = [T'; T''] V (U on lanes 64-127) while W goes out.
        if (pt == 0) {
            uint8_t *dst = first ? rec + REC_W0 : rec_prev + REC_W;
#pragma unroll
            for (int r = 0; r < 2; ++r) bulk_store(dst + r * 8192, sm + PP_KQ + r * kRegP, 8192);
            bulk_commit();
            ok = mbar_wait(&ctl.vfull, ph, budget);
            if (ok) {
                tc_fence_after();
#pragma unroll
                for (int k = 0; k < 4; ++k)
                    mma_f16(tmem, sw128_desc(aTT + k * 32, 16, 1024),
                            sw128_desc(aKQ + 8192 + k * 2048, kRegP, 1024), kIdD2, k > 0);
                mma_commit(&ctl.d3);
                issued |= 32;
                ok = mbar_wait(&ctl.d3, ph, budget);
            }
        }
        failed = bar_any(kBarPrep, kPrepThreads, !ok);
    }
    if (!failed) {
        // U (lanes 64-127) into the spent [T'; T''] tile, as the record's U image.
        tc_fence_after();
        if (q >= 2) {
            const int j = row - 64;
#pragma unroll
            for (int c0 = 0; c0 < 64; c0 += 32) {
                uint32_t r[32];
                tmem_ld32(tmem + lane_base + 64 * hf + c0, r);
                tmem_ld_wait();
                float x[32];
#pragma unroll
                for (int e = 0; e < 32; ++e) x[e] = __uint_as_float(r[e]);
#pragma unroll
                for (int q8 = 0; q8 < 4; ++q8)
                    *reinterpret_cast<uint4 *>(sm + PP_TT + hf * 8192 + sw128_offset(j, (c0 >> 3) + q8)) =
                        pack8<IO>(x + 8 * q8);
            }
        }
        fence_async_smem();
        tc_fence_before();
        named_bar(kBarPrep, kPrepThreads);
        // U goes out; then M_c = W_c K_{c-1}^T (U has left TMEM: M overwrites its lanes).
        if (pt == 0) {
            bulk_store(rec + REC_U, sm + PP_TT, 16384);
            bulk_commit();
            if (!first) {
                ok = mbar_wait(&ctl.kprev, phk, budget);
                if (ok) {
                    tc_fence_after();
                    const uint32_t aKp = smem_u32(sm + PP_AS);
#pragma unroll
                    for (int k = 0; k < 8; ++k)
                        mma_f16(tmem, sw128_desc(aKQ + (k >> 2) * kRegP + (k & 3) * 32, 16, 1024),
                                sw128_desc(aKp + (k >> 2) * 8192 + (k & 3) * 32, 16, 1024), kIdD1, k > 0);
                    mma_commit(&ctl.dm);
                    issued |= 16;
                    ok = mbar_wait(&ctl.dm, phk, budget);
                }
            }
        }
        if (!first) {
            failed = bar_any(kBarPrep, kPrepThreads, !ok);
            if (!failed) {
                // M_c[i][j] = (W_c K_{c-1}^T)[i][j] e^{G_C - G_j} of chunk c - 1, rows on lanes
                // 0-63, staged over the spent V rows for the previous chunk's record.
                tc_fence_after();
                if (q < 2) {
                    uint32_t r[32];
                    tmem_ld32(tmem + lane_base + 32 * hf, r);
                    tmem_ld_wait();
                    float x[32];
#pragma unroll
                    for (int e = 0; e < 32; ++e) x[e] = __uint_as_float(r[e]) * ctl.kfp[32 * hf + e];
#pragma unroll
                    for (int q8 = 0; q8 < 4; ++q8)
                        *reinterpret_cast<uint4 *>(sm + PP_KQ + 8192 + sw128_offset(row, 4 * hf + q8)) =
                            pack8<IO>(x + 8 * q8);
                }
                fence_async_smem();
                named_bar(kBarPrep, kPrepThreads);
                if (pt == 0) {
                    bulk_store(rec_prev + REC_PM + 8192, sm + PP_KQ + 8192, 8192);
                    bulk_commit();
                }
            }
        }
    }
    if (failed) break;    // the whole CTA, with this item's parities and copies in flight
    // Before the next item's loads overwrite them, the record stores have read their
    // staging tiles and every thread is done with this item's tiles and TMEM.
    if (pt == 0) bulk_wait_read();
    ph ^= 1u;
    if (!first) phk ^= 1u;
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    }   // items
    if (failed && pt == 0) {
        // Let the copies and MMAs already issued land before the CTA leaves (bounded).
        atomicOr(p.status, kDevTimeout);
        mbar_wait(&ctl.full, ph, kWaitBudget);
        if (issued & 1) mbar_wait(&ctl.vfull, ph, kWaitBudget);
        if (issued & 2) mbar_wait(&ctl.d1, ph, kWaitBudget);
        if (issued & 4) mbar_wait(&ctl.d2, ph, kWaitBudget);
        if (issued & 32) mbar_wait(&ctl.d3, ph, kWaitBudget);
        if (issued & 8) mbar_wait(&ctl.kprev, phk, kWaitBudget);
        if (issued & 16) mbar_wait(&ctl.dm, phk, kWaitBudget);
    }
    if (pt == 0) bulk_wait_read();   // the record stores have read their staging tiles
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, kPrepCols);
    }
}

// ===================================================================== chunk prep, per-key decay
// One decay per key dimension (the CUDA page's decay_per_key_dim: Step 1 scales row i of
// the state by e^{g_i}).  With G_t = sum_{s<=t} g_s inside the chunk, a vector over d_k,
//   S_t = diag(e^{G_t}) S_0 + sum_{s<=t} diag(e^{G_t - G_s}) k_s delta_s^T,
// so the chunk algebra keeps its shape with the gates moved into the operands:
//   A_ts = beta_t sum_i k_ti k_si e^{G_ti - G_si} (s < t),
//   P_ts = scale sum_i q_ti k_si e^{G_ti - G_si} (s <= t),
//   W = T diag(beta) (K o e^G),  U = T diag(beta) V,  Delta = U - W S_c,
//   o = scale (Q o e^G) S_c + P Delta,  S_{c+1} = diag(e^{G_C}) S_c + (K o e^{G_C - G})^T Delta.
// The record keeps the scalar layout with the gates folded in: W'_{c+1} = W_{c+1}
// diag(e^{G_C(c)}) and M_{c+1} = W_{c+1} (K_c o e^{G_C - G})^T, so the scan's lookahead
// takes no gate (gC = 1), and the gate record holds e^{G_C} per key dimension (gam:
// dimensions 0-63, kf: 64-127) for the scan's state update.  Q~ = Q o e^G and K~ =
// K o e^{G_C - G} go to two workspace arrays ([tokens][h_v][128], I/O type), from which
// the scan loads Q and K.
// e^{G_t - G_s} depends on the key dimension, so A and P are no scaled Gram matrix: they
// are formed on the FP32 cores.  Every exponent taken is <= 0 (G never grows along the
// chunk): a 4 x 4 tile below the diagonal (rows t0 .. t0 + 3, columns s0 .. s0 + 3 < t0)
// uses e^{G_t - G_t0} e^{G_t0 - G_s}; the 16 tiles on the diagonal take e^{G_t - G_s} per
// pair.
constexpr int kGs = 132;                        // row stride (floats) of the G tile
constexpr int PK_KQ = 0;                        // [K; Q] per d_k half: K -> K o e^G -> W; Q -> V
constexpr int PK_TT = 2 * kRegP;                // [T diag(beta); T diag(beta)], then U
constexpr int PK_AS = PK_TT + 16384;            // the chunk's gate logits, A, T (fp32 [64][68]), W' staging
constexpr int PK_G = PK_AS + 64 * kAs * 4;      // G (fp32 [64][132]); then the previous chunk's
                                                // logits and keys (o e^{G_C - G}), 16 KB each
constexpr int kPkSmem = PK_G + 64 * kGs * 4 + 1024;

struct PkCtl {
    uint64_t full, vfull, d2, d3, kprev, dm;   // kprev: the previous chunk's logits and keys
    PrepItem nxt;
    uint32_t tmem;
    float beta[kC], ones[kC];
    float tot[2][kDK];     // per key dimension: the decay summed over each half of a chunk
    float gcp[kDK];        // per key dimension: e^{G_C} of the previous chunk
};

// Four key dimensions of one row of a [K; Q] region (K rows 0-63, Q rows 64-127), widened.
template <typename IO>
__device__ __forceinline__ void pk_ld4(const uint8_t *reg, int row, int st, float (&x)[4]) {
    const uint2 u = *reinterpret_cast<const uint2 *>(reg + sw128_offset(row, st >> 1) + (st & 1) * 8);
    const float2 a = Pack<IO>::unpack(u.x), b = Pack<IO>::unpack(u.y);
    x[0] = a.x; x[1] = a.y; x[2] = b.x; x[3] = b.y;
}

// Persistent CTAs, two to an SM, walk the (chunk slot, value head) items with the grid's
// stride, as gdn_chunk_prep does, for the rules with decay and one decay per key dimension.
// Per item: K, Q and the gate logits by TMA, then G per key dimension (and beta); A and P
// on the FP32 cores; Q~, K~ out and K o e^G in place; T = (I + A)^-1 while V lands over
// the spent Q rows and the previous chunk's logits and keys over G; D2 = [T'; T'']
// (K o e^G) -> W; the previous chunk's gates scale its keys in place for M; D3 -> U;
// M = W (K_{c-1} o e^{G_C - G})^T.
template <typename IO>
__global__ void __launch_bounds__(kPrepThreads, 2) gdn_chunk_prep_pk(const __grid_constant__ TcParams p) {
    constexpr bool kBf16 = std::is_same<IO, __nv_bfloat16>::value;
    const bool has_delta = p.has_delta != 0;
    const bool beta_shared = p.beta_shared != 0;
    constexpr uint32_t kIdM = idesc_f16(kBf16, 128, 64, false, false);
    constexpr uint32_t kIdD2 = idesc_f16(kBf16, 128, 128, false, true);

    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                              ~static_cast<uintptr_t>(1023));
    __shared__ PkCtl ctl;
    const int pt = threadIdx.x, warp = pt >> 5, lane = pt & 31;
    const long long budget = p.wait_budget > 0 ? p.wait_budget : kWaitBudget;
    const int q = warp & 3, hf = warp >> 2;        // TMEM lane quarter, column half
    float *const As = reinterpret_cast<float *>(sm + PK_AS);
    float *const G = reinterpret_cast<float *>(sm + PK_G);
    const uint32_t aKQ = smem_u32(sm + PK_KQ), aTT = smem_u32(sm + PK_TT);
    const size_t tstride = (size_t)p.h_v * kDK;   // elements between tokens of a, Q~, K~
    if (warp == 0) {
        tmem_alloc(&ctl.tmem, kPrepCols);
        tmem_relinquish();
    }
    if (pt == 0) {
        mbar_init(&ctl.full, 1);
        mbar_init(&ctl.vfull, 1);
        mbar_init(&ctl.d2, 1);
        mbar_init(&ctl.d3, 1);
        mbar_init(&ctl.kprev, 1);
        mbar_init(&ctl.dm, 1);
        fence_mbar_init();
        ctl.nxt = prep_item(p, blockIdx.x);
    }
    if (pt < kC) ctl.ones[pt] = 1.f;
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = ctl.tmem;
    const uint32_t lane_base = static_cast<uint32_t>(32 * q) << 16;
    const int row = 32 * q + lane;
    const int gi = pt & (kDK - 1), gh = pt >> 7;    // gate work: key dimension, half chunk
    // mbarrier parities: full, vfull, d2 and d3 complete once per item, kprev and dm once
    // per item that is not a segment's first chunk.
    uint32_t ph = 0, phk = 0;
    // thread 0: 1 = V load, 4 = D2, 8 = K_{c-1} load, 16 = M, 32 = D3
    uint32_t issued = 0;
    bool ok = true, failed = false;
    for (int64_t item = blockIdx.x; item < p.prep_items; item += gridDim.x) {
    const PrepItem it = ctl.nxt;
    if (!it.valid) {
        __syncthreads();   // every thread has read ctl.nxt
        if (pt == 0) ctl.nxt = prep_item(p, item + gridDim.x);
        __syncthreads();
        continue;
    }
    const int h = it.h, hq = it.hq, Lc = it.Lc;
    const bool first = it.first != 0;
    const int64_t tc0 = it.tc0;
    uint8_t *rec = p.ws + ((size_t)it.slot * p.h_v + h) * kRecord;
    uint8_t *const rec_prev = rec - (size_t)p.h_v * kRecord;   // chunk c - 1, same head
    const size_t ahk = (size_t)h * kDK + gi;                  // this thread's A_log / dt_bias
    issued = 0;

    for (int e = pt; e < 16384 / 16; e += kPrepThreads)
        *reinterpret_cast<uint4 *>(sm + PK_TT + 16 * e) = make_uint4(0, 0, 0, 0);
    fence_async_smem();
    const int tok = (int)tc0;
    if (pt == 0) {
        mbar_arrive_expect_tx(&ctl.full, 6 * 8192);
#pragma unroll
        for (int r = 0; r < 2; ++r) {
            tma_load_3d(sm + PK_KQ + r * kRegP, &p.tm_k, r * 64, hq, tok, &ctl.full);
            tma_load_3d(sm + PK_KQ + r * kRegP + 8192, &p.tm_q, r * 64, hq, tok, &ctl.full);
            tma_load_3d(sm + PK_AS + r * 8192, &p.tm_a, r * 64, h, tok, &ctl.full);
        }
    }
    // G per key dimension from the logits tile: thread (gi, gh) sums tokens 32 gh .. 32 gh
    // + 31 of dimension gi; the second half adds the first half's sum after the barrier.
    // Padded tokens of a ragged chunk (the next sequence's rows) decay by nothing and have
    // beta 0.
    // g = -e^{A_log} softplus(a + dt_bias) for this thread's key dimension, in fp32 with the
    // fast exp / log (absolute error near 1e-7 per token; the scalar gates use the libm
    // forms, which cost several times more here, where every token has 128 gates).
    const float nA = -expf(p.A_log[ahk]), Db = p.dt_bias[ahk];
    auto gate = [&](float x) {
        const float y = x + Db;
        return nA * (fmaxf(y, 0.f) + __logf(1.f + __expf(-fabsf(y))));
    };
    if (pt < kC) {
        float be = 0.f;
        if (pt < Lc)
            be = has_delta ? sigmoid_f(IoType<IO>::ld(static_cast<const IO *>(p.b) +
                                                      (beta_shared ? (size_t)(tc0 + pt)
                                                                   : (size_t)(tc0 + pt) * p.h_v + h)))
                           : 1.f;
        ctl.beta[pt] = be;
    }
    ok = mbar_wait(&ctl.full, ph, budget);
    if (ok) {
        const uint8_t *at = sm + PK_AS + (gi >> 6) * 8192 + (gi & 7) * 2;
        float run = 0.f;
#pragma unroll 8
        for (int r = 0; r < 32; ++r) {
            const int t = 32 * gh + r;
            if (t < Lc) run += gate(IoType<IO>::ld(reinterpret_cast<const IO *>(at + sw128_offset(t, (gi & 63) >> 3))));
            G[t * kGs + gi] = run;
        }
        ctl.tot[gh][gi] = run;
    }
    failed = bar_any(kBarPrep, kPrepThreads, !ok);
    if (!failed && gh == 1) {
        const float off = ctl.tot[0][gi];
#pragma unroll 8
        for (int r = 0; r < 32; ++r) G[(32 + r) * kGs + gi] += off;
    }
    named_bar(kBarPrep, kPrepThreads);   // G and beta complete; the logits tile is spent
    if (!failed) {
        // A (times beta_t, fp32, to As) and P (times scale, to the record), s <= t.
        //  - The six 16 x 16 blocks below the diagonal (rows 16b .., columns 16a .., a < b),
        //    one warp each on tf32 warp MMAs: every term factors through the block's first
        //    row r = 16b, e^{G_t - G_r} e^{G_r - G_s} with s < r <= t, both factors <= 1, so
        //    A and P are products of (K, Q) o e^{G - G_r} and K o e^{G_r - G}.
        //  - Inside each diagonal block, its lower-left 8 x 8 part the same way through row
        //    16b + 8 (warps 6 and 7, the block's 8 K rows stacked over its 8 Q rows).
        //  - The 24 remaining 4 x 4 tiles on the FP32 cores: lane l takes key dimensions
        //    4l .. 4l + 3, below a tile's diagonal through its first row as above, on it per
        //    pair; the tile's 32 sums are reduced across the warp.
        {
            const uint8_t *kq = sm + PK_KQ;
            // Element (row, dimension) of the [K; Q] tiles (K rows 0-63, Q rows 64-127).
            auto el = [&](int r, int i) {
                return IoType<IO>::ld(reinterpret_cast<const IO *>(
                    kq + (i >> 6) * kRegP + sw128_offset(r, (i & 63) >> 3) + (i & 7) * 2));
            };
            if (warp < 6) {
                const int b = warp < 1 ? 1 : (warp < 3 ? 2 : 3);
                const int a = warp - (b * (b - 1)) / 2;
                const int rt = 16 * b, cs = 16 * a, g = lane >> 2, tq = lane & 3;
                float accA[2][4] = {}, accP[2][4] = {};
#pragma unroll 2
                for (int ks = 0; ks < 16; ++ks) {
                    const int d0 = 8 * ks + tq, d1 = d0 + 4;
                    const float r0 = G[rt * kGs + d0], r1 = G[rt * kGs + d1];
                    const float f00 = __expf(G[(rt + g) * kGs + d0] - r0), f10 = __expf(G[(rt + g + 8) * kGs + d0] - r0);
                    const float f01 = __expf(G[(rt + g) * kGs + d1] - r1), f11 = __expf(G[(rt + g + 8) * kGs + d1] - r1);
                    const uint32_t xk[4] = {to_tf32(el(rt + g, d0) * f00), to_tf32(el(rt + g + 8, d0) * f10),
                                            to_tf32(el(rt + g, d1) * f01), to_tf32(el(rt + g + 8, d1) * f11)};
                    const uint32_t xq[4] = {to_tf32(el(64 + rt + g, d0) * f00), to_tf32(el(64 + rt + g + 8, d0) * f10),
                                            to_tf32(el(64 + rt + g, d1) * f01), to_tf32(el(64 + rt + g + 8, d1) * f11)};
#pragma unroll
                    for (int nt = 0; nt < 2; ++nt) {
                        const int sc = cs + 8 * nt + g;
                        const uint32_t y[2] = {to_tf32(el(sc, d0) * __expf(r0 - G[sc * kGs + d0])),
                                               to_tf32(el(sc, d1) * __expf(r1 - G[sc * kGs + d1]))};
                        mma_tf32_16x8x8(accA[nt], xk, y);
                        mma_tf32_16x8x8(accP[nt], xq, y);
                    }
                }
                const float sc = p.scale;
#pragma unroll
                for (int nt = 0; nt < 2; ++nt) {
                    const int c = cs + 8 * nt + 2 * tq;
#pragma unroll
                    for (int hh = 0; hh < 2; ++hh) {
                        const int t = rt + g + 8 * hh;
                        const float bt = has_delta ? ctl.beta[t] : 0.f;
                        *reinterpret_cast<float2 *>(As + t * kAs + c) =
                            make_float2(bt * accA[nt][2 * hh], bt * accA[nt][2 * hh + 1]);
                        *reinterpret_cast<uint32_t *>(rec + REC_PM + sw128_offset(t, c >> 3) + (c & 7) * 2) =
                            Pack<IO>::two(sc * accP[nt][2 * hh], sc * accP[nt][2 * hh + 1]);
                    }
                }
                // The mirrored block above the diagonal is zero: rows 16a .., columns 16b ..
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int idx = lane + 32 * e, t = cs + (idx >> 3), c = rt + 2 * (idx & 7);
                    *reinterpret_cast<uint32_t *>(rec + REC_PM + sw128_offset(t, c >> 3) + (c & 7) * 2) = 0u;
                }
            }
            if (warp >= 6) {
                const int g = lane >> 2, tq = lane & 3;
#pragma unroll 1
                for (int bb = 2 * (warp - 6); bb < 2 * (warp - 6) + 2; ++bb) {
                    const int rt = 16 * bb + 8, cs = 16 * bb, t = rt + g;
                    float acc[4] = {};
#pragma unroll 2
                    for (int ks = 0; ks < 16; ++ks) {
                        const int d0 = 8 * ks + tq, d1 = d0 + 4;
                        const float r0 = G[rt * kGs + d0], r1 = G[rt * kGs + d1];
                        const float f0 = __expf(G[t * kGs + d0] - r0), f1 = __expf(G[t * kGs + d1] - r1);
                        const uint32_t x[4] = {to_tf32(el(t, d0) * f0), to_tf32(el(64 + t, d0) * f0),
                                               to_tf32(el(t, d1) * f1), to_tf32(el(64 + t, d1) * f1)};
                        const int sc = cs + g;
                        const uint32_t y[2] = {to_tf32(el(sc, d0) * __expf(r0 - G[sc * kGs + d0])),
                                               to_tf32(el(sc, d1) * __expf(r1 - G[sc * kGs + d1]))};
                        mma_tf32_16x8x8(acc, x, y);
                    }
                    const int c = cs + 2 * tq;
                    const float bt = has_delta ? ctl.beta[t] : 0.f;
                    *reinterpret_cast<float2 *>(As + t * kAs + c) = make_float2(bt * acc[0], bt * acc[1]);
                    *reinterpret_cast<uint32_t *>(rec + REC_PM + sw128_offset(t, c >> 3) + (c & 7) * 2) =
                        Pack<IO>::two(p.scale * acc[2], p.scale * acc[3]);
                    // Its mirror above the diagonal (rows 16b .., columns 16b + 8 ..) is zero.
                    const int tz = cs + g, cz = rt + 2 * tq;
                    *reinterpret_cast<uint32_t *>(rec + REC_PM + sw128_offset(tz, cz >> 3) + (cz & 7) * 2) = 0u;
                }
            }
            // The 4 x 4 tiles of the two 8 x 8 diagonal parts of each diagonal block (three
            // each): tile j = 6 (block) + 3 (part) + (0: upper diagonal, 1: below, 2: lower
            // diagonal); three tiles a warp.
            const int rg = lane >> 4, st = lane & 15, i4 = 4 * lane;
            const uint8_t *reg = kq + rg * kRegP;
            auto ldg = [&](int r, float (&x)[4]) {
                const float4 g4 = *reinterpret_cast<const float4 *>(G + r * kGs + i4);
                x[0] = g4.x; x[1] = g4.y; x[2] = g4.z; x[3] = g4.w;
            };
#pragma unroll 1
            for (int j = 3 * warp; j < 3 * warp + 3; ++j) {
                const int base = 16 * (j / 6) + 8 * ((j % 6) / 3), k3 = j % 3;
                const int rb = k3 == 0 ? 0 : 1, cb = k3 == 2 ? 1 : 0;
                const int t0 = base + 4 * rb, s0 = base + 4 * cb;
                float v[32];
                if (cb < rb) {
                    // Below the diagonal: e^{G_t - G_s} = e^{G_t - G_t0} e^{G_t0 - G_s}.
                    float g0[4], kc[4][4];
                    ldg(t0, g0);
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        float ks[4], gs[4];
                        pk_ld4<IO>(reg, s0 + c, st, ks);
                        ldg(s0 + c, gs);
#pragma unroll
                        for (int e = 0; e < 4; ++e) kc[c][e] = ks[e] * __expf(g0[e] - gs[e]);
                    }
#pragma unroll
                    for (int r = 0; r < 4; ++r) {
                        float kr[4], qr[4];
                        pk_ld4<IO>(reg, t0 + r, st, kr);
                        pk_ld4<IO>(reg, 64 + t0 + r, st, qr);
                        if (r > 0) {
                            float gt[4];
                            ldg(t0 + r, gt);
#pragma unroll
                            for (int e = 0; e < 4; ++e) {
                                const float f = __expf(gt[e] - g0[e]);
                                kr[e] *= f;
                                qr[e] *= f;
                            }
                        }
#pragma unroll
                        for (int c = 0; c < 4; ++c) {
                            float a = 0.f, pq = 0.f;
#pragma unroll
                            for (int e = 0; e < 4; ++e) {
                                a = fmaf(kr[e], kc[c][e], a);
                                pq = fmaf(qr[e], kc[c][e], pq);
                            }
                            v[4 * r + c] = a;
                            v[16 + 4 * r + c] = pq;
                        }
                    }
                } else {
                    // On the diagonal: e^{G_t - G_s} per pair s < t; P also takes s = t.
                    float kx[4][4], gx[4][4];
#pragma unroll
                    for (int r = 0; r < 4; ++r) {
                        pk_ld4<IO>(reg, t0 + r, st, kx[r]);
                        ldg(t0 + r, gx[r]);
                    }
#pragma unroll
                    for (int t = 0; t < 4; ++t) {
                        float qx[4];
                        pk_ld4<IO>(reg, 64 + t0 + t, st, qx);
#pragma unroll
                        for (int s = 0; s < 4; ++s) {
                            float a = 0.f, pq = 0.f;
                            if (s < t) {
#pragma unroll
                                for (int e = 0; e < 4; ++e) {
                                    const float w = kx[s][e] * __expf(gx[t][e] - gx[s][e]);
                                    a = fmaf(kx[t][e], w, a);
                                    pq = fmaf(qx[e], w, pq);
                                }
                            } else if (s == t) {
#pragma unroll
                                for (int e = 0; e < 4; ++e) pq = fmaf(qx[e], kx[t][e], pq);
                            }
                            v[4 * t + s] = a;
                            v[16 + 4 * t + s] = pq;
                        }
                    }
                }
                // Reduce-scatter over the warp: at each step a lane keeps the half of its
                // values that its lane bit selects and adds the partner's copy of it.
#pragma unroll
                for (int o = 16; o >= 1; o >>= 1) {
                    const bool up = (lane & o) != 0;
#pragma unroll
                    for (int k = 0; k < o; ++k) {
                        const float send = up ? v[k] : v[k + o];
                        const float keep = up ? v[k + o] : v[k];
                        v[k] = keep + __shfl_xor_sync(0xffffffffu, send, o);
                    }
                }
                const int r = (lane >> 2) & 3, c = lane & 3;
                if (lane < 16) {
                    const bool below = cb < rb || c < r;
                    const float b = has_delta ? ctl.beta[t0 + r] : 0.f;
                    As[(t0 + r) * kAs + s0 + c] = below ? b * v[0] : 0.f;
                } else {
                    const bool on = cb < rb || c <= r;
                    const int s = s0 + c;
                    IoType<IO>::st(reinterpret_cast<IO *>(rec + REC_PM + sw128_offset(t0 + r, s >> 3)) + (s & 7),
                                   on ? p.scale * v[0] : 0.f);
                    if (cb < rb) {   // the mirrored tile above the diagonal is zero
                        const int s2 = t0 + c;
                        IoType<IO>::st(reinterpret_cast<IO *>(rec + REC_PM + sw128_offset(s0 + r, s2 >> 3)) + (s2 & 7),
                                       0.f);
                    }
                }
            }
        }
        named_bar(kBarPrep, kPrepThreads);
        // Q~ and K~ to the workspace (real tokens only: the rows past a ragged chunk's end
        // belong to the next sequence), K o e^G in place for D2, and e^{G_C} per key
        // dimension to the gate record.  Thread: token row pt / 4, four 8-dimension groups.
        {
            const int t = pt >> 2;
            const float *Gt = G + t * kGs, *GC = G + (kC - 1) * kGs;
            IO *qdst = static_cast<IO *>(p.qt) + (size_t)(tc0 + t) * tstride + (size_t)h * kDK;
            IO *kdst = static_cast<IO *>(p.kt) + (size_t)(tc0 + t) * tstride + (size_t)h * kDK;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int cc = (pt & 3) + 4 * j, i = 8 * cc;
                uint8_t *kp = sm + PK_KQ + (cc >> 3) * kRegP + sw128_offset(t, cc & 7);
                const uint8_t *qp = sm + PK_KQ + (cc >> 3) * kRegP + sw128_offset(64 + t, cc & 7);
                float kx[8], qx[8], ko[8], g[8], gc[8];
                unpack8<IO>(*reinterpret_cast<const uint4 *>(kp), kx);
                unpack8<IO>(*reinterpret_cast<const uint4 *>(qp), qx);
                *reinterpret_cast<float4 *>(g) = *reinterpret_cast<const float4 *>(Gt + i);
                *reinterpret_cast<float4 *>(g + 4) = *reinterpret_cast<const float4 *>(Gt + i + 4);
                *reinterpret_cast<float4 *>(gc) = *reinterpret_cast<const float4 *>(GC + i);
                *reinterpret_cast<float4 *>(gc + 4) = *reinterpret_cast<const float4 *>(GC + i + 4);
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    const float e1 = __expf(g[e]);
                    ko[e] = kx[e] * __expf(gc[e] - g[e]);
                    qx[e] *= e1;
                    kx[e] *= e1;
                }
                *reinterpret_cast<uint4 *>(kp) = pack8<IO>(kx);
                if (t < Lc) {
                    *reinterpret_cast<uint4 *>(qdst + i) = pack8<IO>(qx);
                    *reinterpret_cast<uint4 *>(kdst + i) = pack8<IO>(ko);
                }
            }
            if (pt < kDK) {
                GateRec *grec = reinterpret_cast<GateRec *>(rec + REC_G);
                const float gc = __expf(GC[pt]);
                if (pt < 64) grec->gam[pt] = gc;
                else grec->kf[pt - 64] = gc;
                if (pt == 0) grec->gC = 1.f;
            }
        }
        // Q and G are spent: V lands over the Q rows and, for M and W', the previous
        // chunk's logits and keys over G, during the inversion (the generic reads above
        // come first).
        fence_async_smem();
        named_bar(kBarPrep, kPrepThreads);
        if (pt == 0) {
            mbar_arrive_expect_tx(&ctl.vfull, 2 * 8192);
#pragma unroll
            for (int r = 0; r < 2; ++r)
                tma_load_3d(sm + PK_KQ + r * kRegP + 8192, &p.tm_v, r * 64, h, tok, &ctl.vfull);
            issued |= 1;
            if (!first) {
                mbar_arrive_expect_tx(&ctl.kprev, 4 * 8192);
#pragma unroll
                for (int r = 0; r < 2; ++r) {
                    tma_load_3d(sm + PK_G + r * 8192, &p.tm_a, r * 64, h, tok - kC, &ctl.kprev);
                    tma_load_3d(sm + PK_G + 16384 + r * 8192, &p.tm_k, r * 64, hq, tok - kC, &ctl.kprev);
                }
                issued |= 8;
            }
        }
        auto next_item = [&](int t) {
            if (t == 0) ctl.nxt = prep_item(p, item + gridDim.x);
        };
        invert_chunk<IO>(As, sm + PK_TT, ctl.beta, ctl.ones, has_delta ? 1.f : 0.f, pt, next_item);
        fence_async_smem();
        tc_fence_before();
        named_bar(kBarPrep, kPrepThreads);
        if (pt == 0) {
            // D2 = [T'; T''] (K o e^G): W on lanes 0-63.
            tc_fence_after();
#pragma unroll
            for (int k = 0; k < 4; ++k)
                mma_f16(tmem, sw128_desc(aTT + k * 32, 16, 1024), sw128_desc(aKQ + k * 2048, kRegP, 1024),
                        kIdD2, k > 0);
            mma_commit(&ctl.d2);
            issued |= 4;
        }
        if (!first) {
            // The previous chunk (full: only a sequence's last chunk is ragged): its decay per
            // key dimension, G', and e^{G'_C - G'} applied to its keys in place, so that
            // M = W (K_{c-1} o e^{G'_C - G'})^T; e^{G'_C} scales W into W'.
            ok = mbar_wait(&ctl.kprev, phk, budget);
            float lg[32];
            float run = 0.f;
            const int col = (gi >> 6) * 8192 + (gi & 7) * 2, ch = (gi & 63) >> 3;
#pragma unroll
            for (int r = 0; r < 32; ++r) {
                if (ok) run += gate(IoType<IO>::ld(reinterpret_cast<const IO *>(sm + PK_G + col + sw128_offset(32 * gh + r, ch))));
                lg[r] = run;
            }
            ctl.tot[gh][gi] = run;
            named_bar(kBarPrep, kPrepThreads);
            const float gC = ctl.tot[0][gi] + ctl.tot[1][gi], off = gh ? ctl.tot[0][gi] : 0.f;
            if (gh == 0) ctl.gcp[gi] = __expf(gC);
            if (ok) {
                uint8_t *kp = sm + PK_G + 16384 + col;
#pragma unroll
                for (int r = 0; r < 32; ++r) {
                    IO *e = reinterpret_cast<IO *>(kp + sw128_offset(32 * gh + r, ch));
                    IoType<IO>::st(e, IoType<IO>::ld(e) * __expf(gC - (lg[r] + off)));
                }
            }
            fence_async_smem();
        }
        if (pt == 0) ok = ok && mbar_wait(&ctl.d2, ph, budget);
        failed = bar_any(kBarPrep, kPrepThreads, !ok);
    }
    if (!failed) {
        // W (fp32, lanes 0-63) in the I/O type over the spent K rows: the A operand of M and,
        // for a segment's first chunk, the record's W_0; W' = W diag(e^{G'_C}) for the
        // previous chunk's record, staged over the spent A/T tile.
        tc_fence_after();
        if (q < 2) {
#pragma unroll
            for (int c0 = 0; c0 < 64; c0 += 32) {
                uint32_t r[32];
                tmem_ld32(tmem + lane_base + 64 * hf + c0, r);
                tmem_ld_wait();
                float x[32];
#pragma unroll
                for (int e = 0; e < 32; ++e) x[e] = __uint_as_float(r[e]);
#pragma unroll
                for (int q8 = 0; q8 < 4; ++q8)
                    *reinterpret_cast<uint4 *>(sm + PK_KQ + hf * kRegP + sw128_offset(row, (c0 >> 3) + q8)) =
                        pack8<IO>(x + 8 * q8);
                if (!first) {
#pragma unroll
                    for (int e = 0; e < 32; ++e) x[e] *= ctl.gcp[64 * hf + c0 + e];
#pragma unroll
                    for (int q8 = 0; q8 < 4; ++q8)
                        *reinterpret_cast<uint4 *>(sm + PK_AS + hf * 8192 + sw128_offset(row, (c0 >> 3) + q8)) =
                            pack8<IO>(x + 8 * q8);
                }
            }
        }
        fence_async_smem();
        tc_fence_before();
        named_bar(kBarPrep, kPrepThreads);
        // D3 = [T'; T''] V (U on lanes 64-127) while W (or W') goes out.
        if (pt == 0) {
            if (first) {
#pragma unroll
                for (int r = 0; r < 2; ++r) bulk_store(rec + REC_W0 + r * 8192, sm + PK_KQ + r * kRegP, 8192);
            } else {
                bulk_store(rec_prev + REC_W, sm + PK_AS, 16384);
            }
            bulk_commit();
            ok = mbar_wait(&ctl.vfull, ph, budget);
            if (ok) {
                tc_fence_after();
#pragma unroll
                for (int k = 0; k < 4; ++k)
                    mma_f16(tmem, sw128_desc(aTT + k * 32, 16, 1024),
                            sw128_desc(aKQ + 8192 + k * 2048, kRegP, 1024), kIdD2, k > 0);
                mma_commit(&ctl.d3);
                issued |= 32;
                ok = mbar_wait(&ctl.d3, ph, budget);
            }
        }
        failed = bar_any(kBarPrep, kPrepThreads, !ok);
    }
    if (!failed) {
        // U (lanes 64-127) into the spent [T'; T''] tile, as the record's U image.
        tc_fence_after();
        if (q >= 2) {
            const int j = row - 64;
#pragma unroll
            for (int c0 = 0; c0 < 64; c0 += 32) {
                uint32_t r[32];
                tmem_ld32(tmem + lane_base + 64 * hf + c0, r);
                tmem_ld_wait();
                float x[32];
#pragma unroll
                for (int e = 0; e < 32; ++e) x[e] = __uint_as_float(r[e]);
#pragma unroll
                for (int q8 = 0; q8 < 4; ++q8)
                    *reinterpret_cast<uint4 *>(sm + PK_TT + hf * 8192 + sw128_offset(j, (c0 >> 3) + q8)) =
                        pack8<IO>(x + 8 * q8);
            }
        }
        fence_async_smem();
        tc_fence_before();
        named_bar(kBarPrep, kPrepThreads);
        // U goes out; then M = W (K_{c-1} o e^{G'_C - G'})^T (U has left TMEM).
        if (pt == 0) {
            bulk_store(rec + REC_U, sm + PK_TT, 16384);
            bulk_commit();
            if (!first) {
                tc_fence_after();
                const uint32_t aKp = smem_u32(sm + PK_G + 16384);
#pragma unroll
                for (int k = 0; k < 8; ++k)
                    mma_f16(tmem, sw128_desc(aKQ + (k >> 2) * kRegP + (k & 3) * 32, 16, 1024),
                            sw128_desc(aKp + (k >> 2) * 8192 + (k & 3) * 32, 16, 1024), kIdM, k > 0);
                mma_commit(&ctl.dm);
                issued |= 16;
                ok = mbar_wait(&ctl.dm, phk, budget);
            }
        }
        if (!first) {
            failed = bar_any(kBarPrep, kPrepThreads, !ok);
            if (!failed) {
                // M rows on lanes 0-63, staged over the spent V rows for the previous
                // chunk's record.
                tc_fence_after();
                if (q < 2) {
                    uint32_t r[32];
                    tmem_ld32(tmem + lane_base + 32 * hf, r);
                    tmem_ld_wait();
                    float x[32];
#pragma unroll
                    for (int e = 0; e < 32; ++e) x[e] = __uint_as_float(r[e]);
#pragma unroll
                    for (int q8 = 0; q8 < 4; ++q8)
                        *reinterpret_cast<uint4 *>(sm + PK_KQ + 8192 + sw128_offset(row, 4 * hf + q8)) =
                            pack8<IO>(x + 8 * q8);
                }
                fence_async_smem();
                named_bar(kBarPrep, kPrepThreads);
                if (pt == 0) {
                    bulk_store(rec_prev + REC_PM + 8192, sm + PK_KQ + 8192, 8192);
                    bulk_commit();
                }
            }
        }
    }
    if (failed) break;    // the whole CTA, with this item's parities and copies in flight
    if (pt == 0) bulk_wait_read();
    ph ^= 1u;
    if (!first) phk ^= 1u;
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    }   // items
    if (failed && pt == 0) {
        // Let the copies and MMAs already issued land before the CTA leaves (bounded).
        atomicOr(p.status, kDevTimeout);
        mbar_wait(&ctl.full, ph, kWaitBudget);
        if (issued & 1) mbar_wait(&ctl.vfull, ph, kWaitBudget);
        if (issued & 4) mbar_wait(&ctl.d2, ph, kWaitBudget);
        if (issued & 32) mbar_wait(&ctl.d3, ph, kWaitBudget);
        if (issued & 8) mbar_wait(&ctl.kprev, phk, kWaitBudget);
        if (issued & 16) mbar_wait(&ctl.dm, phk, kWaitBudget);
    }
    if (pt == 0) bulk_wait_read();   // the record stores have read their staging tiles
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, kPrepCols);
    }
}

// ===================================================================== state scan
// The chain runs one chunk ahead on W S: with S' = gamma_C S + K^T diag(e^{G_C - G}) Delta
// the state after chunk c,
//   W_{c+1} S' = W'_{c+1} S + M_{c+1} Delta,  W'_{c+1} = gamma_C W_{c+1},
//   M_{c+1} = W_{c+1} K^T diag(e^{G_C - G})   (64 x 64, chunk c's K and gates),
// so one M = 128 product X(c) = [P_c; M_{c+1}] Delta_c beside D4'(c) = [Q_c; W_{c+1}] S_c
// yields both o_c = scale diag(gamma) (rows 0-63 of D4') + (rows 0-63 of X) and
// W_{c+1} S_{c+1} = gamma_C (rows 64-127 of D4') + (rows 64-127 of X).  The next Delta waits only
// for X(c); the state update and D4'(c + 1) run beside it.  The prep of chunk c + 1
// writes W'_{c+1} and M_{c+1} into chunk c's record; the first chunk of a segment starts
// from W_0 S_0.
//
// Shared memory (from a 1024-aligned base): two stages, then the chain's own tiles.
constexpr int kRegion = 24576;                 // 192 rows x 128 B for 64 d_k: K | Q | W
constexpr int SS_KQW = 0;                      // K_c, Q_c (TMA) | W_{c+1}, two d_k regions
constexpr int SS_U = 2 * kRegion;              // this column half of U_c, 64 x 128 B
constexpr int SS_PM = SS_U + 8192;             // [P_c; M_{c+1}], 128 x 128 B
constexpr int SS_G = SS_PM + 16384;            // GateRec
constexpr int kScanStage = SS_G + 1024;        // 73 KB
constexpr int SS_SB = 2 * kScanStage;          // S in the I/O type, MN-major (d_k rows)
constexpr int SS_DB0 = SS_SB + 16384;          // Delta, MN-major (token rows)
constexpr int SS_DB1 = SS_DB0 + 8192;          // diag(e^{G_C - G}) Delta
constexpr int SS_OUT = SS_DB1 + 8192;          // output tile staging, two buffers
constexpr int kScanSmem = SS_OUT + 2 * 8192 + 1024;
// With the norm epilogue: the gate rows of two chunks (each state-warp thread copies its
// own row, so no barrier guards them), this half's norm scale, the per-row sums of squares
// of the two 32-column groups (two chunks), and the other half's row sums (four chunks),
// which the other CTA of the pair writes.
constexpr int SS_Z = SS_OUT + 2 * 8192;
constexpr int SS_NS = SS_Z + 2 * 8192;
constexpr int SS_SSP = SS_NS + 256;            // [chunk & 1][column group][row]
constexpr int SS_PEER = SS_SSP + 1024;         // [chunk & 3][row]
constexpr int kScanSmemNorm = SS_PEER + 1024 + 1024;
// A stage arrives in two parts with their own barriers: part B ([Q; W], read only by
// D4') is refilled as soon as D4' has run; part A (K, U, [P; M], gates) once the chunk's
// last MMA has run and every thread has read the gates.
constexpr uint32_t kTxA = 2 * 8192 + 8192 + 16384 + sizeof(GateRec);
constexpr uint32_t kTxB = 2 * 16384;
// TMEM columns: D4' at 0 / 64 and X at 128 / 192 by chunk parity, DS at 256.
constexpr uint32_t TS_D4 = 0, TS_X = 128, TS_DS = 256, kScanCols = 512;
constexpr int kChainWarps = 8;                 // Delta, state update, readout
// + an MMA-issue warp, a copy warp and two state warps (S rows 64-127, TMEM lanes 64-127)
constexpr int kScanAllThreads = 32 * kChainWarps + 128;
constexpr uint32_t kBarOut = 2;                // named barrier of the 128 readout threads
constexpr uint32_t kBarNorm = 3;               // named barrier of the 64 state-warp threads
constexpr int kLptMax = 128;                   // packed batches up to this size run longest first

struct ScanCtl {
    uint64_t full_a[2], full_b[2], full_w;     // stage parts landed; W_0
    uint64_t d4, ds, x;                        // MMA groups done (tcgen05.commit)
    uint64_t delta_ready, sb_ready, out_done;  // chain warps -> issuing warp
    uint64_t ld_b, ld_a;                       // copy warp -> issuing warp: phase c seen
    uint64_t drain;
    uint64_t peer_full[4];                     // norm: the other half's row sums of chunk c (c & 3)
    uint64_t o_staged[2], ob_free[2];          // norm: readout -> state warps, and back
    uint32_t tmem;
    int32_t abort;                             // a wait gave up: everyone leaves
    int32_t seq;
    int32_t cu[kLptMax + 1];
};

// Bounded wait that also gives up as soon as another thread has given up.  Waiting
// threads sleep in the barrier rather than poll, except the single thread that issues
// the MMAs, which polls so that it wakes the moment the phase completes.
template <bool kPoll = false>
__device__ __forceinline__ bool wait_or_abort(uint64_t *bar, uint32_t parity, volatile int32_t *abort,
                                              long long budget) {
    if (mbar_try_wait(bar, parity)) return true;
    const long long t0 = clock64();
    while (!(kPoll ? mbar_try_wait(bar, parity) : mbar_try_wait_sleep(bar, parity, 20000u))) {
        if (*abort) return false;
        if (clock64() - t0 > budget) {
            *abort = 1;
            return false;
        }
    }
    return true;
}

// The same, agreed by the whole warp: the tensor-memory loads that follow a wait are
// warp-wide instructions, so every lane must take the same branch after it.
__device__ __forceinline__ bool warp_wait_or_abort(uint64_t *bar, uint32_t parity, volatile int32_t *abort,
                                                   long long budget) {
    return __all_sync(0xffffffffu, wait_or_abort(bar, parity, abort, budget));
}

// The norm epilogue's wait for the other CTA of the pair: it stores its row sums into this
// CTA's shared memory and then arrives here with release at cluster scope, so this wait
// acquires at cluster scope.  Bounded, and it gives up as soon as another thread has.
__device__ __forceinline__ bool wait_peer_or_abort(uint64_t *bar, uint32_t parity,
                                                   volatile int32_t *abort, long long budget) {
    const uint32_t addr = smem_u32(bar);
    const long long t0 = clock64();
    for (;;) {
        uint32_t done;
        asm volatile(
            "{\n\t.reg .pred p;\n\t"
            "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2, %3;\n\t"
            "selp.u32 %0, 1, 0, p;\n\t}"
            : "=r"(done)
            : "r"(addr), "r"(parity), "r"(20000u)
            : "memory");
        if (done) return true;
        if (*abort) return false;
        if (clock64() - t0 > budget) {
            *abort = 1;
            return false;
        }
    }
}

// Scan CTAs: one per (sequence, value head, half of the 128 state columns).  Chunk c, with
// S_c in registers (fp32) and in SB (I/O type):
//   D4'(c) = [Q_c; W_{c+1}] S_c              issued once SB holds S_c      (commit d4)
//   Delta_c = U_c - (W_c S_c)                warps on TMEM lanes 64-127:
//                                            gamma_C(c - 1) D4'(c - 1) + X(c - 1)
//   DS(c) = K_c^T diag(e^{G_C - G}) Delta_c                                 (commit ds)
//   X(c) = [P_c; M_{c+1}] Delta_c                                          (commit x)
//   S_{c+1} = gamma_C S_c + DS(c), SB        readout warps (rows 0-63), state warps (64-127)
//   o_c = scale gamma (Q_c S_c) + P_c Delta_c    warps on lanes 0-63, overlapping chunk c + 1
// X phases: 0 is W_0 S_0 (into D4' block 1), c + 1 is X(c).  D4' and X alternate between
// two TMEM column blocks each.  One warp issues every MMA and copy; the chain warps wait only on the
// barriers of the work they consume, and it learns of their progress through arrival
// counts.
// kNorm: the gated RMS norm of each o row is applied in the readout.  The two column
// halves of a (sequence, head) run as a cluster pair; per chunk, each readout thread
// squares its 32 rounded o values, the two column groups are summed through shared
// memory, and each row's sum goes to the other CTA (a store into its shared memory, then
// an arrival on its barrier), so both halves scale the row by the same 1 / rms.
// kPK: one decay per key dimension (records of gdn_chunk_prep_pk): Q and K arrive already
// scaled (Q o e^G, K o e^{G_C - G}), W' carries e^{G_C} (gC = 1), and the state update
// scales S row i by e^{G_C,i} from the gate record (gam: rows 0-63, kf: rows 64-127).
template <typename IO, bool kNorm = false, bool kPK = false>
__global__ void __launch_bounds__(kScanAllThreads, 1) gdn_chunk_scan(const __grid_constant__ TcParams p) {
    constexpr bool kBf16 = std::is_same<IO, __nv_bfloat16>::value;
    constexpr uint32_t kIdNV = idesc_f16(kBf16, 128, kNV, false, true);
    constexpr uint32_t kIdDS = idesc_f16(kBf16, 128, kNV, true, true);

    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                              ~static_cast<uintptr_t>(1023));
    __shared__ ScanCtl ctl;
    volatile int32_t *abort = &ctl.abort;
    const long long budget = p.wait_budget > 0 ? p.wait_budget : kWaitBudget;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const bool issue_warp = (warp == kChainWarps);
    const bool copy_warp = (warp == kChainWarps + 1);
    const bool state_warp = (warp >= kChainWarps + 2);
    // Time-parallel job of this CTA: 0 is segment 0; 2k - 1 is segment k from a zero
    // state; 2k is segment k's operator pass (identity state, U = 0).
    int64_t unit = blockIdx.x;
    int job = 0;
    if (p.tp_seg > 0) {
        const int64_t units = (int64_t)p.num_seqs * p.h_v * (kDK / kNV);
        job = (int)(unit / units);
        unit %= units;
    }
    const int tseg = (job + 1) / 2;
    const bool op_pass = job > 0 && (job & 1) == 0;
    const int half = (int)(unit & 1);
    const int h = (int)((unit >> 1) % p.h_v);
    int64_t n = (unit >> 1) / p.h_v;
    const int hq = h / (p.h_v / p.h_qk);
    const int v0 = half * kNV;

    // Packed sequences of unequal length: CTA position n takes the n-th longest sequence
    // (ties by index), so that the longest chains start first.
    if (p.cu_seqlens != nullptr && p.num_seqs <= kLptMax) {
        for (int i = tid; i <= p.num_seqs; i += kScanAllThreads) ctl.cu[i] = p.cu_seqlens[i];
        __syncthreads();
        for (int j = tid; j < p.num_seqs; j += kScanAllThreads) {
            const int64_t lj = (int64_t)ctl.cu[j + 1] - ctl.cu[j];
            int rank = 0;
            for (int i = 0; i < p.num_seqs; ++i) {
                const int64_t li = (int64_t)ctl.cu[i + 1] - ctl.cu[i];
                rank += (li > lj) || (li == lj && i < j);
            }
            if (rank == n) ctl.seq = j;
        }
        __syncthreads();
        n = ctl.seq;
    }

    int64_t t0, t1;
    if (!seq_range(p.cu_seqlens, p.seqlen, p.num_seqs, p.status, n, t0, t1)) return;
    // This launch walks chunks [seg_begin, seg_end) of the sequence; below, chunk c
    // counts from the segment's first chunk, and t0 / L / base_slot are shifted to it.
    const int64_t all_chunks = (t1 - t0 + kC - 1) / kC;
    const int64_t seg_b = p.tp_seg > 0 ? (int64_t)tseg * p.tp_seg : p.seg_begin;
    const int64_t seg_e = p.tp_seg > 0 ? seg_b + p.tp_seg : p.seg_end;
    const int64_t cb = seg_b < all_chunks ? seg_b : all_chunks;
    const int64_t ce = seg_e < all_chunks ? seg_e : all_chunks;
    const int nchunks = (int)(ce - cb);
    const int64_t base_slot = slot_base(p, n) + cb;
    t0 += cb * kC;
    const int64_t L = t1 - t0;

    if (warp == 0) {
        tmem_alloc(&ctl.tmem, kScanCols);
        tmem_relinquish();
    }
    if (tid == 0) {
        for (int i = 0; i < 2; ++i) {
            mbar_init(&ctl.full_a[i], 1);
            mbar_init(&ctl.full_b[i], 1);
        }
        mbar_init(&ctl.full_w, 1);
        mbar_init(&ctl.d4, 1);
        mbar_init(&ctl.ds, 1);
        mbar_init(&ctl.x, 1);
        mbar_init(&ctl.delta_ready, kChainWarps / 2);   // the Delta warps
        mbar_init(&ctl.sb_ready, kChainWarps / 2 + 2);   // readout warps and state warps
        mbar_init(&ctl.out_done, kChainWarps / 2);
        mbar_init(&ctl.ld_b, 1);
        mbar_init(&ctl.ld_a, 1);
        mbar_init(&ctl.drain, 1);
        if (kNorm) {
            for (int i = 0; i < 4; ++i) mbar_init(&ctl.peer_full[i], 64);   // the other CTA's row sums
            for (int i = 0; i < 2; ++i) {
                mbar_init(&ctl.o_staged[i], 1);
                mbar_init(&ctl.ob_free[i], 1);
            }
        }
        ctl.abort = 0;
        fence_mbar_init();
        tma_prefetch_desc(&p.tm_k);
        tma_prefetch_desc(&p.tm_q);
        tma_prefetch_desc(op_pass ? &p.tm_r : &p.tm_o);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    // Both CTAs of the pair have initialised their barriers before either signals the other.
    if constexpr (kNorm) cluster_sync();
    const uint32_t tmem = ctl.tmem;
    const size_t sbase = ((size_t)n * p.h_v + h) * kDK * kDK;

    auto record = [&](int c) { return p.ws + (size_t)((base_slot + c) * p.h_v + h) * kRecord; };
    auto load_a = [&](int c) {   // K, U half, [P; M] and gates of chunk c into stage c & 1
        const int s = c & 1;
        uint8_t *st = sm + s * kScanStage;
        const uint8_t *rec = record(c);
        mbar_arrive_expect_tx(&ctl.full_a[s], kTxA);
#pragma unroll
        for (int r = 0; r < 2; ++r)
            tma_load_3d(st + SS_KQW + r * kRegion, &p.tm_k, r * 64, hq, (int)(t0 + (int64_t)c * kC),
                        &ctl.full_a[s]);
        bulk_load(st + SS_U, rec + REC_U + half * 8192, 8192, &ctl.full_a[s]);
        bulk_load(st + SS_PM, rec + REC_PM, 16384, &ctl.full_a[s]);
        bulk_load(st + SS_G, rec + REC_G, sizeof(GateRec), &ctl.full_a[s]);
    };
    auto load_b = [&](int c) {   // [Q_c; W_{c+1}] of chunk c into stage c & 1
        const int s = c & 1;
        uint8_t *st = sm + s * kScanStage;
        const uint8_t *rec = record(c);
        mbar_arrive_expect_tx(&ctl.full_b[s], kTxB);
#pragma unroll
        for (int r = 0; r < 2; ++r) {
            tma_load_3d(st + SS_KQW + r * kRegion + 8192, &p.tm_q, r * 64, hq, (int)(t0 + (int64_t)c * kC),
                        &ctl.full_b[s]);
            bulk_load(st + SS_KQW + r * kRegion + 16384, rec + REC_W + r * 8192, 8192, &ctl.full_b[s]);
        }
    };

    if (issue_warp) {
        // ------------------------------------------------------------ MMA issue
        if (lane == 0 && nchunks > 0) {
            const uint32_t aSB = smem_u32(sm + SS_SB), aDB0 = smem_u32(sm + SS_DB0),
                           aDB1 = smem_u32(sm + SS_DB1);
            bool b1_issued = false;
            // [rows 64-191 of a stage's regions] S into TMEM block `blk`.
            auto issue_qw = [&](int s, int blk) {
                tc_fence_after();
                const uint32_t aSt = smem_u32(sm + s * kScanStage);
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                    const uint32_t off = (k >> 2) * kRegion + 8192 + (k & 3) * 32;
                    mma_f16(tmem + TS_D4 + 64 * blk, sw128_desc(aSt + off, 16, 1024),
                            sw128_desc(aSB + k * 2048, 16384, 1024), kIdNV, k > 0);
                }
            };
            bool ok = true;
            do {
                // X phase 0: W_0 S_0 into block 1 (the Q~ rows there are unused).
                if (!(ok = wait_or_abort<true>(&ctl.sb_ready, 0, abort, budget) && wait_or_abort<true>(&ctl.full_w, 0, abort, budget))) break;
                issue_qw(1, 1);
                mma_commit(&ctl.x);
                // D4'(0) into block 0.
                if (!(ok = wait_or_abort<true>(&ctl.full_b[0], 0, abort, budget))) break;
                issue_qw(0, 0);
                mma_commit(&ctl.d4);
                // Stage 1's part B, once W_0 S_0 has read its rows.
                if (nchunks > 1) {
                    if (!(ok = wait_or_abort<true>(&ctl.x, 0, abort, budget))) break;
                    load_b(1);
                    b1_issued = true;
                }
            } while (false);
            for (int c = 0; ok && c < nchunks; ++c) {
                const int s = c & 1;
                const uint32_t aSt = smem_u32(sm + s * kScanStage);
                // DS(c) once Delta_c is in DB0 / DB1; the copy warp has seen X phase c
                // and sb_ready phase c, so neither can run two phases ahead of it.
                ok = wait_or_abort<true>(&ctl.delta_ready, c & 1, abort, budget) &&
                     wait_or_abort<true>(&ctl.full_a[s], (c >> 1) & 1, abort, budget) &&
                     (c == 0 || wait_or_abort<true>(&ctl.ld_a, (c - 1) & 1, abort, budget));
                if (!ok) break;
                tc_fence_after();
#pragma unroll
                for (int k = 0; k < 4; ++k)
                    mma_f16(tmem + TS_DS, sw128_desc(aSt + k * 2048, kRegion, 1024),
                            sw128_desc((kPK ? aDB0 : aDB1) + k * 2048, 8192, 1024), kIdDS, k > 0);
                mma_commit(&ctl.ds);
                // X(c) into block c & 1.  The readout of chunk c - 1 is done, so the readout
                // warps have seen X phase c, the X block of chunk c - 2 is free, and D4'
                // block (c + 1) & 1 is free for D4'(c + 1).
                if (c > 0 && !(ok = wait_or_abort<true>(&ctl.out_done, (c - 1) & 1, abort, budget))) break;
#pragma unroll
                for (int k = 0; k < 4; ++k)
                    mma_f16(tmem + TS_X + 64 * s, sw128_desc(aSt + SS_PM + k * 32, 16, 1024),
                            sw128_desc(aDB0 + k * 2048, 8192, 1024), kIdNV, k > 0);
                mma_commit(&ctl.x);
                if (c + 1 < nchunks) {
                    // D4'(c + 1) once SB holds S_{c+1} (and the copy warp has seen D4'(c)).
                    ok = wait_or_abort<true>(&ctl.sb_ready, (c + 1) & 1, abort, budget) &&
                         wait_or_abort<true>(&ctl.full_b[(c + 1) & 1], ((c + 1) >> 1) & 1, abort, budget) &&
                         wait_or_abort<true>(&ctl.ld_b, c & 1, abort, budget);
                    if (!ok) break;
                    issue_qw((c + 1) & 1, (c + 1) & 1);
                    mma_commit(&ctl.d4);
                }
            }
            if (!ok) {
                // Let the MMAs already issued (and stage 1's part B) finish before the CTA
                // leaves (bounded): one commit covers every earlier MMA of this thread.
                *abort = 1;
                if (b1_issued) mbar_wait(&ctl.full_b[1], 0, kWaitBudget);
                mma_commit(&ctl.drain);
                mbar_wait(&ctl.drain, 0, kWaitBudget);
            }
        }
        __syncwarp();
    } else if (copy_warp) {
        // ------------------------------------------------------------ stage copies
        if (lane == 0 && nchunks > 0) {
            int last_a[2] = {-1, -1}, last_b[2] = {-1, -1};
            mbar_arrive_expect_tx(&ctl.full_w, 16384);
#pragma unroll
            for (int r = 0; r < 2; ++r)
                bulk_load(sm + kScanStage + SS_KQW + r * kRegion + 16384, record(0) + REC_W0 + r * 8192, 8192,
                          &ctl.full_w);
            load_a(0);
            load_b(0);
            last_a[0] = 0;
            last_b[0] = 0;
            if (nchunks > 1) {
                load_a(1);
                last_a[1] = 1;
            }
            bool ok = true;
            for (int c = 0; ok && c < nchunks; ++c) {
                const int s = c & 1;
                // D4'(c) has read part B of stage s: refill it with chunk c + 2.  The
                // arrivals only say which phases this warp has seen, so they go first.
                if (!(ok = wait_or_abort(&ctl.d4, c & 1, abort, budget))) break;
                mbar_arrive(&ctl.ld_b);
                if (c + 2 < nchunks) {
                    load_b(c + 2);
                    last_b[s] = c + 2;
                }
                // X(c) has read the rest of stage s and every thread has read chunk c's
                // gates (they arrive on sb_ready after that): refill part A.
                if (!(ok = wait_or_abort(&ctl.x, (c + 1) & 1, abort, budget) &&
                           wait_or_abort(&ctl.sb_ready, (c + 1) & 1, abort, budget)))
                    break;
                mbar_arrive(&ctl.ld_a);
                if (c + 2 < nchunks) {
                    load_a(c + 2);
                    last_a[s] = c + 2;
                }
            }
            // Copies still in flight land before the CTA leaves (bounded).
            mbar_wait(&ctl.full_w, 0, kWaitBudget);
            for (int s2 = 0; s2 < 2; ++s2) {
                if (last_a[s2] >= 0) mbar_wait(&ctl.full_a[s2], (last_a[s2] >> 1) & 1, kWaitBudget);
                if (last_b[s2] >= 0) mbar_wait(&ctl.full_b[s2], (last_b[s2] >> 1) & 1, kWaitBudget);
            }
            if (!ok) *abort = 1;
        }
        __syncwarp();
    } else if (!state_warp) {
        // ------------------------------------------------------------ chain warps
        const int q = warp & 3, g = warp >> 2;     // TMEM lane quarter, 32-column group
        const int row = 32 * q + lane;             // this thread's TMEM lane
        const bool out_warp = q < 2;               // lanes 0-63: output rows
        const uint32_t lane_base = static_cast<uint32_t>(32 * q) << 16;
        IO *go = static_cast<IO *>(op_pass ? p.tp_r : p.o);
        const CUtensorMap *omap = op_pass ? &p.tm_r : &p.tm_o;
        // The readout warps hold S rows 0-63 (this thread's row, 32 columns); the Delta
        // warps hold none: rows 64-127 belong to the state warps.
        float S[32];                               // S[row][v0 + 32 g + e]
        if (op_pass || !out_warp) {
            // The identity, this thread's row and columns.
#pragma unroll
            for (int e = 0; e < 32; ++e) S[e] = (row == v0 + 32 * g + e) ? 1.f : 0.f;
        } else {
            const bool zero = p.state_in == nullptr || tseg > 0;
            const float4 *src = reinterpret_cast<const float4 *>(p.state_in + sbase + (size_t)row * kDK + v0 + 32 * g);
#pragma unroll
            for (int q4 = 0; q4 < 8; ++q4) {
                const float4 f = zero ? make_float4(0.f, 0.f, 0.f, 0.f) : src[q4];
                S[4 * q4] = f.x; S[4 * q4 + 1] = f.y; S[4 * q4 + 2] = f.z; S[4 * q4 + 3] = f.w;
            }
        }
        // S (fp32 registers) -> MN-major operand tile (rows = d_k), then tell the issuer.
        auto publish_sb = [&](bool write) {
            if (write) {
#pragma unroll
                for (int q8 = 0; q8 < 4; ++q8)
                    *reinterpret_cast<uint4 *>(sm + SS_SB + sw128_offset(row, 4 * g + q8)) = pack8<IO>(S + 8 * q8);
            }
            fence_async_smem();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&ctl.sb_ready);
        };
        if (out_warp) publish_sb(true);
        // Norm epilogue: the readout warps stage chunk c's rounded o in its output tile and
        // publish the rows' sums of squares (ssp, and the other CTA's peer_ss); the state
        // warps turn the tile into y one chunk later and store it.
        float *const ssp = reinterpret_cast<float *>(sm + SS_SSP);
        float *const peer_ss = reinterpret_cast<float *>(sm + SS_PEER);
        // o (or y) of chunk cc to its tile staging buffer, or row by row for a ragged chunk.
        auto store_rows = [&](int cc, const uint4 (&pk)[4]) {
            const int Lcc = (int)((L - (int64_t)cc * kC) < kC ? (L - (int64_t)cc * kC) : kC);
            if (Lcc == kC) {
                uint8_t *obb = sm + SS_OUT + (cc & 1) * 8192;
#pragma unroll
                for (int q8 = 0; q8 < 4; ++q8)
                    *reinterpret_cast<uint4 *>(obb + sw128_offset(row, 4 * g + q8)) = pk[q8];
            } else if (row < Lcc) {
                uint4 *dst = reinterpret_cast<uint4 *>(
                    go + ((size_t)(t0 + (int64_t)cc * kC + row) * p.h_v + h) * kDK + v0 + 32 * g);
#pragma unroll
                for (int q8 = 0; q8 < 4; ++q8) dst[q8] = pk[q8];
            }
        };
        auto is_tile = [&](int cc) { return L - (int64_t)cc * kC >= kC; };
        bool ok = true;
        float gC_prev = 1.f;   // e^{G_C} of chunk c - 1 (1 before the first: W_0 S_0 is exact)
        for (int c = 0; c < nchunks; ++c) {
            const int s = c & 1;
            const uint8_t *st = sm + s * kScanStage;
            const GateRec &gr = *reinterpret_cast<const GateRec *>(st + SS_G);
            // Every reader of the stage observes its arrival itself.  The gates are read
            // here: part A of the stage is refilled once every thread has arrived on sb_ready.
            ok = ok && warp_wait_or_abort(&ctl.full_a[s], (c >> 1) & 1, abort, budget);
            const float gC = ok ? gr.gC : 0.f;
            const float fo = (ok && out_warp) ? p.scale * (kPK ? 1.f : gr.gam[row]) : 0.f;   // o row scale
            // Decay of this thread's S row (readout warps): e^{G_C} or, per key, e^{G_C,row}.
            const float gS = kPK ? ((ok && out_warp) ? gr.gam[row] : 0.f) : gC;

            if (!out_warp) {
                // Delta_c = U_c - W_c S_c on lanes 64-127 (token rows), this thread's 32
                // columns; W_c S_c is the sum of blocks (c - 1) & 1 of D4' and X after X
                // phase c (D4' alone for c = 0: W_0 S_0).
                ok = ok && warp_wait_or_abort(&ctl.x, c & 1, abort, budget);
                if (ok) {
                    tc_fence_after();
                    const int j = row - 64;
                    const float kfj = kPK ? 1.f : gr.kf[j];
                    const uint32_t wcol = TS_D4 + 64 * ((c + 1) & 1), xcol = TS_X + 64 * ((c + 1) & 1);
#pragma unroll
                    for (int ps = 0; ps < 2; ++ps) {
                        uint32_t ws[16], xs[16];
                        tmem_ld16(tmem + lane_base + wcol + 32 * g + 16 * ps, ws);
                        if (c > 0) {
                            tmem_ld16(tmem + lane_base + xcol + 32 * g + 16 * ps, xs);
                        } else {
#pragma unroll
                            for (int e = 0; e < 16; ++e) xs[e] = 0u;   // +0.0f
                        }
                        float x[16];
#pragma unroll
                        for (int q8 = 0; q8 < 2; ++q8) {
                            const uint4 u = *reinterpret_cast<const uint4 *>(
                                st + SS_U + sw128_offset(j, 4 * g + 2 * ps + q8));
                            const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
                            for (int k2 = 0; k2 < 4; ++k2) {
                                const float2 t2 = Pack<IO>::unpack(w[k2]);
                                x[8 * q8 + 2 * k2] = t2.x;
                                x[8 * q8 + 2 * k2 + 1] = t2.y;
                            }
                        }
                        tmem_ld_wait();
                        if (op_pass) {
#pragma unroll
                            for (int e = 0; e < 16; ++e) x[e] = 0.f;
                        }
#pragma unroll
                        for (int e = 0; e < 16; ++e) x[e] -= fmaf(gC_prev, __uint_as_float(ws[e]), __uint_as_float(xs[e]));
#pragma unroll
                        for (int q8 = 0; q8 < 2; ++q8)
                            *reinterpret_cast<uint4 *>(sm + SS_DB0 + sw128_offset(j, 4 * g + 2 * ps + q8)) =
                                pack8<IO>(x + 8 * q8);
                        if constexpr (!kPK) {   // with per-key decay, K~ carries e^{G_C - G}
#pragma unroll
                            for (int e = 0; e < 16; ++e) x[e] *= kfj;
#pragma unroll
                            for (int q8 = 0; q8 < 2; ++q8)
                                *reinterpret_cast<uint4 *>(sm + SS_DB1 + sw128_offset(j, 4 * g + 2 * ps + q8)) =
                                    pack8<IO>(x + 8 * q8);
                        }
                    }
                }
                fence_async_smem();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&ctl.delta_ready);
                // The next Delta waits only for X(c): the state warps update rows 64-127.
                gC_prev = gC;
                if (!ok) break;
                continue;
            }

            // S_{c+1} = gamma_C S_c + DS(c) (fp32 registers), then the operand tile.
            ok = ok && warp_wait_or_abort(&ctl.ds, c & 1, abort, budget);
            if (ok) {
                tc_fence_after();
#pragma unroll
                for (int ps = 0; ps < 2; ++ps) {
                    uint32_t r[16];
                    tmem_ld16(tmem + lane_base + TS_DS + 32 * g + 16 * ps, r);
                    tmem_ld_wait();
#pragma unroll
                    for (int e = 0; e < 16; ++e) S[16 * ps + e] = fmaf(gS, S[16 * ps + e], __uint_as_float(r[e]));
                }
            }
            publish_sb(ok);

            // o_c = scale gamma (rows 0-63 of D4' block c & 1) + (rows 0-63 of X block
            // c & 1) after X(c), while chunk c + 1 runs.  A full
            // chunk goes out as one TMA store of the staged 64 x 64 tile; a sequence's
            // ragged last chunk is stored row by row so that no row of the next sequence
            // is touched.  The readout warps leave the loop together, at their barrier.
            ok = ok && warp_wait_or_abort(&ctl.x, (c + 1) & 1, abort, budget);
            uint4 packed[4];
            if (ok) {
                tc_fence_after();
#pragma unroll
                for (int ps = 0; ps < 2; ++ps) {
                    uint32_t r[16], rx[16];
                    tmem_ld16(tmem + lane_base + TS_D4 + 64 * s + 32 * g + 16 * ps, r);
                    tmem_ld16(tmem + lane_base + TS_X + 64 * s + 32 * g + 16 * ps, rx);
                    tmem_ld_wait();
                    float x[16];
#pragma unroll
                    for (int e = 0; e < 16; ++e) x[e] = fmaf(fo, __uint_as_float(r[e]), __uint_as_float(rx[e]));
                    packed[2 * ps] = pack8<IO>(x);
                    packed[2 * ps + 1] = pack8<IO>(x + 8);
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&ctl.out_done);
            }
            if constexpr (kNorm) {
                // The tile of chunk c - 2 has been turned into y and stored from this buffer.
                if (c >= 2) ok = ok && warp_wait_or_abort(&ctl.ob_free[c & 1], ((c - 2) >> 1) & 1, abort, budget);
                float ss = 0.f;
                if (ok) {
                    uint8_t *obb = sm + SS_OUT + (c & 1) * 8192;
#pragma unroll
                    for (int q8 = 0; q8 < 4; ++q8) {
                        *reinterpret_cast<uint4 *>(obb + sw128_offset(row, 4 * g + q8)) = packed[q8];
                        float v[8];
                        unpack8<IO>(packed[q8], v);
#pragma unroll
                        for (int i = 0; i < 8; ++i) ss = fmaf(v[i], v[i], ss);
                    }
                }
                ssp[128 * (c & 1) + 64 * g + row] = ss;
                named_bar(kBarOut, 128);
                if (ok && g == 0) {
                    const float local = ssp[128 * (c & 1) + row] + ssp[128 * (c & 1) + 64 + row];
                    const uint32_t peer = cluster_ctarank() ^ 1u;
                    st_cluster_f32(mapa_shared(smem_u32(peer_ss + 64 * (c & 3) + row), peer), local);
                    mbar_arrive_cluster(mapa_shared(smem_u32(&ctl.peer_full[c & 3]), peer));
                }
                if (tid == 0) mbar_arrive(&ctl.o_staged[c & 1]);   // after every readout thread's writes
            } else if (ok) {
                store_rows(c, packed);
            }
            fence_async_smem();
            if (tid == 0) bulk_wait_read();    // the previous tile store has read its buffer
            if (bar_any(kBarOut, 128, !ok)) {
                ok = false;
                break;
            }
            if (!kNorm && tid == 0 && is_tile(c)) {
                tma_store_3d(omap, sm + SS_OUT + (c & 1) * 8192, v0, h, (int)(t0 + (int64_t)c * kC));
                bulk_commit();
            }
        }
        if (tid == 0) bulk_wait_all();    // the output tiles have reached global memory
        if (ok && out_warp) {
            float *sdst = p.state_out;
            if (p.tp_seg > 0)
                sdst = (op_pass ? p.tp_phi : p.tp_psi) + (size_t)tseg * p.num_seqs * p.h_v * kDK * kDK;
            float4 *dst = reinterpret_cast<float4 *>(sdst + sbase + (size_t)row * kDK + v0 + 32 * g);
#pragma unroll
            for (int q4 = 0; q4 < 8; ++q4)
                dst[q4] = make_float4(S[4 * q4], S[4 * q4 + 1], S[4 * q4 + 2], S[4 * q4 + 3]);
        } else if (!ok) {
            *abort = 1;
        }
    } else {
        // ------------------------------------------------------------ state warps
        // S rows 64-127 (this thread's row, all 64 columns of the half): S_{c+1} =
        // gamma_C S_c + DS(c) from TMEM lanes 64-127, then the operand tile.
        const int q = warp & 3;                    // 2 or 3
        const int row = 32 * q + lane;
        const uint32_t lane_base = static_cast<uint32_t>(32 * q) << 16;
        float S[kNV];                              // S[row][v0 + e]
        if (op_pass) {
#pragma unroll
            for (int e = 0; e < kNV; ++e) S[e] = (row == v0 + e) ? 1.f : 0.f;
        } else {
            const bool zero = p.state_in == nullptr || tseg > 0;
            const float4 *src = reinterpret_cast<const float4 *>(p.state_in + sbase + (size_t)row * kDK + v0);
#pragma unroll
            for (int q4 = 0; q4 < kNV / 4; ++q4) {
                const float4 f = zero ? make_float4(0.f, 0.f, 0.f, 0.f) : src[q4];
                S[4 * q4] = f.x; S[4 * q4 + 1] = f.y; S[4 * q4 + 2] = f.z; S[4 * q4 + 3] = f.w;
            }
        }
        auto publish_rows = [&](bool write) {
            if (write) {
#pragma unroll
                for (int q8 = 0; q8 < kNV / 8; ++q8)
                    *reinterpret_cast<uint4 *>(sm + SS_SB + sw128_offset(row, q8)) = pack8<IO>(S + 8 * q8);
            }
            fence_async_smem();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&ctl.sb_ready);
        };
        publish_rows(true);

        // Norm epilogue (kNorm), one chunk behind the readout: this thread owns token row
        // nrow of the staged tile (all 64 columns of the half).  Chunk cc's gate row comes
        // in by cp.async at the top of iteration cc (one group per chunk, empty past the
        // end), so cp.async.wait_group 1 in iteration cc + 1 means it has landed.
        const int nrow = 32 * (warp - (kChainWarps + 2)) + lane;
        float *const nsc = reinterpret_cast<float *>(sm + SS_NS);
        const float *const ssp = reinterpret_cast<const float *>(sm + SS_SSP);
        const float *const peer_ss = reinterpret_cast<const float *>(sm + SS_PEER);
        const CUtensorMap *omap = &p.tm_o;
        auto fetch_gate = [&](int c2) {
            if (c2 < nchunks && (int64_t)nrow < L - (int64_t)c2 * kC) {
                const IO *src = static_cast<const IO *>(p.norm_gate) +
                                ((size_t)(t0 + (int64_t)c2 * kC + nrow) * p.h_v + h) * kDK + v0;
                uint8_t *dst = sm + SS_Z + (c2 & 1) * 8192;
#pragma unroll
                for (int i = 0; i < 8; ++i) cp_async16(dst + sw128_offset(nrow, i), src + 8 * i);
            }
            cp_async_commit();
        };
        // y = o * rsqrt(mean(o^2) + eps) * scale * act(gate) for chunk cc's rows, in place in
        // its staging tile (or straight to memory for a ragged chunk), then one TMA store.
        // Every state thread comes here, whatever ok says, for the barrier.
        auto norm_tile = [&](int cc, bool ok) -> bool {
            ok = ok && wait_or_abort(&ctl.o_staged[cc & 1], (cc >> 1) & 1, abort, budget) &&
                 wait_peer_or_abort(&ctl.peer_full[cc & 3], (cc >> 2) & 1, abort, budget);
            const int Lcc = (int)((L - (int64_t)cc * kC) < kC ? (L - (int64_t)cc * kC) : kC);
            uint8_t *obb = sm + SS_OUT + (cc & 1) * 8192;
            if (ok && nrow < Lcc) {
                const float local = ssp[128 * (cc & 1) + nrow] + ssp[128 * (cc & 1) + 64 + nrow];
                const float inv = rsqrtf((local + peer_ss[64 * (cc & 3) + nrow]) / (float)kDK + p.norm_eps);
                const uint8_t *zr = sm + SS_Z + (cc & 1) * 8192;
                uint4 *gdst = reinterpret_cast<uint4 *>(
                    static_cast<IO *>(p.o) + ((size_t)(t0 + (int64_t)cc * kC + nrow) * p.h_v + h) * kDK + v0);
                // Not unrolled: the warps of this CTA run several large code paths at once,
                // and an unrolled copy of this loop cost instruction-cache misses everywhere.
#pragma unroll 1
                for (int q8 = 0; q8 < 8; ++q8) {
                    float v[8], z[8], y[8];
                    unpack8<IO>(*reinterpret_cast<const uint4 *>(obb + sw128_offset(nrow, q8)), v);
                    unpack8<IO>(*reinterpret_cast<const uint4 *>(zr + sw128_offset(nrow, q8)), z);
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        const float sg = __fdividef(1.0f, 1.0f + __expf(-z[i]));
                        const float act = p.norm_silu ? z[i] * sg : sg;
                        y[i] = v[i] * inv * nsc[8 * q8 + i] * act;
                    }
                    if (Lcc == kC) *reinterpret_cast<uint4 *>(obb + sw128_offset(nrow, q8)) = pack8<IO>(y);
                    else gdst[q8] = pack8<IO>(y);
                }
            }
            fence_async_smem();
            if (bar_any(kBarNorm, 64, !ok)) return false;
            if (nrow == 0 && Lcc == kC) {
                tma_store_3d(omap, obb, v0, h, (int)(t0 + (int64_t)cc * kC));
                bulk_commit();
            }
            return true;
        };
        // Chunk cc's staging tile is free again once its store has read it.
        auto free_tile = [&](int cc) {
            if (nrow == 0) {
                bulk_wait_read();
                mbar_arrive(&ctl.ob_free[cc & 1]);
            }
        };
        if constexpr (kNorm) {
            nsc[nrow] = IoType<IO>::ld(static_cast<const IO *>(p.norm_scale) + v0 + nrow);
            named_bar(kBarNorm, 64);
        }

        bool ok = true;
        for (int c = 0; c < nchunks; ++c) {
            const int s = c & 1;
            if constexpr (kNorm) {
                fetch_gate(c);
                if (c >= 2) free_tile(c - 2);
            }
            const GateRec &gr = *reinterpret_cast<const GateRec *>(sm + s * kScanStage + SS_G);
            ok = ok && warp_wait_or_abort(&ctl.full_a[s], (c >> 1) & 1, abort, budget);
            const float gC = ok ? (kPK ? gr.kf[row - 64] : gr.gC) : 0.f;
            ok = ok && warp_wait_or_abort(&ctl.ds, c & 1, abort, budget);
            if (ok) {
                tc_fence_after();
#pragma unroll
                for (int ps = 0; ps < kNV / 16; ++ps) {
                    uint32_t r[16];
                    tmem_ld16(tmem + lane_base + TS_DS + 16 * ps, r);
                    tmem_ld_wait();
#pragma unroll
                    for (int e = 0; e < 16; ++e) S[16 * ps + e] = fmaf(gC, S[16 * ps + e], __uint_as_float(r[e]));
                }
            }
            publish_rows(ok);
            if constexpr (kNorm) {
                // ok is agreed by both state warps here (they meet at a barrier inside
                // norm_tile, and at one of their own in chunk 0), so they leave together.
                if (c >= 1) {
                    cp_async_wait<1>();
                    ok = norm_tile(c - 1, ok);
                } else {
                    ok = !bar_any(kBarNorm, 64, !ok);
                }
            }
            if (!ok) break;
        }
        if constexpr (kNorm) {
            // The last chunk's norm, and every store read and written before the CTA leaves.
            if (ok && nchunks > 0) {
                cp_async_wait<0>();
                ok = norm_tile(nchunks - 1, ok);
            }
            cp_async_wait<0>();
            if (nrow == 0) bulk_wait_all();
        }
        if (ok) {
            float *sdst = p.state_out;
            if (p.tp_seg > 0)
                sdst = (op_pass ? p.tp_phi : p.tp_psi) + (size_t)tseg * p.num_seqs * p.h_v * kDK * kDK;
            float4 *dst = reinterpret_cast<float4 *>(sdst + sbase + (size_t)row * kDK + v0);
#pragma unroll
            for (int q4 = 0; q4 < kNV / 4; ++q4)
                dst[q4] = make_float4(S[4 * q4], S[4 * q4 + 1], S[4 * q4 + 2], S[4 * q4 + 3]);
        } else {
            *abort = 1;
        }
    }
    tc_fence_before();
    __syncthreads();
    // Neither CTA of a pair leaves while the other may still write into its shared memory.
    if constexpr (kNorm) cluster_sync();
    if (tid == 0 && ctl.abort) atomicOr(p.status, kDevTimeout);
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, kScanCols);
    }
}

// ===================================================================== convolution pass
// The streaming form of the convolution before the scan: every (token, 8-channel group) of
// x once, written to q, k and v ([tokens][heads][128]) for the plain prep, and each
// sequence's present conv state by the thread that holds its last token.
//  - A CTA owns 256 channels over kPassChunk tokens. x comes in by TMA, a stage at a
//    time: 32 tokens and the 3 rows before them in one 256 x 35 box (rows outside x read
//    as zero), kPassDepth stages in flight. Warp 0 issues; each warp computes from a
//    stage once its `full` barrier completes, then releases it on `empty`.
//  - Thread (cg, tg) forms 8 channels x 4 tokens from seven shared-memory rows and stores
//    each token as one 16-byte store, so a warp writes whole 512-byte rows.
//  - Window rows before a sequence's first token come from its past conv state (zeros
//    without one). Four tokens that reach back past a sequence start, or run into the
//    next sequence, are formed one by one.
//  - Every wait is bounded. A CTA that gives up lets the copies it issued land before it
//    exits.
constexpr int kPassWidth = 256;                  // channels of a CTA
constexpr int kPassTokens = 32;                  // tokens of a stage
constexpr int kPassRows = kPassTokens + 3;       // rows of a stage
constexpr int kPassRowB = kPassWidth * 2;        // bytes of a row
constexpr int kPassBufB = kPassRows * kPassRowB;
constexpr int kPassDepth = 4;                    // stages in flight
constexpr int kPassChunk = 256;                  // tokens of a CTA
constexpr int kPassSmem = kPassDepth * kPassBufB + 128;
template <typename IO>
__global__ void __launch_bounds__(256, 2) conv_pass(const __grid_constant__ TcParams p,
                                                     const __grid_constant__ CUtensorMap tm_x) {
    extern __shared__ unsigned char pass_raw[];
    unsigned char *smem = reinterpret_cast<unsigned char *>(
        (reinterpret_cast<uintptr_t>(pass_raw) + 127) & ~static_cast<uintptr_t>(127));
    __shared__ uint64_t full[kPassDepth], empty[kPassDepth];
    __shared__ int32_t abort_flag;
    volatile int32_t *abort = &abort_flag;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int64_t T = p.cu_seqlens ? p.seqlen : p.seqlen * p.num_seqs;
    const int cbase = blockIdx.x * kPassWidth;
    const int64_t t_begin = (int64_t)blockIdx.y * kPassChunk;
    if (t_begin >= T) return;   // the whole CTA, before any barrier
    const int64_t t_end = t_begin + kPassChunk < T ? t_begin + kPassChunk : T;
    const int nstage = (int)((t_end - t_begin + kPassTokens - 1) / kPassTokens);
    const long long budget = p.wait_budget > 0 ? p.wait_budget : kWaitBudget;
    if (tid == 0) {
#pragma unroll
        for (int i = 0; i < kPassDepth; ++i) {
            mbar_init(&full[i], 1);    // the issuing lane, plus the copy's bytes
            mbar_init(&empty[i], 8);   // one arrival per warp
        }
        fence_mbar_init();
        abort_flag = 0;
    }
    __syncthreads();

    // Warp 0: stage st into its buffer once the stage before it there has been released.
    auto issue = [&](int st) -> bool {
        const int i = st % kPassDepth;
        if (st >= kPassDepth && !warp_wait_or_abort(&empty[i], (uint32_t)(st / kPassDepth - 1) & 1u, abort, budget))
            return false;
        if (lane == 0) {
            mbar_arrive_expect_tx(&full[i], kPassBufB);
            tma_load_3d(smem + i * kPassBufB, &tm_x, cbase, (int)(t_begin + (int64_t)st * kPassTokens - 3), 0,
                        &full[i]);
        }
        return true;
    };

    const int cg = lane, tg = warp;
    const int c0 = cbase + 8 * cg;
    const bool live = c0 < p.conv_C;
    const int hk = p.h_qk * kDK;
    IO *dst = nullptr;
    int64_t stride = 0;
    ConvTaps taps = {};
    if (live) {
        if (c0 < hk) { dst = static_cast<IO *>(p.cq) + c0; stride = hk; }
        else if (c0 < 2 * hk) { dst = static_cast<IO *>(p.ck) + (c0 - hk); stride = hk; }
        else { dst = static_cast<IO *>(p.cv) + (c0 - 2 * hk); stride = (int64_t)p.h_v * kDK; }
        taps = conv_taps<IO>(p, c0);
    }
    // The sequence of token t: batched, t / seqlen; packed, the last n with cu[n] <= t.
    auto seq_of = [&](int64_t t, int64_t &n, int64_t &ts, int64_t &te) {
        if (p.cu_seqlens == nullptr) {
            n = t / p.seqlen;
        } else {
            int64_t lo = 0, hi = p.num_seqs - 1;
            while (lo < hi) {
                const int64_t mid = (lo + hi + 1) >> 1;
                if (p.cu_seqlens[mid] <= t) lo = mid; else hi = mid - 1;
            }
            n = lo;
        }
        return seq_range(p.cu_seqlens, p.seqlen, p.num_seqs, p.status, n, ts, te);
    };

    int issued = 0;   // warp 0: stages issued so far
    bool ok = true, bad = !live;
    if (warp == 0) {
        if (lane == 0) tma_prefetch_desc(&tm_x);
        for (; issued < kPassDepth - 1 && issued < nstage; ++issued) issue(issued);
    }
    int64_t n = -1, ts = 0, te = 0;   // the sequence of the tokens at hand
    for (int st = 0; st < nstage; ++st) {
        if (warp == 0 && issued < nstage) {
            if (!issue(issued)) ok = false;
            else ++issued;
        }
        if (ok && !warp_wait_or_abort(&full[st % kPassDepth], (uint32_t)(st / kPassDepth) & 1u, abort, budget))
            ok = false;
        if (!ok) break;
        // Buffer row r holds token s0 - 3 + r.
        const unsigned char *buf = smem + (st % kPassDepth) * kPassBufB;
        const int64_t s0 = t_begin + (int64_t)st * kPassTokens;
        const int64_t t0 = s0 + 4 * tg;
        auto srow = [&](int64_t pos) {
            return *reinterpret_cast<const uint4 *>(buf + (int)(pos - s0 + 3) * kPassRowB + cg * 16);
        };
        if (!bad && t0 < t_end) {
            if (t0 >= te && !seq_of(t0, n, ts, te)) bad = true;
        }
        if (!bad && t0 < t_end) {
            if (t0 - 3 >= ts && t0 + 3 < te && t0 + 3 < t_end) {
                conv4<IO>(p, taps, t0, srow, [&](int e, const uint4 &u) {
                    *reinterpret_cast<uint4 *>(dst + (size_t)(t0 + e) * stride) = u;
                });
                if (te - 1 == t0 + 3) conv_state_group<IO>(p, n, ts, te, c0);
            } else {
                for (int e = 0; e < 4 && !bad; ++e) {
                    const int64_t t = t0 + e;
                    if (t >= t_end) break;
                    if (t >= te && !seq_of(t, n, ts, te)) {
                        bad = true;
                        break;
                    }
                    // Rows before the sequence's first token: its past conv state.
                    auto row = [&](int64_t pos) -> uint4 {
                        if (pos >= ts) return srow(pos);
                        const int64_t r = (p.conv_k - 1) + (pos - ts);
                        if (p.conv_in == nullptr || r < 0) return make_uint4(0, 0, 0, 0);
                        return *reinterpret_cast<const uint4 *>(static_cast<const IO *>(p.conv_in) +
                                                                ((size_t)n * (p.conv_k - 1) + r) * p.conv_C + c0);
                    };
                    *reinterpret_cast<uint4 *>(dst + (size_t)t * stride) = conv1<IO>(p, taps, t, row);
                    if (t == te - 1) conv_state_group<IO>(p, n, ts, te, c0);
                }
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[st % kPassDepth]);
    }
    if (!ok) {
        if (tid == 0) atomicOr(p.status, kDevTimeout);
        if (warp == 0) {
            // Let the copies this CTA issued land before it exits: the latest phase of
            // each buffer's `full` barrier.
            for (int s2 = issued - kPassDepth < 0 ? 0 : issued - kPassDepth; s2 < issued; ++s2)
                mbar_wait(&full[s2 % kPassDepth], (uint32_t)(s2 / kPassDepth) & 1u, kWaitBudget);
        }
    }
}

// ===================================================================== conv state, empty sequences
// The present conv state of a packed sequence with no tokens is its past state (zeros
// without one); the prep writes it for every other sequence.  One CTA per sequence.
template <typename IO>
__global__ void __launch_bounds__(256) conv_state_empty(const __grid_constant__ TcParams p) {
    const int64_t n = blockIdx.x;
    int64_t t0, t1;
    if (!seq_range(p.cu_seqlens, p.seqlen, p.num_seqs, p.status, n, t0, t1) || t1 > t0) return;
    const size_t cnt = (size_t)(p.conv_k - 1) * p.conv_C;
    IO *dst = static_cast<IO *>(p.conv_out) + n * cnt;
    const IO *src = p.conv_in != nullptr ? static_cast<const IO *>(p.conv_in) + n * cnt : nullptr;
    for (size_t e = threadIdx.x; e < cnt; e += blockDim.x)
        IoType<IO>::st(dst + e, src != nullptr ? IoType<IO>::ld(src + e) : 0.f);
}

// ===================================================================== time-parallel combine
// The state entering segment k of a sequence: S_1 = Psi_0 (segment 0 ran from state_in),
// S_{k+1} = Phi_k S_k + Psi_k.  One launch per step k: a CTA owns a 32 x 32 tile of
// S_{k+1} for one (sequence, head), with its 32 rows of Phi_k and 32 columns of S_k staged
// in shared memory, and writes it over Psi_k (each element is read, then written, by one
// thread), so Psi_k holds S_{k+1} afterwards and Psi_{k-1} holds S_k, in fp32, for the
// correction below; the last step writes state_out as well.
template <typename IO>
__global__ void __launch_bounds__(256) gdn_tp_combine(const __grid_constant__ TcParams p, int k) {
    __shared__ float Ph[32][kDK + 1];     // rows rb .. rb + 31 of Phi_k
    __shared__ float Sc[kDK][33];         // columns cb .. cb + 31 of S_k
    const size_t off = (size_t)blockIdx.x * kDK * kDK;           // (n, h) slab
    const size_t slab = (size_t)p.num_seqs * p.h_v * kDK * kDK;   // one segment
    const int cb = 32 * (blockIdx.y & 3), rb = 32 * (blockIdx.y >> 2);
    const int tid = threadIdx.x;
    const float *sprev = p.tp_psi + (size_t)(k - 1) * slab + off;   // S_k
    const float *phi = p.tp_phi + (size_t)k * slab + off;
    float *psi = p.tp_psi + (size_t)k * slab + off;
    // All 32 loads of a thread in flight at once, then the stores to shared memory.
    float ph[16], sc[16];
#pragma unroll
    for (int u = 0; u < 16; ++u) {
        const int e = tid + 256 * u;
        ph[u] = phi[(size_t)(rb + (e >> 7)) * kDK + (e & 127)];
        sc[u] = sprev[(size_t)(e >> 5) * kDK + cb + (e & 31)];
    }
#pragma unroll
    for (int u = 0; u < 16; ++u) {
        const int e = tid + 256 * u;
        Ph[e >> 7][e & 127] = ph[u];
        Sc[e >> 5][e & 31] = sc[u];
    }
    __syncthreads();
    // Thread: column j, rows i0 .. i0 + 3.
    const int j = tid & 31, i0 = 4 * (tid >> 5);
    float acc[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) acc[i] = psi[(size_t)(rb + i0 + i) * kDK + cb + j];
#pragma unroll 8
    for (int m = 0; m < kDK; ++m) {
        const float sv = Sc[m][j];
#pragma unroll
        for (int i = 0; i < 4; ++i) acc[i] = fmaf(Ph[i0 + i][m], sv, acc[i]);
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const size_t at = (size_t)(rb + i0 + i) * kDK + cb + j;
        psi[at] = acc[i];
        if (k == p.tp_nseg - 1) p.state_out[off + at] = acc[i];
    }
}

// ===================================================================== time-parallel correction
// o_t += R_t S_k for the tokens t of segment k >= 1, where o_t came from the run of the
// segment from a zero state and R_t from its operator pass.  One CTA per (sequence, head,
// segment k, 128-token tile): D = R_tile S_k on tcgen05 (M = 128 tokens, N = 128 value
// columns, K = 128 key rows), with R by TMA and S_k read in fp32 and split into two 16-bit
// parts S_hi + S_lo (S_k - S_hi rounded), so that S_k enters the product to about 2^-16
// relative; then o = round(o + D) row by row.
constexpr int kCorrThreads = 128;
constexpr int CR_R = 0;               // R tile: 2 d_k regions of 128 token rows (K-major)
constexpr int CR_SH = 32768;          // S_hi: 2 d_v regions of 128 d_k rows (MN-major)
constexpr int CR_SL = 65536;          // S_lo
constexpr int kCorrSmem = 98304 + 1024;

// x rounded to the nearest value of the I/O type, as a float.
template <typename IO>
__device__ __forceinline__ float round_io(float x) {
    const float2 r = Pack<IO>::unpack(Pack<IO>::two(x, 0.f));
    return r.x;
}

template <typename IO>
__global__ void __launch_bounds__(kCorrThreads) gdn_tp_correct(const __grid_constant__ TcParams p) {
    constexpr bool kBf16 = std::is_same<IO, __nv_bfloat16>::value;
    constexpr uint32_t kId = idesc_f16(kBf16, 128, 128, false, true);
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                              ~static_cast<uintptr_t>(1023));
    __shared__ uint64_t full, done;
    __shared__ uint32_t tmem_base;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int unit = blockIdx.x;                       // (sequence, head)
    const int h = unit % p.h_v;
    const int64_t n = unit / p.h_v;
    const int tiles = (p.tp_seg + 1) / 2;              // 128-token tiles per segment
    const int k = 1 + (int)(blockIdx.y / tiles);
    const int tile = (int)(blockIdx.y % tiles);
    const int64_t seg0 = (int64_t)k * p.tp_seg * kC;
    const int64_t seg1 = seg0 + (int64_t)p.tp_seg * kC < p.seqlen ? seg0 + (int64_t)p.tp_seg * kC : p.seqlen;
    const int64_t tb = seg0 + (int64_t)tile * 128;
    if (tb >= seg1) return;
    const int rows = (int)(seg1 - tb < 128 ? seg1 - tb : 128);
    const int64_t tok0 = n * p.seqlen + tb;            // batched layout (the path runs batched calls only)

    if (warp == 0) {
        tmem_alloc(&tmem_base, 128);
        tmem_relinquish();
    }
    if (tid == 0) {
        mbar_init(&full, 1);
        mbar_init(&done, 1);
        fence_mbar_init();
    }
    __syncthreads();
    if (tid == 0) {
        mbar_arrive_expect_tx(&full, 4 * 8192);
#pragma unroll
        for (int r = 0; r < 2; ++r) {
            tma_load_3d(sm + CR_R + r * 16384, &p.tm_r, r * 64, h, (int)tok0, &full);
            tma_load_3d(sm + CR_R + r * 16384 + 8192, &p.tm_r, r * 64, h, (int)(tok0 + 64), &full);
        }
    }
    // This thread's row of o (token tok0 + tid), read now so that the loads overlap the
    // rest; rows past the segment's end are neither read nor written.
    const bool live = tid < rows;
    IO *const orow = static_cast<IO *>(p.o) + ((size_t)(tok0 + (live ? tid : 0)) * p.h_v + h) * kDK;
    uint4 ov[16];
    if (live) {
#pragma unroll
        for (int q = 0; q < 16; ++q) ov[q] = reinterpret_cast<const uint4 *>(orow)[q];
    }
    // S_k (fp32, row-major [d_k][d_v]) -> S_hi, S_lo in 16-byte chunks of 8 value columns
    // (128-byte swizzle); a warp reads two whole rows (1 KiB) per step, eight steps in flight.
    {
        const float *S = p.tp_psi + ((size_t)(k - 1) * p.num_seqs * p.h_v + (size_t)unit) * kDK * kDK;
#pragma unroll
        for (int half = 0; half < 2; ++half) {
            float4 a[8], b[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const int e = tid + kCorrThreads * (8 * half + i);
                const float4 *src = reinterpret_cast<const float4 *>(S + (size_t)(e >> 4) * kDK) + 2 * (e & 15);
                a[i] = src[0];
                b[i] = src[1];
            }
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const int e = tid + kCorrThreads * (8 * half + i);
                const int row = e >> 4, ch = e & 15;
                const float x[8] = {a[i].x, a[i].y, a[i].z, a[i].w, b[i].x, b[i].y, b[i].z, b[i].w};
                float hi[8], lo[8];
#pragma unroll
                for (int q = 0; q < 8; ++q) {
                    hi[q] = round_io<IO>(x[q]);
                    lo[q] = x[q] - hi[q];
                }
                const uint32_t off = (ch >> 3) * 16384 + sw128_offset(row, ch & 7);
                *reinterpret_cast<uint4 *>(sm + CR_SH + off) = pack8<IO>(hi);
                *reinterpret_cast<uint4 *>(sm + CR_SL + off) = pack8<IO>(lo);
            }
        }
    }
    fence_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_base;
    bool ok = true;
    if (tid == 0) {
        const long long budget = p.wait_budget > 0 ? p.wait_budget : kWaitBudget;
        bool issued = false;
        ok = mbar_wait(&full, 0, budget);
        if (ok) {
            tc_fence_after();
            const uint32_t aR = smem_u32(sm + CR_R), aH = smem_u32(sm + CR_SH), aL = smem_u32(sm + CR_SL);
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {
                const uint64_t da = sw128_desc(aR + (kk >> 2) * 16384 + (kk & 3) * 32, 16, 1024);
                mma_f16(tmem, da, sw128_desc(aH + kk * 2048, 16384, 1024), kId, kk > 0);
                mma_f16(tmem, da, sw128_desc(aL + kk * 2048, 16384, 1024), kId, 1u);
            }
            mma_commit(&done);
            issued = true;
            ok = mbar_wait(&done, 0, budget);
        }
        if (!ok) {
            // Let the copy and the MMAs already issued land before the CTA leaves (bounded).
            atomicOr(p.status, kDevTimeout);
            mbar_wait(&full, 0, kWaitBudget);
            if (issued) mbar_wait(&done, 0, kWaitBudget);
        }
    }
    ok = !bar_any(kBarPrep, kCorrThreads, !ok);       // the same value in every thread
    if (ok) {
        // Thread = token row tid (its TMEM lane): o = round(o + D).  The tensor-memory load
        // is a warp-wide instruction, so every lane takes it; rows past the segment's end
        // skip only their global read and write.
        tc_fence_after();
#pragma unroll
        for (int c0 = 0; c0 < kDK; c0 += 32) {
            uint32_t r[32];
            __syncwarp();                              // every lane at the warp-wide load
            tmem_ld32(tmem + (static_cast<uint32_t>(32 * warp) << 16) + c0, r);
            tmem_ld_wait();
            if (!live) continue;
#pragma unroll
            for (int q8 = 0; q8 < 4; ++q8) {
                const uint4 u = ov[c0 / 8 + q8];
                const uint32_t w[4] = {u.x, u.y, u.z, u.w};
                float x[8];
#pragma unroll
                for (int k2 = 0; k2 < 4; ++k2) {
                    const float2 t2 = Pack<IO>::unpack(w[k2]);
                    x[2 * k2] = t2.x + __uint_as_float(r[8 * q8 + 2 * k2]);
                    x[2 * k2 + 1] = t2.y + __uint_as_float(r[8 * q8 + 2 * k2 + 1]);
                }
                reinterpret_cast<uint4 *>(orow)[c0 / 8 + q8] = pack8<IO>(x);
            }
        }
    }
    // Rows past the segment's end (and every row after a failed wait) are left as they are.
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, 128);
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



// Streaming multiprocessors of the current device (looked up once per device; 0 when
// there is no device).
int sm_count() {
    static int cache[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
    if (cache[dev] == 0) {
        int v = 0;
        if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
        cache[dev] = v;
    }
    return cache[dev];
}

constexpr int kMaxSegments = 4;
constexpr int kMinSegmentChunks = 32;

// An internal stream and events of the current device, created on first use, on which
// the prep of later chunk segments runs beside the scan of earlier ones.
struct SideStream {
    cudaStream_t stream = nullptr;
    cudaEvent_t ev[kMaxSegments] = {};
    bool ready = false;
    std::mutex launch_mu;   // one call's event records and waits at a time
};
SideStream *side_stream() {
    static SideStream cache[64];
    static std::mutex mu;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
    std::lock_guard<std::mutex> lock(mu);
    SideStream &s = cache[dev];
    if (!s.ready) {
        if (cudaStreamCreateWithFlags(&s.stream, cudaStreamNonBlocking) != cudaSuccess) return nullptr;
        for (int i = 0; i < kMaxSegments; ++i)
            if (cudaEventCreateWithFlags(&s.ev[i], cudaEventDisableTiming) != cudaSuccess) return nullptr;
        s.ready = true;
    }
    return &s;
}

// The kernels' dynamic shared-memory limits, a per-device function attribute (set once
// per device and I/O type).
// Resident prep CTAs per device and I/O type (SMs x CTAs per SM), set by configure().
int g_prep_slots[64][2] = {};
int g_prep_pk_slots[64][2] = {};   // the same for the per-key prep

template <typename IO>
cudaError_t configure() {
    static bool configured[64] = {false};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (!configured[dev]) {
        e = cudaFuncSetAttribute(gdn_chunk_prep<IO, false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 kPrepSmem);
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(gdn_chunk_prep<IO, true>,
                                     cudaFuncAttributeMaxDynamicSharedMemorySize, kPrepSmem);
        // Three prep CTAs to an SM need the largest shared-memory carve-out.
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(gdn_chunk_prep<IO, false>, cudaFuncAttributePreferredSharedMemoryCarveout,
                                     (int)cudaSharedmemCarveoutMaxShared);
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(gdn_chunk_prep<IO, true>, cudaFuncAttributePreferredSharedMemoryCarveout,
                                     (int)cudaSharedmemCarveoutMaxShared);
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(gdn_chunk_prep<IO, false, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     kPrepSmem);
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(gdn_chunk_prep<IO, false, true>, cudaFuncAttributePreferredSharedMemoryCarveout,
                                     (int)cudaSharedmemCarveoutMaxShared);
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(gdn_chunk_prep_pk<IO>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     kPkSmem);
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(gdn_chunk_prep_pk<IO>, cudaFuncAttributePreferredSharedMemoryCarveout,
                                     (int)cudaSharedmemCarveoutMaxShared);
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(gdn_chunk_scan<IO>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     kScanSmem);
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(gdn_chunk_scan<IO, false, true>,
                                     cudaFuncAttributeMaxDynamicSharedMemorySize, kScanSmem);
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(gdn_chunk_scan<IO, true>,
                                     cudaFuncAttributeMaxDynamicSharedMemorySize, kScanSmemNorm);
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(gdn_tp_correct<IO>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     kCorrSmem);
        if (e != cudaSuccess) return e;
        // Persistent prep CTAs: as many as the SMs' shared memory holds, at most the three
        // the launch bounds size the registers for.
        int sms = 0, smem_sm = 0, reserved = 0;
        cudaFuncAttributes fa;
        e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        if (e == cudaSuccess) e = cudaDeviceGetAttribute(&smem_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev);
        if (e == cudaSuccess) e = cudaDeviceGetAttribute(&reserved, cudaDevAttrReservedSharedMemoryPerBlock, dev);
        if (e == cudaSuccess) e = cudaFuncGetAttributes(&fa, gdn_chunk_prep<IO, false>);
        if (e != cudaSuccess) return e;
        const int per_cta = kPrepSmem + (int)fa.sharedSizeBytes + reserved;
        int per_sm = per_cta > 0 ? smem_sm / per_cta : 0;
        if (per_sm > 3) per_sm = 3;
        if (sms <= 0 || per_sm <= 0) return cudaErrorInvalidConfiguration;
        g_prep_slots[dev][std::is_same<IO, __nv_bfloat16>::value] = sms * per_sm;
        e = cudaFuncGetAttributes(&fa, gdn_chunk_prep_pk<IO>);
        if (e != cudaSuccess) return e;
        const int per_cta_pk = kPkSmem + (int)fa.sharedSizeBytes + reserved;
        int per_sm_pk = smem_sm / per_cta_pk;
        if (per_sm_pk > 2) per_sm_pk = 2;
        if (per_sm_pk <= 0) return cudaErrorInvalidConfiguration;
        g_prep_pk_slots[dev][std::is_same<IO, __nv_bfloat16>::value] = sms * per_sm_pk;
        configured[dev] = true;
    }
    return cudaSuccess;
}

template <typename IO>
cudaError_t launch_prep(const TcParams &tp, int64_t items, cudaStream_t stream) {
    if (items <= 0) return cudaSuccess;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    const int slots = (tp.per_key ? g_prep_pk_slots : g_prep_slots)[dev][std::is_same<IO, __nv_bfloat16>::value];
    if (slots <= 0) return cudaErrorInvalidConfiguration;
    TcParams pk = tp;
    pk.prep_items = items;
    if (tp.cx != nullptr) {   // the convolution prologue, with the default rule
        const int64_t ctas_cv = items <= 3 * (int64_t)slots ? items : slots;
        gdn_chunk_prep<IO, false, true><<<(unsigned)ctas_cv, kPrepThreads, kPrepSmem, stream>>>(pk);
        return cudaGetLastError();
    }
    if (tp.per_key) {
        const int64_t ctas_pk = items <= 2 * (int64_t)slots ? items : slots;
        gdn_chunk_prep_pk<IO><<<(unsigned)ctas_pk, kPrepThreads, kPkSmem, stream>>>(pk);
        return cudaGetLastError();
    }
    // Persistent CTAs pay off on long item lists; up to three items per resident CTA, one
    // CTA per item leaves a shorter tail.
    const int64_t ctas = items <= 3 * (int64_t)slots ? items : slots;
    if (tp.has_decay && tp.has_delta && !tp.beta_shared)
        gdn_chunk_prep<IO, false><<<(unsigned)ctas, kPrepThreads, kPrepSmem, stream>>>(pk);
    else
        gdn_chunk_prep<IO, true><<<(unsigned)ctas, kPrepThreads, kPrepSmem, stream>>>(pk);
    return cudaGetLastError();
}

// The scan's view of a call with one decay per key dimension: Q and K come from the prep's
// Q~ and K~ arrays, one head per value head.
TcParams scan_view(const TcParams &tp) {
    TcParams ts = tp;
    if (tp.per_key) {
        ts.tm_q = tp.tm_qt;
        ts.tm_k = tp.tm_kt;
        ts.h_qk = tp.h_v;
    }
    return ts;
}

template <typename IO>
cudaError_t launch_scan(const TcParams &tp, cudaStream_t stream) {
    const int64_t ctas = (int64_t)tp.num_seqs * tp.h_v * (kDK / kNV);
    if (ctas > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    if (tp.per_key) {   // never with the norm epilogue
        gdn_chunk_scan<IO, false, true><<<(unsigned)ctas, kScanAllThreads, kScanSmem, stream>>>(scan_view(tp));
        return cudaGetLastError();
    }
    if (tp.norm_gate != nullptr) {
        // The two column halves of a (sequence, head), CTAs 2i and 2i + 1, as a cluster.
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3((unsigned)ctas);
        cfg.blockDim = dim3(kScanAllThreads);
        cfg.dynamicSmemBytes = kScanSmemNorm;
        cfg.stream = stream;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = 2;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        return cudaLaunchKernelEx(&cfg, gdn_chunk_scan<IO, true>, tp);
    }
    gdn_chunk_scan<IO><<<(unsigned)ctas, kScanAllThreads, kScanSmem, stream>>>(tp);
    return cudaGetLastError();
}

// One call: the prep over every workspace slot, then the scan; or, split into `nseg`
// chunk segments, the prep of segment k + 1 on the side stream beside the scan of
// segment k.  Every launch stays ordered after the work already on `stream`, and the
// last scan after every side launch.
template <typename IO>
cudaError_t launch_typed(TcParams tp, int64_t n_slots, int nseg, cudaStream_t stream) {
    cudaError_t e = configure<IO>();
    if (e != cudaSuccess) return e;
    SideStream *side = nseg > 1 ? side_stream() : nullptr;
    if (side == nullptr) {
        tp.seg_begin = 0;
        tp.seg_end = 0x7fffffff;
        tp.seg_direct = 0;
        e = launch_prep<IO>(tp, n_slots * tp.h_v, stream);
        return e != cudaSuccess ? e : launch_scan<IO>(tp, stream);
    }
    const int cps = tp.chunks_per_seq;
    auto bound = [&](int k) { return (int)((int64_t)k * cps / nseg); };
    float *const state_out = tp.state_out;
    const float *const state_in = tp.state_in;
    tp.seg_direct = 1;
    std::lock_guard<std::mutex> lock(side->launch_mu);
    for (int k = 0; e == cudaSuccess && k < nseg; ++k) {
        TcParams pk = tp;
        if (k == 0) {
            // The side stream starts once the first prep is done, i.e. when the first
            // scan starts, so that later preps take the SMs the scan leaves free rather
            // than delaying the first prep.
            pk.seg_begin = bound(0);
            pk.seg_end = bound(1);
            e = launch_prep<IO>(pk, (int64_t)tp.num_seqs * (pk.seg_end - pk.seg_begin) * tp.h_v, stream);
            if (e == cudaSuccess) e = cudaEventRecord(side->ev[0], stream);
            if (e == cudaSuccess) e = cudaStreamWaitEvent(side->stream, side->ev[0], 0);
        }
        if (e == cudaSuccess && k + 1 < nseg) {
            pk.seg_begin = bound(k + 1);
            pk.seg_end = bound(k + 2);
            e = launch_prep<IO>(pk, (int64_t)tp.num_seqs * (pk.seg_end - pk.seg_begin) * tp.h_v, side->stream);
            if (e == cudaSuccess) e = cudaEventRecord(side->ev[k + 1], side->stream);
        }
        if (e == cudaSuccess && k > 0) e = cudaStreamWaitEvent(stream, side->ev[k], 0);
        if (e == cudaSuccess) {
            pk.seg_begin = bound(k);
            pk.seg_end = bound(k + 1);
            pk.state_in = k == 0 ? state_in : state_out;
            pk.state_out = state_out;
            e = launch_scan<IO>(pk, stream);
        }
    }
    return e;
}

// Chunk slots the prep kernel covers (an upper bound for packed sequences).
int64_t chunk_slots(bool varlen, int64_t seqlen, int64_t batch, int64_t num_seqs) {
    if (!varlen) return batch * ((seqlen + kC - 1) / kC);
    return seqlen / kC + num_seqs + 1;
}

constexpr int kMaxTpSegments = 4;
constexpr int kMinTpChunks = 16;
// Segments of the time-parallel scan for a batched shape (1: not used).  Every segment
// after the first costs two scan CTAs per (sequence, head, column half), and all of them
// must fit on the GPU at once.
int tp_segments(bool varlen, int64_t seqlen, int64_t batch, int h_v) {
    if (varlen) return 1;
    const int sms = sm_count();
    const int64_t units = batch * h_v * (kDK / kNV);
    const int64_t chunks = (seqlen + kC - 1) / kC;
    int best = 1;
    for (int s2 = 2; s2 <= kMaxTpSegments; ++s2)
        if (units * (2 * s2 - 1) <= sms && chunks >= (int64_t)s2 * kMinTpChunks) best = s2;
    return best;
}

// Bytes the time-parallel scan adds after the records: R, Phi and Psi, each 1 KiB aligned.
struct TpLayout {
    size_t r, phi, psi, total;
};
TpLayout tp_layout(int64_t seqlen, int64_t batch, int h_v, int nseg) {
    auto up = [](size_t x) { return (x + 1023) & ~(size_t)1023; };
    TpLayout L{};
    const size_t tok = (size_t)seqlen * batch;
    const size_t states = (size_t)nseg * batch * h_v * kDK * kDK;
    L.r = 0;
    L.phi = L.r + up(tok * h_v * kDK * 2);
    L.psi = L.phi + up(states * 4);
    L.total = L.psi + up(states * 4);
    return L;
}

// The time-parallel call: prep, the scan of every segment and operator pass at once, the
// combine (one launch per segment boundary), then o_t += R_t S_k for the tokens of every
// segment k >= 1.
template <typename IO>
cudaError_t launch_tp(TcParams tp, int64_t n_slots, int nseg, uint8_t *extra, cudaStream_t stream) {
    cudaError_t e = configure<IO>();
    if (e != cudaSuccess) return e;
    const TpLayout L = tp_layout(tp.seqlen, tp.num_seqs, tp.h_v, nseg);
    const int cps = tp.chunks_per_seq;
    tp.tp_nseg = nseg;
    tp.tp_seg = (cps + nseg - 1) / nseg;
    tp.tp_r = extra + L.r;
    tp.tp_phi = reinterpret_cast<float *>(extra + L.phi);
    tp.tp_psi = reinterpret_cast<float *>(extra + L.psi);
    tp.seg_begin = 0;
    tp.seg_end = 0x7fffffff;
    tp.seg_direct = 0;
    e = launch_prep<IO>(tp, n_slots * tp.h_v, stream);
    if (e != cudaSuccess) return e;
    const int64_t units = (int64_t)tp.num_seqs * tp.h_v * (kDK / kNV);
    if (tp.per_key)
        gdn_chunk_scan<IO, false, true><<<(unsigned)(units * (2 * nseg - 1)), kScanAllThreads, kScanSmem, stream>>>(
            scan_view(tp));
    else
        gdn_chunk_scan<IO><<<(unsigned)(units * (2 * nseg - 1)), kScanAllThreads, kScanSmem, stream>>>(tp);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    for (int k = 1; k < nseg; ++k) {
        gdn_tp_combine<IO><<<dim3((unsigned)(tp.num_seqs * tp.h_v), 16), 256, 0, stream>>>(tp, k);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
    const unsigned tiles = (unsigned)((tp.tp_seg + 1) / 2);
    gdn_tp_correct<IO><<<dim3((unsigned)(tp.num_seqs * tp.h_v), (unsigned)(nseg - 1) * tiles), kCorrThreads,
                         kCorrSmem, stream>>>(tp);
    return cudaGetLastError();
}

}  // namespace

long long g_wait_budget = 0;   // 0: the kernels' default budget

bool encode_map_3d(CUtensorMap *m, const void *base, gdn_dtype io, const uint64_t dims[3],
                   const uint64_t strides[2], const uint32_t box[3]) {
    auto fn = encode_fn();
    if (fn == nullptr || io == GDN_F32) return false;
    const cuuint64_t d[3] = {dims[0], dims[1], dims[2]};
    const cuuint64_t st[2] = {strides[0], strides[1]};
    const cuuint32_t bx[3] = {box[0], box[1], box[2]};
    const cuuint32_t estr[3] = {1, 1, 1};
    const CUresult r = fn(m, io == GDN_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16,
                          3, const_cast<void *>(base), d, st, bx, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                          CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

size_t prefill_tc_conv_v_bytes(int64_t total_tokens, int h_v) {
    return ((size_t)total_tokens * h_v * kDK * 2 + 1023) & ~(size_t)1023;
}

size_t prefill_tc_conv_bytes(int64_t total_tokens, int h_qk) {
    const size_t each = ((size_t)total_tokens * h_qk * kDK * 2 + 1023) & ~(size_t)1023;
    return 2 * each;
}

size_t prefill_tc_pk_bytes(int64_t total_tokens, int h_v) {
    const size_t each = ((size_t)total_tokens * h_v * kDK * 2 + 1023) & ~(size_t)1023;
    return 2 * each;
}

size_t prefill_tc_tp_bytes(bool varlen, int64_t seqlen, int64_t batch, int h_v) {
    const int nseg = tp_segments(varlen, seqlen, batch, h_v);
    return nseg > 1 ? tp_layout(seqlen, batch, h_v, nseg).total : 0;
}

int prefill_tc_tp_nseg(bool varlen, int64_t seqlen, int64_t batch, int h_v) {
    return tp_segments(varlen, seqlen, batch, h_v);
}

bool prefill_tc_shape_ok(gdn_dtype io, int d_k, int d_v, int64_t total_tokens) {
    return (io == GDN_BF16 || io == GDN_F16) && d_k == kDK && d_v == kDK && total_tokens > 0 &&
           total_tokens <= 0x7fffff00LL;
}

size_t prefill_tc_workspace(bool varlen, int64_t seqlen, int64_t batch, int64_t num_seqs, int h_v) {
    return (size_t)chunk_slots(varlen, seqlen, batch, num_seqs) * (size_t)h_v * kRecord;
}

int prefill_tc_segments(bool varlen, int64_t seqlen, int64_t batch, int h_v) {
    if (varlen) return 1;
    const int sms = sm_count();
    if (sms <= 0 || batch * h_v * (kDK / kNV) * 3 > sms) return 1;   // the scan alone fills the GPU
    const int64_t nseg = ((seqlen + kC - 1) / kC) / kMinSegmentChunks;
    return (int)(nseg < 1 ? 1 : (nseg > kMaxSegments ? kMaxSegments : nseg));
}

bool prefill_tc_supported(const ScanParams &p, gdn_dtype io, int64_t total_tokens) {
    if (!prefill_tc_shape_ok(io, p.d_k, p.d_v, total_tokens)) return false;
    const void *ptrs[] = {p.q, p.k, p.v, p.o};
    for (const void *ptr : ptrs)
        if (reinterpret_cast<uintptr_t>(ptr) % 16 != 0) return false;
    return encode_fn() != nullptr;
}

cudaError_t launch_prefill_tc(const ScanParams &p, gdn_dtype io, int64_t total_tokens, void *workspace,
                              size_t workspace_bytes, bool allow_overlap, cudaStream_t stream) {
    TcParams tp;
    memset(&tp, 0, sizeof(tp));
    if (!make_map(&tp.tm_q, p.q, io, p.h_qk, total_tokens) ||
        !make_map(&tp.tm_k, p.k, io, p.h_qk, total_tokens) ||
        !make_map(&tp.tm_v, p.v, io, p.h_v, total_tokens) ||
        !make_map(&tp.tm_o, p.o, io, p.h_v, total_tokens))
        return cudaErrorInvalidValue;
    tp.a = p.a; tp.b = p.b; tp.A_log = p.A_log; tp.dt_bias = p.dt_bias;
    tp.state_in = p.state_in; tp.state_out = p.state_out; tp.o = p.o;
    tp.cu_seqlens = p.cu_seqlens; tp.seqlen = p.seqlen; tp.num_seqs = p.num_seqs;
    tp.h_qk = p.h_qk; tp.h_v = p.h_v; tp.scale = p.scale; tp.status = p.status;
    tp.chunks_per_seq = (int32_t)((p.seqlen + kC - 1) / kC);
    tp.ws = static_cast<uint8_t *>(workspace);
    tp.wait_budget = __atomic_load_n(&g_wait_budget, __ATOMIC_RELAXED);
    tp.has_decay = p.rule == GDN_RULE_GATED_DELTA || p.rule == GDN_RULE_GATED;
    tp.has_delta = p.rule == GDN_RULE_GATED_DELTA || p.rule == GDN_RULE_DELTA;
    tp.beta_shared = p.beta_shared;
    tp.norm_scale = p.norm_scale;
    tp.norm_gate = p.norm_gate;
    tp.norm_eps = p.norm_eps;
    tp.norm_silu = p.norm_silu;
    const bool varlen = p.cu_seqlens != nullptr;
    const int64_t n_slots = chunk_slots(varlen, p.seqlen, p.num_seqs, p.num_seqs);
    // The time-parallel scan, when the shape suits it, the caller allows internal
    // resources and the workspace holds its buffers (not with the norm epilogue: the
    // correction adds to o after the scan).
    size_t records = prefill_tc_workspace(varlen, p.seqlen, p.num_seqs, p.num_seqs, p.h_v);
    if (tp.has_decay && p.decay_per_key) {
        // Q~ and K~ follow the records; the caller has checked that the workspace holds them.
        const size_t each = prefill_tc_pk_bytes(total_tokens, p.h_v) / 2;
        uint8_t *base = static_cast<uint8_t *>(workspace) + records;
        tp.per_key = 1;
        tp.qt = base;
        tp.kt = base + each;
        if (!make_map(&tp.tm_qt, tp.qt, io, p.h_v, total_tokens) ||
            !make_map(&tp.tm_kt, tp.kt, io, p.h_v, total_tokens) ||
            !make_map(&tp.tm_a, p.a, io, p.h_v, total_tokens))   // a: 16-byte aligned (checked)
            return cudaErrorInvalidValue;
        records += 2 * each;
    }
    bool conv_pass_first = false;
    if (p.conv_x != nullptr) {
        // The convolved q and k (and, for the streaming pass, v) follow the records; the
        // caller has checked the room.
        const size_t each = prefill_tc_conv_bytes(total_tokens, p.h_qk) / 2;
        uint8_t *base = static_cast<uint8_t *>(workspace) + records;
        tp.cx = p.conv_x;
        tp.conv_w = p.conv_w;
        tp.conv_b = p.conv_b;
        tp.conv_in = p.conv_in;
        tp.conv_out = p.conv_out;
        tp.conv_k = p.conv_k;
        tp.conv_silu = p.conv_silu;
        tp.conv_C = 2 * p.h_qk * kDK + p.h_v * kDK;
        tp.cq = base;
        tp.ck = base + each;
        if (!make_map(&tp.tm_q, tp.cq, io, p.h_qk, total_tokens) ||
            !make_map(&tp.tm_k, tp.ck, io, p.h_qk, total_tokens))
            return cudaErrorInvalidValue;
        records += 2 * each;
        if (!p.conv_fuse) {
            // The streaming pass writes v too; the plain prep then reads q, k and v by TMA.
            tp.cv = static_cast<uint8_t *>(workspace) + records;
            if (!make_map(&tp.tm_v, tp.cv, io, p.h_v, total_tokens)) return cudaErrorInvalidValue;
            records += prefill_tc_conv_v_bytes(total_tokens, p.h_v);
            conv_pass_first = true;
        }
    }
    if (conv_pass_first) {
        // x [tokens][C] as a 3-D map (the third extent 1), one stage box of 256 x 35.
        CUtensorMap tm_x;
        const uint64_t dims[3] = {(uint64_t)tp.conv_C, (uint64_t)total_tokens, 1};
        const uint64_t strides[2] = {(uint64_t)tp.conv_C * 2, (uint64_t)tp.conv_C * 2 * (uint64_t)total_tokens};
        const uint32_t box[3] = {(uint32_t)kPassWidth, (uint32_t)kPassRows, 1};
        if (!encode_map_3d(&tm_x, tp.cx, io, dims, strides, box)) return cudaErrorInvalidValue;
        const dim3 grid((unsigned)((tp.conv_C + kPassWidth - 1) / kPassWidth),
                        (unsigned)((total_tokens + kPassChunk - 1) / kPassChunk));
        auto kern = io == GDN_BF16 ? conv_pass<__nv_bfloat16> : conv_pass<__half>;
        cudaError_t ce = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kPassSmem);
        if (ce != cudaSuccess) return ce;
        kern<<<grid, 256, kPassSmem, stream>>>(tp, tm_x);
        ce = cudaGetLastError();
        if (ce != cudaSuccess) return ce;
    }
    // The launches' parameters, taken once every field is set (the time-parallel branch
    // adds the R map first): the prep's convolution form only when the convolution is
    // fused into it.
    auto launch_view = [&]() {
        TcParams t = tp;
        if (conv_pass_first) t.cx = nullptr;
        return t;
    };
    const int tps = allow_overlap && p.norm_gate == nullptr
                        ? tp_segments(varlen, p.seqlen, p.num_seqs, p.h_v) : 1;
    if (tps > 1 && workspace_bytes >= records + tp_layout(p.seqlen, p.num_seqs, p.h_v, tps).total) {
        uint8_t *extra = static_cast<uint8_t *>(workspace) + records;
        if (!make_map(&tp.tm_r, extra + tp_layout(p.seqlen, p.num_seqs, p.h_v, tps).r, io, p.h_v, total_tokens))
            return cudaErrorInvalidValue;
        cudaError_t e = io == GDN_BF16 ? launch_tp<__nv_bfloat16>(launch_view(), n_slots, tps, extra, stream)
                                       : launch_tp<__half>(launch_view(), n_slots, tps, extra, stream);
        return e;   // batched: no sequence is empty
    }
    const int nseg = allow_overlap ? prefill_tc_segments(varlen, p.seqlen, p.num_seqs, p.h_v) : 1;
    cudaError_t e = io == GDN_BF16 ? launch_typed<__nv_bfloat16>(launch_view(), n_slots, nseg, stream)
                                   : launch_typed<__half>(launch_view(), n_slots, nseg, stream);
    if (e == cudaSuccess && tp.cx != nullptr && varlen && p.conv_k > 1) {
        if (io == GDN_BF16) conv_state_empty<__nv_bfloat16><<<(unsigned)p.num_seqs, 256, 0, stream>>>(tp);
        else conv_state_empty<__half><<<(unsigned)p.num_seqs, 256, 0, stream>>>(tp);
        e = cudaGetLastError();
    }
    return e;
}

}  // namespace gdn
