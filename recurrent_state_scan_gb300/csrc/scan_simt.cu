// scan_simt.cu -- the token-sequential gated delta-rule scan on FP32 ALUs.
//
// Serves gdn_decode_step (one token, state updated in place: the decode hot path)
// and gdn_prefill for fp32 I/O and for shapes the tensor-core chunked path does not
// take.  It evaluates, per token, Steps 1-4 of `linear_attention_core`
// (onnx-runtime-ep-cuda 0.1.0-dev.6, src/kernels/linear_attention.rs): decay,
// retrieval r = S^T k, delta update S += k (x) beta (v - r), readout o = scale S^T q.
//
// Design (GB300-first, not the page's one-thread-per-column / one-warp-per-column):
//  - One CTA of 128 threads owns the full d_k rows of a tile of 4*LPR state columns
//    of one (sequence, value head).  The page's "Parallelization" note -- columns
//    evolve independently -- is what lets a CTA own a column tile.
//  - A row of LPR lanes covers the tile's columns with one float4 each, so each
//    warp reads/writes whole 256 B row segments of S[d_k][d_v]: fully coalesced
//    128-bit accesses.  Each thread keeps RPT rows x 4 columns of S in registers for the
//    whole scan (fp32), so S is read from HBM once and written once.
//  - Per token the d_k reductions for both Sk and Sq run in ONE pass over the
//    registers; the readout uses S'^T q = alpha S^T q + (q.k) delta, which is the
//    updated-state readout re-associated, so no second pass is needed.
//  - Cross-row partial sums go through shared memory (three barriers per token).
//  - The page's variants (its rule list and Step 1's per-key-dim decay) run through the
//    same kernel: a rule drops the decay and/or the delta; with one decay factor a_i per
//    key dimension, row i of S is scaled by a_i, which folds into the reductions as the
//    weights a_i k_i and a_i q_i (compile-time, so the per-head path is unchanged).
#include "gdn_internal.cuh"

namespace gdn {
namespace {

// Up to d_k = 128 four 128-thread CTAs must fit on an SM (at most 128 registers a
// thread): the state tiles of four CTAs in flight are what keeps HBM busy.
template <int DKMAX, int kThreads>
constexpr int simt_min_blocks() { return DKMAX <= 128 ? 512 / kThreads : 1; }

template <typename IO, int DKMAX, int LPR, int kThreads, bool kPerKey>
__global__ void __launch_bounds__(kThreads, (simt_min_blocks<DKMAX, kThreads>()))
    scan_simt_kernel(const ScanParams p) {
    constexpr int RPP = kThreads / LPR;   // rows covered per pass
    constexpr int RPT = DKMAX / RPP;      // rows held per thread
    constexpr int TILE = 4 * LPR;         // state columns per CTA
    static_assert(RPT >= 1 && DKMAX % RPP == 0, "bad tiling");
    constexpr int kBetaThread = kThreads > 32 ? 32 : 0;

    __shared__ float sq[DKMAX], sk[DKMAX];
    __shared__ float sa[kPerKey ? DKMAX : 1];   // per-key decay factors of this token
    __shared__ float sv[TILE], sdelta[TILE];
    __shared__ __align__(16) float red_k[RPP * TILE];
    __shared__ __align__(16) float red_q[RPP * TILE];
    __shared__ float s_alpha, s_beta, s_qk;

    const int tid = threadIdx.x;
    const int lr = tid % LPR, rg = tid / LPR;
    const int tiles = (p.d_v + TILE - 1) / TILE;
    int64_t unit = blockIdx.x;
    const int tile = (int)(unit % tiles);
    unit /= tiles;
    const int h = (int)(unit % p.h_v);
    const int64_t n = unit / p.h_v;
    const int hq = h / (p.h_v / p.h_qk);
    const int col0 = tile * TILE + 4 * lr;
    const bool col_ok = col0 < p.d_v;   // d_v is a multiple of 4

    int64_t t0, t1;
    if (!seq_range(p, n, t0, t1)) return;
    // A state pool: sequence n reads and writes entry slots[n]; a slot outside the pool
    // skips the sequence and sets the check word.
    int64_t ns = n;
    if (p.slots != nullptr) {
        ns = p.slots[n];
        if (ns < 0 || ns >= p.pool_size) {
            if (tid == 0) atomicOr(p.status, kDevBadSlot);
            return;
        }
    }

    const size_t sbase = ((size_t)ns * p.h_v + h) * (size_t)p.d_k * p.d_v;
    float4 S[RPT];
#pragma unroll
    for (int m = 0; m < RPT; ++m) {
        const int i = rg + RPP * m;
        S[m] = make_float4(0.f, 0.f, 0.f, 0.f);
        if (p.state_in != nullptr && col_ok && i < p.d_k)
            S[m] = __ldcs(reinterpret_cast<const float4 *>(p.state_in + sbase +
                                                          (size_t)i * p.d_v + col0));
    }

    // This thread's rows and columns of slab w of the state window.
    auto store_slab = [&](int64_t w, const float4 (&X)[RPT]) {
        float *base = p.window + (((size_t)w * p.num_seqs + n) * p.h_v + h) * (size_t)p.d_k * p.d_v;
#pragma unroll
        for (int m = 0; m < RPT; ++m) {
            const int i = rg + RPP * m;
            if (col_ok && i < p.d_k) __stcs(reinterpret_cast<float4 *>(base + (size_t)i * p.d_v + col0), X[m]);
        }
    };

    const IO *q = static_cast<const IO *>(p.q);
    const IO *k = static_cast<const IO *>(p.k);
    const IO *v = static_cast<const IO *>(p.v);
    const IO *ga = static_cast<const IO *>(p.a);
    const IO *gb = static_cast<const IO *>(p.b);
    IO *o = static_cast<IO *>(p.o);
    const bool has_decay = (p.rule == GDN_RULE_GATED_DELTA || p.rule == GDN_RULE_GATED);
    const bool has_delta = (p.rule == GDN_RULE_GATED_DELTA || p.rule == GDN_RULE_DELTA);

    // The inputs of token t + 1 are loaded into registers while token t is computed, so a
    // token's loads are not on the chain: this thread's q and k entries (and per-key decay
    // logits), its v column, and the scalar gate logits.
    constexpr int QPT = (DKMAX + kThreads - 1) / kThreads;   // q / k entries a thread loads
    float nq[QPT], nk[QPT], na[kPerKey ? QPT : 1], nv = 0.f, ng_a = 0.f, ng_b = 0.f;
    float pA[kPerKey ? QPT : 1], pD[kPerKey ? QPT : 1];     // this thread's per-key A_log, dt_bias
#pragma unroll
    for (int u = 0; u < QPT; ++u) {
        nq[u] = nk[u] = 0.f;
        if (kPerKey) na[u] = pA[u] = pD[u] = 0.f;
    }
    if (kPerKey) {
        const size_t hk = (size_t)h * p.d_k;
#pragma unroll
        for (int u = 0; u < QPT; ++u) {
            const int i = tid + u * kThreads;
            if (i < p.d_k) {
                pA[u] = p.A_log[hk + i];
                pD[u] = p.dt_bias[hk + i];
            }
        }
    }
    auto load_token = [&](int64_t t) {
        const size_t qk_off = ((size_t)t * p.h_qk + hq) * p.d_k;
#pragma unroll
        for (int u = 0; u < QPT; ++u) {
            const int i = tid + u * kThreads;
            nq[u] = i < p.d_k ? IoType<IO>::ld(q + qk_off + i) : 0.f;
            nk[u] = i < p.d_k ? IoType<IO>::ld(k + qk_off + i) : 0.f;
            if (kPerKey)
                na[u] = (has_decay && i < p.d_k) ? IoType<IO>::ld(ga + ((size_t)t * p.h_v + h) * p.d_k + i) : 0.f;
        }
        if (tid < TILE) {
            const int c = tile * TILE + tid;
            nv = c < p.d_v ? IoType<IO>::ld(v + ((size_t)t * p.h_v + h) * p.d_v + c) : 0.f;
        }
        const size_t gi = (size_t)t * p.h_v + h;
        if (tid == 0 && has_decay && !kPerKey) ng_a = IoType<IO>::ld(ga + gi);
        if (tid == kBetaThread && has_delta) ng_b = IoType<IO>::ld(gb + (p.beta_shared ? (size_t)t : gi));
    };
    if (t0 < t1) load_token(t0);

    for (int64_t t = t0; t < t1; ++t) {
        __syncthreads();   // previous token's shared values are no longer read
        const size_t v_off = ((size_t)t * p.h_v + h) * p.d_v;
#pragma unroll
        for (int u = 0; u < QPT; ++u) {
            const int i = tid + u * kThreads;
            if (i < DKMAX) {
                sq[i] = nq[u];
                sk[i] = nk[u];
                if (kPerKey)
                    sa[i] = (has_decay && i < p.d_k) ? expf(decay_f(na[u], pA[u], pD[u])) : 1.f;
            }
        }
        if (tid < TILE) sv[tid] = nv;
        // The two scalar gates come from two different warps.
        if (tid == 0) s_alpha = (has_decay && !kPerKey) ? expf(decay_f(ng_a, p.A_log[h], p.dt_bias[h])) : 1.f;
        if (tid == kBetaThread) s_beta = has_delta ? sigmoid_f(ng_b) : 1.f;
        if (t + 1 < t1) load_token(t + 1);
        __syncthreads();

        // Partial retrieval S^T k and readout S^T q over this thread's rows.
        float4 pk = make_float4(0.f, 0.f, 0.f, 0.f), pq = pk;
#pragma unroll
        for (int m = 0; m < RPT; ++m) {
            const int i = rg + RPP * m;
            const float ai = kPerKey ? sa[i] : 1.f;
            const float kk = ai * sk[i], qq = ai * sq[i];
            pk.x = fmaf(S[m].x, kk, pk.x); pk.y = fmaf(S[m].y, kk, pk.y);
            pk.z = fmaf(S[m].z, kk, pk.z); pk.w = fmaf(S[m].w, kk, pk.w);
            pq.x = fmaf(S[m].x, qq, pq.x); pq.y = fmaf(S[m].y, qq, pq.y);
            pq.z = fmaf(S[m].z, qq, pq.z); pq.w = fmaf(S[m].w, qq, pq.w);
        }
        *reinterpret_cast<float4 *>(&red_k[rg * TILE + 4 * lr]) = pk;
        *reinterpret_cast<float4 *>(&red_q[rg * TILE + 4 * lr]) = pq;
        if (tid < 32) {
            float acc = 0.f;
            for (int i = tid; i < DKMAX; i += 32) acc = fmaf(sq[i], sk[i], acc);
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
            if (tid == 0) s_qk = acc;
        }
        __syncthreads();

        const float alpha = s_alpha;
        if (tid < TILE) {
            float rk = 0.f, rq = 0.f;
#pragma unroll 8
            for (int r = 0; r < RPP; ++r) {
                rk += red_k[r * TILE + tid];
                rq += red_q[r * TILE + tid];
            }
            // r = (alpha S)^T k; delta = beta (v - r) (or v without the delta rule);
            // o = scale (alpha S + k delta^T)^T q
            const float delta = has_delta ? s_beta * (sv[tid] - alpha * rk) : sv[tid];
            sdelta[tid] = delta;
            const int c = tile * TILE + tid;
            if (c < p.d_v) IoType<IO>::st(o + v_off + c, p.scale * fmaf(s_qk, delta, alpha * rq));
        }
        __syncthreads();

        const float4 d4 = *reinterpret_cast<const float4 *>(&sdelta[4 * lr]);
#pragma unroll
        for (int m = 0; m < RPT; ++m) {
            const float kk = sk[rg + RPP * m];
            const float am = kPerKey ? sa[rg + RPP * m] : alpha;
            S[m].x = fmaf(am, S[m].x, kk * d4.x);
            S[m].y = fmaf(am, S[m].y, kk * d4.y);
            S[m].z = fmaf(am, S[m].z, kk * d4.z);
            S[m].w = fmaf(am, S[m].w, kk * d4.w);
        }
        // One of the last window_len steps: its state goes to slab window_len - (t1 - t).
        if (p.window != nullptr && t1 - t <= p.window_len)
            store_slab(p.window_len - (t1 - t), S);
    }
    // Fewer steps than slabs: the leading slabs are zero.
    if (p.window != nullptr) {
        float4 Z[RPT];
#pragma unroll
        for (int m = 0; m < RPT; ++m) Z[m] = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int64_t w = 0; w < (int64_t)p.window_len - (t1 - t0); ++w) store_slab(w, Z);
    }

    if (p.state_out == nullptr) return;
#pragma unroll
    for (int m = 0; m < RPT; ++m) {
        const int i = rg + RPP * m;
        if (col_ok && i < p.d_k)
            __stcs(reinterpret_cast<float4 *>(p.state_out + sbase + (size_t)i * p.d_v + col0),
                   S[m]);
    }
}

// ------------------------------------------------------------------ streaming decode step
// The decode step (one token per sequence, d_k = 128, d_v a multiple of 64, any rule and
// gate layout, optionally against a state pool) with persistent CTAs: each CTA walks
// (sequence, head, 64-column tile) units in a grid-stride loop and prefetches the next
// unit's inputs while it computes the current one.  The tiling and the math per unit are
// those of scan_simt_kernel (128 threads, 16 rows x 4 columns a thread), so one unit is
// one token of that kernel.
//  - The next unit's state tile streams into shared memory with 16-byte cp.async copies,
//    each thread copying exactly the elements it will hold, so it needs no barrier of its
//    own: the thread waits for its copies (cp.async.wait_group) and moves them to
//    registers.  The copies are issued only after this unit's reductions have read every
//    state register, so the copy-in never overtakes a pending read of the same slot.
//  - q, k, the 64 values of v and, with per-key decay, the d_k decay logits for the next
//    unit come the same way into a staging tile that the unit's barriers protect; its
//    scalar gate inputs (and per-key parameters) are prefetched into the registers of the
//    threads that evaluate them.
__device__ __forceinline__ void stream_cp16(void *smem, const void *gmem) {
    const unsigned a = static_cast<unsigned>(__cvta_generic_to_shared(smem));
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(a), "l"(gmem) : "memory");
}
__device__ __forceinline__ void stream_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
__device__ __forceinline__ void stream_wait_all() { asm volatile("cp.async.wait_group 0;\n" ::: "memory"); }

template <typename IO, bool kPerKey>
__global__ void __launch_bounds__(128, 4) decode_stream_kernel(const ScanParams p) {
    constexpr int kThreads = 128, LPR = 16, RPP = kThreads / LPR, RPT = 128 / RPP, TILE = 64;
    constexpr int ES = (int)sizeof(IO);
    constexpr int QB = 128 * ES, VB = TILE * ES;            // staged bytes of q (= k, a) and v
    constexpr int SB = 2 * QB + VB + (kPerKey ? QB : 0);    // next q | k | v [| a] tile
    constexpr int kBetaThread = 32;
    __shared__ __align__(16) float4 pre[RPT][kThreads];      // the next unit's state slots
    __shared__ __align__(16) unsigned char stage[SB];
    __shared__ float sq[128], sk[128], sv[TILE], sdelta[TILE];
    __shared__ float sa[kPerKey ? 128 : 1];                  // per-key decay factors
    __shared__ __align__(16) float red_k[RPP * TILE];
    __shared__ __align__(16) float red_q[RPP * TILE];
    __shared__ float s_alpha, s_beta, s_qk;

    const int tid = threadIdx.x;
    const int lr = tid % LPR, rg = tid / LPR;
    const int tiles = p.d_v / TILE;
    const int64_t units = (int64_t)p.num_seqs * p.h_v * tiles;
    const IO *q = static_cast<const IO *>(p.q);
    const IO *k = static_cast<const IO *>(p.k);
    const IO *v = static_cast<const IO *>(p.v);
    const IO *ga = static_cast<const IO *>(p.a);
    const IO *gb = static_cast<const IO *>(p.b);
    IO *o = static_cast<IO *>(p.o);
    const bool has_decay = (p.rule == GDN_RULE_GATED_DELTA || p.rule == GDN_RULE_GATED);
    const bool has_delta = (p.rule == GDN_RULE_GATED_DELTA || p.rule == GDN_RULE_DELTA);

    struct Unit {
        int64_t n, srow;
        int h, hq, tile;
        bool ok;
    };
    auto unit_of = [&](int64_t u) {
        Unit x;
        x.tile = (int)(u % tiles);
        const int64_t r = u / tiles;
        x.h = (int)(r % p.h_v);
        x.n = r / p.h_v;
        x.hq = x.h / (p.h_v / p.h_qk);
        x.srow = x.n;
        x.ok = true;
        if (p.slots != nullptr) {
            x.srow = p.slots[x.n];
            x.ok = x.srow >= 0 && x.srow < p.pool_size;
        }
        return x;
    };
    float ra = 0.f, rb = 0.f, rA = 0.f, rD = 0.f;   // the next unit's gate inputs
    // Issue the copies of unit u (its state slots, q, k, v) and its gate loads.
    auto prefetch = [&](const Unit &x) {
        const int col0 = x.tile * TILE + 4 * lr;
        const size_t sbase = ((size_t)x.srow * p.h_v + x.h) * (size_t)128 * p.d_v;
#pragma unroll
        for (int m = 0; m < RPT; ++m) {
            if (x.ok && p.state_in != nullptr)
                stream_cp16(&pre[m][tid], p.state_in + sbase + (size_t)(rg + RPP * m) * p.d_v + col0);
            else
                pre[m][tid] = make_float4(0.f, 0.f, 0.f, 0.f);
        }
        const size_t qk_off = ((size_t)x.n * p.h_qk + x.hq) * 128;
        const size_t v_off = ((size_t)x.n * p.h_v + x.h) * p.d_v + (size_t)x.tile * TILE;
        const size_t gi = (size_t)x.n * p.h_v + x.h;
        for (int c = tid; c < SB / 16; c += kThreads) {
            const int byte = 16 * c;
            const unsigned char *src;
            if (byte < QB) src = reinterpret_cast<const unsigned char *>(q + qk_off) + byte;
            else if (byte < 2 * QB) src = reinterpret_cast<const unsigned char *>(k + qk_off) + (byte - QB);
            else if (byte < 2 * QB + VB) src = reinterpret_cast<const unsigned char *>(v + v_off) + (byte - 2 * QB);
            else if (has_decay) src = reinterpret_cast<const unsigned char *>(ga + gi * 128) + (byte - 2 * QB - VB);
            else continue;   // no decay: a is not read (and may be NULL)
            stream_cp16(stage + byte, src);
        }
        stream_commit();
        if (kPerKey) {
            // This thread's key dimension: its decay parameters.
            if (has_decay) {
                rA = p.A_log[(size_t)x.h * 128 + tid];
                rD = p.dt_bias[(size_t)x.h * 128 + tid];
            }
        } else if (tid == 0 && has_decay) {
            ra = IoType<IO>::ld(ga + gi);
            rA = p.A_log[x.h];
            rD = p.dt_bias[x.h];
        }
        if (tid == kBetaThread && has_delta) rb = IoType<IO>::ld(gb + (p.beta_shared ? (size_t)x.n : gi));
    };

    int64_t u = blockIdx.x;
    if (u >= units) return;
    Unit cur = unit_of(u);
    prefetch(cur);
    for (; u < units; u += gridDim.x) {
        stream_wait_all();          // this thread's copies of the unit have landed
        __syncthreads();            // everyone's copies (q, k, v) have landed
        float4 S[RPT];
#pragma unroll
        for (int m = 0; m < RPT; ++m) S[m] = pre[m][tid];
        sq[tid] = IoType<IO>::ld(reinterpret_cast<const IO *>(stage) + tid);
        sk[tid] = IoType<IO>::ld(reinterpret_cast<const IO *>(stage + QB) + tid);
        if (tid < TILE) sv[tid] = IoType<IO>::ld(reinterpret_cast<const IO *>(stage + 2 * QB) + tid);
        if (kPerKey)
            sa[tid] = has_decay ? expf(decay_f(IoType<IO>::ld(reinterpret_cast<const IO *>(stage + 2 * QB + VB) + tid),
                                               rA, rD))
                                : 1.f;
        if (tid == 0) s_alpha = (has_decay && !kPerKey) ? expf(decay_f(ra, rA, rD)) : 1.f;
        if (tid == kBetaThread) s_beta = has_delta ? sigmoid_f(rb) : 1.f;
        __syncthreads();

        // Partial retrieval S^T k and readout S^T q over this thread's rows.
        float4 pk = make_float4(0.f, 0.f, 0.f, 0.f), pq = pk;
#pragma unroll
        for (int m = 0; m < RPT; ++m) {
            const int i = rg + RPP * m;
            const float ai = kPerKey ? sa[i] : 1.f;
            const float kk = ai * sk[i], qq = ai * sq[i];
            pk.x = fmaf(S[m].x, kk, pk.x); pk.y = fmaf(S[m].y, kk, pk.y);
            pk.z = fmaf(S[m].z, kk, pk.z); pk.w = fmaf(S[m].w, kk, pk.w);
            pq.x = fmaf(S[m].x, qq, pq.x); pq.y = fmaf(S[m].y, qq, pq.y);
            pq.z = fmaf(S[m].z, qq, pq.z); pq.w = fmaf(S[m].w, qq, pq.w);
        }
        *reinterpret_cast<float4 *>(&red_k[rg * TILE + 4 * lr]) = pk;
        *reinterpret_cast<float4 *>(&red_q[rg * TILE + 4 * lr]) = pq;
        if (tid < 32) {
            float acc = 0.f;
            for (int i = tid; i < 128; i += 32) acc = fmaf(sq[i], sk[i], acc);
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
            if (tid == 0) s_qk = acc;
        }
        __syncthreads();            // every thread has read the staging tile and its state

        // The next unit streams in while this one finishes.
        const Unit x = cur;
        const int64_t un = u + gridDim.x;
        if (un < units) {
            cur = unit_of(un);
            prefetch(cur);
        }

        const float alpha = s_alpha;
        if (tid < TILE) {
            float rk = 0.f, rq = 0.f;
#pragma unroll 8
            for (int r = 0; r < RPP; ++r) {
                rk += red_k[r * TILE + tid];
                rq += red_q[r * TILE + tid];
            }
            // r = (alpha S)^T k; delta = beta (v - r) (or v without the delta rule);
            // o = scale (alpha S + k delta^T)^T q
            const float delta = has_delta ? s_beta * (sv[tid] - alpha * rk) : sv[tid];
            sdelta[tid] = delta;
            if (x.ok)
                IoType<IO>::st(o + ((size_t)x.n * p.h_v + x.h) * p.d_v + x.tile * TILE + tid,
                               p.scale * fmaf(s_qk, delta, alpha * rq));
        }
        __syncthreads();

        const float4 d4 = *reinterpret_cast<const float4 *>(&sdelta[4 * lr]);
        const int col0 = x.tile * TILE + 4 * lr;
        const size_t sbase = ((size_t)x.srow * p.h_v + x.h) * (size_t)128 * p.d_v;
#pragma unroll
        for (int m = 0; m < RPT; ++m) {
            const float kk = sk[rg + RPP * m];
            const float am = kPerKey ? sa[rg + RPP * m] : alpha;
            S[m].x = fmaf(am, S[m].x, kk * d4.x);
            S[m].y = fmaf(am, S[m].y, kk * d4.y);
            S[m].z = fmaf(am, S[m].z, kk * d4.z);
            S[m].w = fmaf(am, S[m].w, kk * d4.w);
            if (x.ok)
                __stcs(reinterpret_cast<float4 *>(p.state_out + sbase + (size_t)(rg + RPP * m) * p.d_v + col0),
                       S[m]);
        }
        if (!x.ok && tid == 0 && x.tile == 0) atomicOr(p.status, kDevBadSlot);
    }
}

template <typename IO, int DKMAX, int LPR, int NT>
cudaError_t launch_cfg(const ScanParams &p, cudaStream_t stream) {
    const int tiles = (p.d_v + 4 * LPR - 1) / (4 * LPR);
    const int64_t blocks = (int64_t)p.num_seqs * p.h_v * tiles;
    if (blocks <= 0) return cudaSuccess;
    if (blocks > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    if (p.decay_per_key)
        scan_simt_kernel<IO, DKMAX, LPR, NT, true><<<(unsigned)blocks, NT, 0, stream>>>(p);
    else
        scan_simt_kernel<IO, DKMAX, LPR, NT, false><<<(unsigned)blocks, NT, 0, stream>>>(p);
    return cudaGetLastError();
}

// 128-thread CTAs over 64-column tiles (32 for narrow states): at d_k = d_v = 128 a
// thread holds 64 state values (64 registers), four CTAs share an SM, and their
// load / reduce / store phases interleave.  Measured on GB300 for the B=256, H=32
// decode step, this tiling moves the 1.07 GB step at 6.1 TB/s, against 5.2 TB/s for
// 256-thread CTAs over 128 columns.
template <typename IO, int DKMAX>
cudaError_t launch_dk(const ScanParams &p, cudaStream_t stream) {
    if (p.d_v <= 32) return launch_cfg<IO, DKMAX, 8, 128>(p, stream);
    return launch_cfg<IO, DKMAX, 16, 128>(p, stream);
}

// The decode step the streaming kernel covers: one token per sequence, d_k = 128, d_v a
// multiple of 64, no window, a final state, 16-byte aligned q, k, v, state (and a, with
// per-key decay).
bool stream_decode_ok(const ScanParams &p) {
    auto a16 = [](const void *x) { return (reinterpret_cast<uintptr_t>(x) & 15) == 0; };
    const bool decay = p.rule == GDN_RULE_GATED_DELTA || p.rule == GDN_RULE_GATED;
    return p.cu_seqlens == nullptr && p.seqlen == 1 && p.d_k == 128 && p.d_v % 64 == 0 &&
           p.window == nullptr && p.state_out != nullptr && a16(p.q) && a16(p.k) && a16(p.v) &&
           a16(p.state_in) && a16(p.state_out) && (!p.decay_per_key || !decay || a16(p.a));
}

int stream_ctas() {
    static int cache[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 152 * 4;
    if (cache[dev] == 0) {
        int sms = 0;
        if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0)
            sms = 152;
        cache[dev] = 4 * sms;   // four resident CTAs per SM (39 KB of shared memory each)
    }
    return cache[dev];
}

template <typename IO>
cudaError_t launch_io(const ScanParams &p, cudaStream_t stream) {
    if (stream_decode_ok(p)) {
        const int64_t units = (int64_t)p.num_seqs * p.h_v * (p.d_v / 64);
        if (units <= 0) return cudaSuccess;
        const int64_t ctas = stream_ctas();
        const unsigned grid = (unsigned)(units < ctas ? units : ctas);
        if (p.decay_per_key)
            decode_stream_kernel<IO, true><<<grid, 128, 0, stream>>>(p);
        else
            decode_stream_kernel<IO, false><<<grid, 128, 0, stream>>>(p);
        return cudaGetLastError();
    }
    if (p.d_k <= 32) return launch_dk<IO, 32>(p, stream);
    if (p.d_k <= 64) return launch_dk<IO, 64>(p, stream);
    if (p.d_k <= 128) return launch_dk<IO, 128>(p, stream);
    return launch_dk<IO, 256>(p, stream);
}

}  // namespace

cudaError_t launch_scan_simt(const ScanParams &p, gdn_dtype io, cudaStream_t stream) {
    switch (io) {
        case GDN_F32: return launch_io<float>(p, stream);
        case GDN_BF16: return launch_io<__nv_bfloat16>(p, stream);
        default: return launch_io<__half>(p, stream);
    }
}

}  // namespace gdn
