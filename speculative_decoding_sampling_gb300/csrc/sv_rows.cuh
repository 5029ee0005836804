// sv_rows.cuh -- the row pass of the verification step.
//
// Every one of the B*(K+1) target rows is streamed once from HBM.  A row is
// cut into S1 row items of about SV_ROW_ITEM ids; persistent CTAs take them
// round-robin and stream them with 16-byte loads, the next step (possibly of
// the next item) in flight while the current one is folded.  Each thread
// keeps an online (max, normaliser) pair of softmax(z / T) in the base-2 form
// sum_i exp2(z_i * c - fl(M * c)), c = log2(e) / T (one exp2 per element).
// The CTA that finishes a row last merges the item partials and runs the
// accept test of the draft that row
// verifies: a = min(1, p(x) / q(x)), accept iff u < a
// ("推测解码：草稿、验证与实际加速", section 接受与拒绝怎样保住分布, equation for
// a(x); the replay in section 算完三个 token 的全部概率 accepts when the draw
// is strictly below the threshold).  The one that finishes a sequence's last
// row finds the first rejection j* and writes the accepted prefix; later
// drafts are void (same page, section 候选已知，验证才能并行).  Completion is
// detected with arrival counters; each is returned to zero by the CTA that
// saw it complete.
#pragma once

#include "sv_device.cuh"

namespace sv {

// max of two packed bf16 pairs (a NaN operand yields the other operand)
__device__ __forceinline__ uint32_t max_bf16x2(uint32_t a, uint32_t b)
{
    uint32_t r;
    asm("max.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
    return r;
}

__device__ __forceinline__ void warp_merge_ms(float &M, float &S, float c)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const float M2 = __shfl_xor_sync(0xFFFFFFFFu, M, o);
        const float S2 = __shfl_xor_sync(0xFFFFFFFFu, S, o);
        merge_ms(M, S, M2, S2, c);
    }
}

// Largest element of U 16-byte vectors.
template <typename LT, int U>
__device__ __forceinline__ float vec_max(const uint4 (&w)[U])
{
    if constexpr (sizeof(LT) == 2) {
        uint32_t m = max_bf16x2(max_bf16x2(w[0].x, w[0].y), max_bf16x2(w[0].z, w[0].w));
#pragma unroll
        for (int k = 1; k < U; ++k)
            m = max_bf16x2(m, max_bf16x2(max_bf16x2(w[k].x, w[k].y), max_bf16x2(w[k].z, w[k].w)));
        return fmaxf(bf16_lo(m), bf16_hi(m));
    } else {
        float m = fmaxf(fmaxf(__uint_as_float(w[0].x), __uint_as_float(w[0].y)),
                        fmaxf(__uint_as_float(w[0].z), __uint_as_float(w[0].w)));
#pragma unroll
        for (int k = 1; k < U; ++k)
            m = fmaxf(m, fmaxf(fmaxf(__uint_as_float(w[k].x), __uint_as_float(w[k].y)),
                               fmaxf(__uint_as_float(w[k].z), __uint_as_float(w[k].w))));
        return m;
    }
}

// Fold U vectors into the running (M, S) of one lane; S holds four packed
// pairs of partial sums (eight accumulators).
template <typename LT, int U>
__device__ __forceinline__ void fold(const uint4 (&w)[U], float &M, unsigned long long (&S)[4], float c)
{
    const float gm = vec_max<LT, U>(w);
    if (gm > M) {
        // rescale what was summed against the old maximum
        const float f = (M == -INFINITY) ? 0.0f : ex2(mc_of(M, c) - mc_of(gm, c));
        const unsigned long long f2 = pack2(f, f);
#pragma unroll
        for (int a = 0; a < 4; ++a)
            S[a] = mul2(S[a], f2);
        M = gm;
    }
    const float mc = mc_of(M, c);
    const unsigned long long c2 = pack2(c, c), nmc2 = pack2(-mc, -mc);
#pragma unroll
    for (int k = 0; k < U; ++k) {
        const uint32_t v[4] = {w[k].x, w[k].y, w[k].z, w[k].w};
        if constexpr (sizeof(LT) == 2) {
#pragma unroll
            for (int h = 0; h < 4; ++h) {
                float y0, y1;
                unpack2(fma2(pack2(bf16_lo(v[h]), bf16_hi(v[h])), c2, nmc2), y0, y1);
                S[h] = add2(S[h], pack2(ex2(y0), ex2(y1)));
            }
        } else {
#pragma unroll
            for (int h = 0; h < 4; h += 2) {
                float y0, y1;
                unpack2(fma2(pack2(__uint_as_float(v[h]), __uint_as_float(v[h + 1])), c2, nmc2), y0, y1);
                S[h + (k & 1)] = add2(S[h + (k & 1)], pack2(ex2(y0), ex2(y1)));
            }
        }
    }
}

// Per sequence: first rejection, accepted prefix, flags, and the surviving
// row's statistics published for the final draw.  One warp.
template <bool DENSE>
__device__ void finish_sequence(const Params &P, int64_t b, int lane)
{
    const int32_t K = P.K;
    __threadfence();
    const int32_t bad = __ldcg(&P.seq_bad[b]);
    int32_t jstar = K;
    for (int32_t k0 = 0; k0 < K; k0 += 32) {
        const int32_t k = k0 + lane;
        const bool rej = (k < K) && ld_cg_u8(&P.acc[b * K + k]) == 0;
        const unsigned m = __ballot_sync(0xFFFFFFFFu, rej);
        if (m) {
            jstar = k0 + __ffs(m) - 1;
            break;
        }
    }
    const int64_t rsel = b * (K + 1) + (jstar < K ? jstar : K);
    const float m_sel = __ldcg(&P.row_m[rsel]);
    const float s_sel = __ldcg(&P.row_s[rsel]);
    __syncwarp();
    for (int32_t j = lane; j <= K; j += 32) {
        P.row_m[b * (K + 1) + j] = 0.0f;
        P.row_s[b * (K + 1) + j] = 0.0f;
    }
    for (int32_t k = lane; k < K; k += 32)
        P.acc[b * K + k] = 0;
    int32_t *out = P.out_tokens + b * (K + 1);
    if (bad) {
        for (int32_t k = lane; k <= K; k += 32)
            out[k] = -1;
        for (int32_t k = lane; k < K; k += 32) {
            if (P.accept_flags) P.accept_flags[b * K + k] = -1;
            if (P.accept_prob) P.accept_prob[b * K + k] = 0.0f;
        }
    } else {
        for (int32_t k = lane; k <= K; k += 32)
            out[k] = k < jstar ? P.tokens[b * K + k] : -1;
        if (P.accept_flags)
            for (int32_t k = lane; k < K; k += 32)
                P.accept_flags[b * K + k] = k < jstar ? 1 : (k == jstar ? 0 : -1);
    }
    if (lane == 0) {
        if (bad) {
            P.num_emitted[b] = 0;
            if (P.residual_mass) P.residual_mass[b] = 0.0f;
            if (P.status) atomicOr(P.status, bad);
        } else {
            P.num_emitted[b] = jstar + 1;
        }
        P.seq_jstar[b] = bad ? -1 : jstar;
        P.seq_m[b] = m_sel;
        P.seq_s[b] = s_sel;
        P.seq_cnt[b] = 0u;
        P.seq_bad[b] = 0;
    }
}

// What the last warp of a row needs besides the item partials, fetched at
// the start of every row item so that its latency hides behind the stream.
struct RowSide {
    int32_t x;  // draft token verified by this row (j < K)
    float zx;   // its logit
    float qx;   // its draft probability (1 for one-hot drafts)
    float u;    // the row's uniform
};

template <typename LT, bool DENSE>
__device__ __forceinline__ RowSide fetch_side(const Params &P, int64_t r)
{
    RowSide s;
    const int32_t K = P.K, V = P.V;
    const int64_t b = divi(r, K + 1);
    const int32_t j = static_cast<int32_t>(r - b * (K + 1));
    s.u = __ldg(&P.u[b * (K + 1) + j]);
    s.x = -1;
    s.zx = 0.0f;
    s.qx = 1.0f;
    if (j < K) {
        s.x = __ldg(&P.tokens[b * K + j]);
        if (s.x >= 0 && s.x < V) {
            s.zx = load_elem<LT>(static_cast<const LT *>(P.logits) + r * static_cast<int64_t>(V) + s.x);
            if (DENSE)
                s.qx = __ldg(&P.q[(b * K + j) * static_cast<int64_t>(V) + s.x]);
        }
    }
    return s;
}

// The last warp of row r merges the item partials and tests the draft.
// `side` is valid in lane 0.
template <typename LT, bool DENSE>
__device__ __noinline__ void finish_row(const Params &P, int64_t r, int lane, const RowSide &side)
{
    __threadfence();
    const float c = P.c;
    const int32_t K = P.K, V = P.V;
    float M = -INFINITY, S = 0.0f;
    for (int32_t i = lane; i < P.S1; i += 32) {
        const float2 pr = __ldcg(&P.row_part[r * P.S1 + i]);
        P.row_part[r * P.S1 + i] = make_float2(0.0f, 0.0f);
        merge_ms(M, S, pr.x, pr.y, c);
    }
    warp_merge_ms(M, S, c);

    const int64_t b = divi(r, K + 1);
    const int32_t j = static_cast<int32_t>(r - b * (K + 1));
    int last_seq = 0;
    if (lane == 0) {
        int32_t bad = 0;
        const bool row_ok = isfinite(M) && isfinite(S);
        if (!row_ok)
            bad |= kBadRow;
        const float uj = side.u;
        if (!(uj >= 0.0f && uj < 1.0f))
            bad |= kBadU;
        P.row_m[r] = M;
        P.row_s[r] = S;
        P.row_cnt[r] = 0u;
        if (j < K) {
            const int32_t x = side.x;
            float a = 0.0f;
            uint8_t acc = 0;
            if (x < 0 || x >= V) {
                bad |= kBadToken;
            } else {
                const float qx = side.qx;
                if (DENSE && !(qx > 0.0f && isfinite(qx)))
                    bad |= kBadQ;
                else if (row_ok) {
                    const float px = __fdiv_rn(term(side.zx, c, mc_of(M, c)), S);
                    a = fminf(1.0f, __fdiv_rn(px, qx));
                    acc = uj < a ? 1 : 0;
                }
            }
            P.acc[b * K + j] = acc;
            if (P.accept_prob)
                P.accept_prob[b * K + j] = a;
        }
        if (bad)
            atomicOr(&P.seq_bad[b], bad);
        __threadfence();
        last_seq = atomicAdd(&P.seq_cnt[b], 1u) == static_cast<unsigned>(K);
    }
    last_seq = __shfl_sync(0xFFFFFFFFu, last_seq, 0);
    if (last_seq)
        finish_sequence<DENSE>(P, b, lane);
}

// Row item `it`: row r = it / S1, item ch = it % S1.  A row has a scalar head
// (until 16-byte aligned), whole 16-byte vectors shared out over the S1
// items, and a scalar tail.
struct ItemSpan {
    const uint4 *p;  // the item's first whole vector
    int32_t nv;      // its whole vectors
    int32_t nsteps;  // CTA steps covering them (at least one)
};

template <typename LT>
__device__ __forceinline__ const LT *row_ptr(const Params &P, int64_t r)
{
    return static_cast<const LT *>(P.logits) + r * static_cast<int64_t>(P.V);
}

template <typename LT>
__device__ __forceinline__ int32_t row_head(const LT *row, int32_t V)
{
    const int32_t h = static_cast<int32_t>(((16u - (reinterpret_cast<uintptr_t>(row) & 15u)) & 15u) / sizeof(LT));
    return h < V ? h : V;
}

template <typename LT, int STEP>
__device__ __forceinline__ ItemSpan item_span(const Params &P, int64_t it)
{
    constexpr int VW = 16 / sizeof(LT);
    const int64_t r = divi(it, P.S1);
    const int32_t ch = static_cast<int32_t>(it - r * P.S1);
    const LT *row = row_ptr<LT>(P, r);
    const int32_t head = row_head(row, P.V);
    const int32_t nvec = (P.V - head) / VW;
    const int32_t v0 = static_cast<int32_t>(static_cast<int64_t>(nvec) * ch / P.S1);
    const int32_t v1 = static_cast<int32_t>(static_cast<int64_t>(nvec) * (ch + 1) / P.S1);
    ItemSpan s;
    s.p = reinterpret_cast<const uint4 *>(row + head) + v0;
    s.nv = v1 - v0;
    s.nsteps = max(1, (s.nv + STEP - 1) / STEP);
    return s;
}

// Reduce the (max, normaliser) pairs of the 32 lanes through a common
// maximum: one exp2 per lane instead of a rescale per merge step.
__device__ __forceinline__ void warp_common_max(float &M, float &S, float c)
{
    float Mw = M;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
        Mw = fmaxf(Mw, __shfl_xor_sync(0xFFFFFFFFu, Mw, o));
    S = (M == -INFINITY) ? __fmul_rn(S, 0.0f) : __fmul_rn(S, ex2(mc_of(M, c) - mc_of(Mw, c)));
    S = warp_sum_f(S);
    M = Mw;
}

// The row pass.  Persistent CTAs take row items round-robin.  Warps 0..7
// stream: a thread folds its vectors of the item in steps of U, the next step
// (possibly of the next item) already requested while the current one is
// folded; at the end of an item each streaming warp reduces its pairs and
// hands them to warp 8 through a queue of kRowSlots shared-memory slots,
// without waiting.  Warp 8 combines the CTA's pair, publishes it, and, when
// its CTA finishes a row last, runs the accept test; so the fences and
// atomics of an item never stall the stream.  Slot hand-off uses named
// barriers: "full" (8 warps arrive, warp 8 waits) and "free" (warp 8
// arrives, the 8 warps wait before reusing the slot kRowSlots items later).
constexpr int kRowSlots = 4;
constexpr int kRowCtaThreads = kThreads + 32;

template <typename LT, bool DENSE>
__global__ void __launch_bounds__(kRowCtaThreads, SV_ROW_MIN_CTAS) rows_kernel(const Params P)
{
    constexpr int VW = 16 / sizeof(LT);
    constexpr int U = 4;                 // vectors per thread per step
    constexpr int STEP = kThreads * U;   // vectors per CTA step
    __shared__ float sM[kRowSlots][kWarps], sS[kRowSlots][kWarps];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const float c = P.c;
    const int64_t n_items = P.B * P.RI;
    const int64_t G = gridDim.x;
    if (static_cast<int64_t>(blockIdx.x) >= n_items)
        return;
    const int n_mine = static_cast<int>((n_items - 1 - blockIdx.x) / G) + 1; // items of this CTA
    auto bar_full = [](int q) { return 1u + static_cast<uint32_t>(q); };
    auto bar_free = [](int q) { return 1u + kRowSlots + static_cast<uint32_t>(q); };

    if (warp == kWarps) {
        // ---- epilogue warp
        for (int k = 0; k < n_mine; ++k) {
            const int64_t it = blockIdx.x + static_cast<int64_t>(k) * G;
            const int64_t r = divi(it, P.S1);
            RowSide side;
            if (lane == 0)
                side = fetch_side<LT, DENSE>(P, r); // in flight while the item streams
            const int q = k % kRowSlots;
            bar_sync(bar_full(q), kRowCtaThreads);
            float M = lane < kWarps ? sM[q][lane] : -INFINITY;
            float S = lane < kWarps ? sS[q][lane] : 0.0f;
            if (k + kRowSlots < n_mine)
                bar_arrive(bar_free(q), kRowCtaThreads);
            warp_common_max(M, S, c);
            int last = 0;
            if (lane == 0) {
                P.row_part[it] = make_float2(M, S);
                __threadfence();
                last = atomicAdd(&P.row_cnt[r], 1u) == static_cast<unsigned>(P.S1 - 1);
            }
            last = __shfl_sync(0xFFFFFFFFu, last, 0);
            if (last)
                finish_row<LT, DENSE>(P, r, lane, side);
        }
        pdl_launch_dependents();
        return;
    }

    // ---- streaming warps
    const uint4 neg_inf = sizeof(LT) == 2 ? make_uint4(0xFF80FF80u, 0xFF80FF80u, 0xFF80FF80u, 0xFF80FF80u)
                                          : make_uint4(0xFF800000u, 0xFF800000u, 0xFF800000u, 0xFF800000u);
    auto load_step = [&](const ItemSpan &sp, int s, uint4 (&w)[U]) {
#pragma unroll
        for (int k = 0; k < U; ++k) {
            const int32_t e = s * STEP + tid + k * kThreads;
            w[k] = e < sp.nv ? ld_stream_v4(sp.p + e) : neg_inf;
        }
    };
    int k = 0;
    int64_t it = blockIdx.x;
    ItemSpan sp = item_span<LT, STEP>(P, it);
    int s = 0;
    uint4 cur[U], nxt[U];
    load_step(sp, 0, cur);
    float M = -INFINITY;
    unsigned long long S[4] = {0ull, 0ull, 0ull, 0ull}; // packed (+0, +0) pairs
    for (;;) {
        // the next step, possibly of the next item, is requested first
        ItemSpan spn = sp;
        int64_t itn = it;
        int sn = s + 1;
        if (sn >= sp.nsteps) {
            itn = it + G;
            sn = 0;
            if (itn < n_items)
                spn = item_span<LT, STEP>(P, itn);
        }
        const bool more = itn < n_items;
        if (more)
            load_step(spn, sn, nxt);
        fold<LT, U>(cur, M, S, c);

        if (s + 1 >= sp.nsteps) {
            // ---- end of item `it`: reduce and hand the pair to the epilogue warp
            float a0, a1;
            unpack2(add2(add2(S[0], S[1]), add2(S[2], S[3])), a0, a1);
            float Ssum = __fadd_rn(a0, a1);
            const int64_t r = divi(it, P.S1);
            const int32_t ch = static_cast<int32_t>(it - r * P.S1);
            if (ch == 0 || ch == P.S1 - 1) {
                const LT *row = row_ptr<LT>(P, r);
                const int32_t head = row_head(row, P.V);
                const int32_t tail0 = head + (P.V - head) / VW * VW;
                if (ch == 0)
                    for (int32_t e = tid; e < head; e += kThreads)
                        merge_ms(M, Ssum, load_elem<LT>(row + e), 1.0f, c);
                if (ch == P.S1 - 1)
                    for (int32_t e = tail0 + tid; e < P.V; e += kThreads)
                        merge_ms(M, Ssum, load_elem<LT>(row + e), 1.0f, c);
            }
            warp_common_max(M, Ssum, c);
            const int q = k % kRowSlots;
            if (k >= kRowSlots)
                bar_sync(bar_free(q), kRowCtaThreads); // the epilogue has read the slot's last use
            if (lane == 0) {
                sM[q][warp] = M;
                sS[q][warp] = Ssum;
            }
            bar_arrive(bar_full(q), kRowCtaThreads);
            ++k;
            M = -INFINITY;
#pragma unroll
            for (int a = 0; a < 4; ++a)
                S[a] = 0ull;
        }
        if (!more)
            break;
#pragma unroll
        for (int j = 0; j < U; ++j)
            cur[j] = nxt[j];
        sp = spn;
        it = itn;
        s = sn;
    }
    pdl_launch_dependents();
}

} // namespace sv
