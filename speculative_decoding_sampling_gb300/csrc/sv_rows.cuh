// sv_rows.cuh -- the row pass of the verification step.
//
// Every one of the B*(K+1) target rows is streamed once from HBM.  The rows
// are one flat array; each CTA streams one contiguous span of it with 16-byte
// loads, the next step in flight while the current one is folded.  Each thread
// keeps an online (max, normaliser) pair of softmax(z / T) in the base-2 form
// sum_i exp2(z_i * c - fl(M * c)), c = log2(e) / T (one exp2 per element).
// Each CTA publishes one (max, normaliser) pair per row it touches, and the
// CTA holding a row's first id also publishes the row's draft data (x, z(x),
// q(x), u); the draw stream turns these into the sequence's verdict once the
// pass has completed (the kernel boundary is the only synchronisation).
#pragma once

#include <climits>

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

// Fold U vectors into the running (M, S) of one lane; S holds two packed
// pairs of partial sums (four accumulators).
template <typename LT, int U>
__device__ __forceinline__ void fold(const uint4 (&w)[U], float &M, unsigned long long (&S)[2], float c)
{
    const float gm = vec_max<LT, U>(w);
    if (gm > M) {
        // rescale what was summed against the old maximum
        const float f = (M == -INFINITY) ? 0.0f : ex2(mc_of(M, c) - mc_of(gm, c));
        const unsigned long long f2 = pack2(f, f);
        S[0] = mul2(S[0], f2);
        S[1] = mul2(S[1], f2);
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
                S[h & 1] = add2(S[h & 1], pack2(ex2(y0), ex2(y1)));
            }
        } else {
#pragma unroll
            for (int h = 0; h < 4; h += 2) {
                float y0, y1;
                unpack2(fma2(pack2(__uint_as_float(v[h]), __uint_as_float(v[h + 1])), c2, nmc2), y0, y1);
                S[(h >> 1)] = add2(S[(h >> 1)], pack2(ex2(y0), ex2(y1)));
            }
        }
    }
}

// What a row's accept test needs besides its (max, normaliser): fetched by
// the epilogue warp of the CTA holding the row's first id, while the row
// streams, and published beside that CTA's partial.
struct RowSide {
    int32_t x;  // draft token verified by this row (j < K), else -1
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

// The flat view of the logits.  The B*(K+1) rows of V ids are one array of
// R*V elements.  From the first 16-byte boundary on it is cut into whole
// 16-byte vectors 1..nvec; "vector" 0 stands for the h elements before that
// boundary and vector nvec+1 for the ragged end.  CTA g owns the vectors
// [g*span, (g+1)*span): one contiguous piece of HBM.  A vector is streamed
// (read with one 16-byte load by a streaming warp) when it is whole and all
// its ids lie in one row; the others -- the two ragged ends and, when
// V * element size is not a multiple of 16 or the array is not 16-byte
// aligned, the vectors that straddle a row boundary -- are read id by id by
// the epilogue warp of the CTA that owns them, once for each row they touch.
// Each row's partial (max, normaliser) pairs come from the CTAs its ids fall
// in; CTA g writes its pair of row r into slot g - first_cta(r) of the row.

template <typename LT>
__device__ __forceinline__ bool streamed(const Params &P, int64_t vv)
{
    constexpr int VW = 16 / sizeof(LT);
    const int64_t e0 = P.h + (vv - 1) * VW;
    return vv >= 1 && vv <= P.nvec && divi(e0, P.V) == divi(e0 + VW - 1, P.V);
}

// The streamed vectors of row r inside vectors [vbeg, vend), as offsets
// [b, e) relative to vbeg.
template <typename LT>
__device__ __forceinline__ void row_vectors(const Params &P, int64_t r, int64_t vbeg, int64_t vend, int &b, int &e)
{
    constexpr int VW = 16 / sizeof(LT);
    const int64_t lo = r * P.V - P.h, hi = (r + 1) * P.V - P.h; // ids relative to vector 1's first id
    // first vector starting at or after the row's first id; first vector
    // ending after its last id (lo > -VW and hi > -VW, so the divisions of
    // non-negative numbers below are floors)
    const int64_t vs = (lo + VW - 1 + VW) / VW;
    const int64_t ve = (hi + VW) / VW;
    const int64_t vb = max(max(vs, int64_t{1}), vbeg);
    const int64_t vx = min(min(ve, P.nvec + 1), vend);
    b = static_cast<int>(vb - vbeg);
    e = static_cast<int>(max(vx, vb) - vbeg);
}

// The epilogue lane's share of the ids of row r that CTA g reads one by
// one: lanes 16.. take the vector holding the row's first id, lanes 24.. the
// one holding its last id (when it is another vector), each only if that
// vector is not streamed and belongs to CTA g.  A lane's pair is (z, 1), or
// stays (-inf, 0) when it has none.
template <typename LT>
__device__ __forceinline__ void ragged_pair(const Params &P, int64_t g, int64_t r, int lane, float &M, float &S)
{
    constexpr int VW = 16 / sizeof(LT);
    const int64_t vf = vec_of_elem<LT>(P, r * P.V);
    const int64_t vl = vec_of_elem<LT>(P, r * P.V + P.V - 1);
    int64_t vv = -1;
    int i = 0;
    if (lane >= 16 && lane < 16 + VW) {
        vv = vf;
        i = lane - 16;
    } else if (lane >= 24 && lane < 24 + VW && vl != vf) {
        vv = vl;
        i = lane - 24;
    }
    if (vv < 0 || divi(vv, P.span) != g || streamed<LT>(P, vv))
        return;
    const int64_t e = P.h + (vv - 1) * VW + i;
    if (e >= 0 && e < P.total && e / P.V == r) {
        M = load_elem<LT>(static_cast<const LT *>(P.logits) + e);
        S = 1.0f;
    }
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

// The row pass.  The kRowWarps streaming warps walk the CTA's span row by
// row: a thread folds U vectors per step, the next step (possibly of the next
// row) already requested while the current one is folded; a step never
// crosses a row's end.  When a row's part of the span is done, each streaming
// warp reduces its pairs and hands them to the epilogue warp (the last one)
// through a queue of kRowSlots shared-memory slots, without waiting.  The
// epilogue warp adds the row's ids it reads one by one, combines the CTA's
// pair, publishes it, and, when its CTA completes a row last, runs the accept
// test; so the fences and atomics of a row never stall the stream.  Slot
// hand-off uses named barriers: "full" (streaming warps arrive, the epilogue
// warp waits) and "free" (the epilogue warp arrives, the streaming warps wait
// before reusing the slot kRowSlots rows later).
constexpr int kRowSlots = 4;
constexpr int kRowWarps = SV_ROW_WARPS;            // streaming warps of a CTA
constexpr int kRowThreads = kRowWarps * 32;
constexpr int kRowCtaThreads = kRowThreads + 32;   // and the epilogue warp
constexpr int kRowU = SV_ROW_U;                    // vectors per thread per step
constexpr int kRowStep = kRowThreads * kRowU;      // vectors per CTA step
static_assert(kRowWarps >= 1 && kRowWarps <= 16 && kRowU >= 1, "row CTA shape (lanes 16..31 of the epilogue warp read ragged ids)");
constexpr int64_t kRowMaxSpan = int64_t{1} << 30; // keeps offsets inside a span in int

template <typename LT, bool DENSE>
__global__ void __launch_bounds__(kRowCtaThreads, SV_ROW_MIN_CTAS) rows_kernel(const Params P)
{
    constexpr int VW = 16 / sizeof(LT);
    constexpr int U = kRowU;
    constexpr int STEP = kRowStep;
    __shared__ float sM[kRowSlots][kRowWarps], sS[kRowSlots][kRowWarps];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const float c = P.c;
    const int64_t V = P.V;
    const int64_t g = blockIdx.x;
    const int64_t vbeg = g * P.span;
    const int64_t vend = min(P.NV, vbeg + P.span);
    // the span's elements [E0, E1) and rows r0..r1
    const int64_t E0 = max(int64_t{0}, P.h + (vbeg - 1) * VW);
    const int64_t E1 = min(P.total, P.h + (vend - 1) * VW);
    const int64_t r0 = E0 / V;
    const int n_rows = E1 > E0 ? static_cast<int>((E1 - 1) / V - r0 + 1) : 0;
    auto bar_full = [](int q) { return 1u + static_cast<uint32_t>(q); };
    auto bar_free = [](int q) { return 1u + kRowSlots + static_cast<uint32_t>(q); };

    if (warp == kRowWarps) {
        // ---- epilogue warp: the CTA's pair of each row, and the draft data
        // of the rows whose first id it holds (fetched ahead, in parallel)
        RowSide pre = {-1, 0.0f, 1.0f, 0.0f};
        if (lane < n_rows && divi(vec_of_elem<LT>(P, (r0 + lane) * V), P.span) == g)
            pre = fetch_side<LT, DENSE>(P, r0 + lane);
        for (int k = 0; k < n_rows; ++k) {
            const int64_t r = r0 + k;
            const int64_t first = divi(vec_of_elem<LT>(P, r * V), P.span);
            const bool head = g == first; // this CTA holds the row's first id
            RowSide side = {-1, 0.0f, 1.0f, 0.0f};
            if (k < 32) {
                side.x = __shfl_sync(0xFFFFFFFFu, pre.x, k);
                side.zx = __shfl_sync(0xFFFFFFFFu, pre.zx, k);
                side.qx = __shfl_sync(0xFFFFFFFFu, pre.qx, k);
                side.u = __shfl_sync(0xFFFFFFFFu, pre.u, k);
            } else if (lane == 0 && head) {
                side = fetch_side<LT, DENSE>(P, r);
            }
            float M = -INFINITY, S = 0.0f;
            ragged_pair<LT>(P, g, r, lane, M, S);
            const int q = k % kRowSlots;
            bar_sync(bar_full(q), kRowCtaThreads);
            if (lane < kRowWarps) {
                M = sM[q][lane];
                S = sS[q][lane];
            }
            if (k + kRowSlots < n_rows)
                bar_arrive(bar_free(q), kRowCtaThreads);
            warp_common_max(M, S, c);
            if (lane == 0) {
                P.row_part[r * P.PM + (g - first)] = make_float2(M, S);
                if (head)
                    P.row_side[r] = make_float4(__int_as_float(side.x), side.zx, side.qx, side.u);
            }
        }
        pdl_launch_dependents();
        return;
    }

    // ---- streaming warps: row r0 + k's streamed vectors of the span, in
    // steps of STEP vectors; one flush per row
    if (n_rows > 0) {
        const uint4 neg_inf = sizeof(LT) == 2 ? make_uint4(0xFF80FF80u, 0xFF80FF80u, 0xFF80FF80u, 0xFF80FF80u)
                                              : make_uint4(0xFF800000u, 0xFF800000u, 0xFF800000u, 0xFF800000u);
        const uint4 *base = reinterpret_cast<const uint4 *>(static_cast<const LT *>(P.logits) + P.h) + (vbeg - 1);
        // the step at offset off of a row whose streamed vectors end at offset e
        auto load_step = [&](int off, int e, uint4 (&w)[U]) {
#pragma unroll
            for (int k = 0; k < U; ++k) {
                const int i = off + k * kRowThreads + tid;
                w[k] = i < e ? ld_stream_v4(base + i) : neg_inf;
            }
        };
        const int64_t r_last = r0 + n_rows - 1;
        int64_t row = r0;
        int off, e;
        row_vectors<LT>(P, row, vbeg, vend, off, e);
        float M = -INFINITY;
        unsigned long long S[2] = {0ull, 0ull}; // packed (+0, +0) pairs
        uint4 cur[U], nxt[U];
        load_step(off, e, cur);
        for (int k = 0;;) {
            // the next step, possibly of the next row, is requested first
            int noff = off + STEP, ne = e;
            const bool row_done = noff >= e;
            if (row_done && row < r_last)
                row_vectors<LT>(P, row + 1, vbeg, vend, noff, ne);
            const bool more = !row_done || row < r_last;
            if (more)
                load_step(noff, ne, nxt);
            fold<LT, U>(cur, M, S, c);
            if (row_done) {
                // hand the row's pairs to the epilogue warp
                float a0, a1;
                unpack2(add2(S[0], S[1]), a0, a1);
                float Ssum = __fadd_rn(a0, a1);
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
                ++row;
                M = -INFINITY;
                S[0] = S[1] = 0ull;
            }
            if (!more)
                break;
#pragma unroll
            for (int j = 0; j < U; ++j)
                cur[j] = nxt[j];
            off = noff;
            e = ne;
        }
    }
    pdl_launch_dependents();
}

} // namespace sv
