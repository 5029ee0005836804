// sv_survivor.cuh -- the final draw of each sequence.
//
// After its rows, every sequence has one surviving row j*: the row of its
// first rejection, or row K when every draft passed.  The final token is
// drawn from
//   rejected, dense q:  r_i = max(0, p_i - q_i)   (p = softmax(z_{j*} / T))
//   rejected, one-hot:  r_i = p_i for i != x, r_x = 0
//   all accepted:       p_i of row K
// by inverse CDF with the final uniform u_K: the smallest id i with
// u_K * sum(r) < r_0 + ... + r_i ("推测解码：草稿、验证与实际加速", sections
// 接受与拒绝怎样保住分布 (equation for r(x)) and 算完三个 token 的全部概率
// (the replay's sampler and its final draw)).
//
// A lane owns groups of 8 consecutive ids; a warp tile is 32 groups and a
// chunk 4 tiles (1024 ids).  Every sequence's surviving row is cut into
// chunks; the B * CPS chunks of the call are split into one contiguous range
// per warp, which streams them through its async-copy ring several tiles
// ahead, across chunk and sequence boundaries.  Per element:
//   e_i  = exp2(z_i * c - fl(m * c))          (m: the row maximum)
//   pt_i = e_i / s~                           (s~: the row pass's fp32 normaliser)
//   w_i  = max(0, pt_i - q_i) | pt_i with x removed | pt_i
// (the last two with q = 0: an accepted sequence of a dense launch takes
// the dense form with q = 0, of a one-hot launch the one-hot form with no x).
// The 8 masses of a group are added in fp32 in id order and the group total
// is held as an integer multiple of 2^-fix_bits, so every sum over groups,
// tiles and chunks is exact and order-independent; the draw re-forms groups
// with the same arithmetic, so its boundaries agree with the totals.
//
// The dense residual needs the exact normaliser, not s~: with
// S' = sum_i pt_i (accumulated error-free per element, Fast2Sum), the true
// residual is proportional to pt_i - S' q_i = w_i - (S' - 1) q_i on the ids
// where it is positive.  So each chunk also carries Qp = sum of q_i over the
// ids with w_i > 0, and every boundary is taken as A - (S' - 1) * Qp.  (Ids
// within |S' - 1| q_i of the kink move by less than one fp32 ulp of their own
// mass.)  Each chunk publishes one record (A, Qp); the normalisers are
// integer sums, added atomically once per warp and sequence.  The warp that
// completes a sequence's last chunk combines the records, finds the chunk and
// the id that hold u_K * Z, and clears the sequence's scratch.
#pragma once

#include <climits>
#include <type_traits>

#include "sv_verdict.cuh"

namespace sv {

enum { kModeBonus = 0, kModeDense = 1, kModeOneHot = 2 };

struct SurvArgs {
    float c, mc;   // log2(e)/T and fl(m*c) of the surviving row
    float inv_s;   // 1 / s~
    int fb;        // fix_bits: masses are integer multiples of 2^-fb
    int32_t x;     // rejected one-hot draft
};

// z (and q) of the 8 ids of group g; ids at or past group g_end, or past the
// row, read as -inf (and 0).
template <typename LT, bool WANT_Q>
__device__ __forceinline__ void load_group(const LT *row, const float *qrow, int32_t g, int32_t g_end, int32_t V,
                                           bool vec_ok, float (&z)[kGroup], float (&q)[kGroup])
{
    const int32_t e0 = g * kGroup;
    if (g < g_end && vec_ok && e0 + kGroup <= V) {
        if constexpr (sizeof(LT) == 2) {
            const uint4 w = ld_stream_v4(row + e0);
            z[0] = bf16_lo(w.x); z[1] = bf16_hi(w.x);
            z[2] = bf16_lo(w.y); z[3] = bf16_hi(w.y);
            z[4] = bf16_lo(w.z); z[5] = bf16_hi(w.z);
            z[6] = bf16_lo(w.w); z[7] = bf16_hi(w.w);
        } else {
            const uint4 a = ld_stream_v4(row + e0), b = ld_stream_v4(row + e0 + 4);
            z[0] = __uint_as_float(a.x); z[1] = __uint_as_float(a.y);
            z[2] = __uint_as_float(a.z); z[3] = __uint_as_float(a.w);
            z[4] = __uint_as_float(b.x); z[5] = __uint_as_float(b.y);
            z[6] = __uint_as_float(b.z); z[7] = __uint_as_float(b.w);
        }
        if constexpr (WANT_Q) {
            const uint4 a = ld_stream_v4(qrow + e0), b = ld_stream_v4(qrow + e0 + 4);
            q[0] = __uint_as_float(a.x); q[1] = __uint_as_float(a.y);
            q[2] = __uint_as_float(a.z); q[3] = __uint_as_float(a.w);
            q[4] = __uint_as_float(b.x); q[5] = __uint_as_float(b.y);
            q[6] = __uint_as_float(b.z); q[7] = __uint_as_float(b.w);
        } else {
#pragma unroll
            for (int k = 0; k < kGroup; ++k)
                q[k] = 0.0f;
        }
    } else {
#pragma unroll
        for (int k = 0; k < kGroup; ++k) {
            const bool in = g < g_end && e0 + k < V;
            z[k] = in ? load_elem<LT>(row + e0 + k) : -INFINITY;
            q[k] = (WANT_Q && in) ? __ldg(qrow + e0 + k) : 0.0f;
        }
    }
}

// The shape of a draw warp's ring for one launch: a stage holds one chunk,
// the logits of its 128 groups (LB bytes each) then their draft
// probabilities (32 bytes each, dense launches).
template <typename LT, bool DENSE>
struct DrawShape {
    static constexpr int LB = kGroup * static_cast<int>(sizeof(LT));
    static constexpr int QB = DENSE ? kGroup * 4 : 0;
    static constexpr int kChunkBytes = kChunkGroups * (LB + QB);
    static constexpr int kWarpBytes = kDrawStages * kChunkBytes;
    static constexpr int kCtaBytes = kDrawWarps * kWarpBytes;
};

// z (and q) of group gl (0..127) of the chunk in ring stage `st`.
template <typename LT, bool WANT_Q>
__device__ __forceinline__ void load_group_smem(const uint8_t *st, int gl, bool in, float (&z)[kGroup],
                                                float (&q)[kGroup])
{
    constexpr int LB = kGroup * sizeof(LT);
    if (!in) {
#pragma unroll
        for (int k = 0; k < kGroup; ++k) {
            z[k] = -INFINITY;
            q[k] = 0.0f;
        }
        return;
    }
    if constexpr (sizeof(LT) == 2) {
        const uint4 w = lds_v4(st + gl * LB);
        z[0] = bf16_lo(w.x); z[1] = bf16_hi(w.x);
        z[2] = bf16_lo(w.y); z[3] = bf16_hi(w.y);
        z[4] = bf16_lo(w.z); z[5] = bf16_hi(w.z);
        z[6] = bf16_lo(w.w); z[7] = bf16_hi(w.w);
    } else {
        const uint4 a = lds_v4(st + gl * LB), b = lds_v4(st + gl * LB + 16);
        z[0] = __uint_as_float(a.x); z[1] = __uint_as_float(a.y);
        z[2] = __uint_as_float(a.z); z[3] = __uint_as_float(a.w);
        z[4] = __uint_as_float(b.x); z[5] = __uint_as_float(b.y);
        z[6] = __uint_as_float(b.z); z[7] = __uint_as_float(b.w);
    }
    if constexpr (WANT_Q) {
        const uint8_t *qs = st + kChunkGroups * LB + gl * 32;
        const uint4 a = lds_v4(qs), b = lds_v4(qs + 16);
        q[0] = __uint_as_float(a.x); q[1] = __uint_as_float(a.y);
        q[2] = __uint_as_float(a.z); q[3] = __uint_as_float(a.w);
        q[4] = __uint_as_float(b.x); q[5] = __uint_as_float(b.y);
        q[6] = __uint_as_float(b.z); q[7] = __uint_as_float(b.w);
    } else {
#pragma unroll
        for (int k = 0; k < kGroup; ++k)
            q[k] = 0.0f;
    }
}

// load_group with q read only where there is a draft row (qrow != nullptr),
// 0 elsewhere.
template <typename LT, bool DENSE>
__device__ __forceinline__ void load_group_any(const LT *row, const float *qrow, int32_t g, int32_t g_end, int32_t V,
                                               bool vec_ok, float (&z)[kGroup], float (&q)[kGroup])
{
    if (DENSE && qrow != nullptr)
        load_group<LT, true>(row, qrow, g, g_end, V, vec_ok, z, q);
    else
        load_group<LT, false>(row, nullptr, g, g_end, V, vec_ok, z, q);
}

// The masses of one group: pt_i, w_i (the mass the draw uses) and qp_i (q_i
// where w_i > 0, dense; else 0), and the group totals ws = sum w, qs = sum qp.
// Ids are taken in pairs (2h, 2h+1) with packed fp32 arithmetic; each total
// is added in the fixed order ((x0 + x2) + x4) + x6 + ((x1 + x3) + x5) + x7.
// The fold and the draw's scan both use this routine, so they see identical
// group totals.  NORM: pt_i = e_i / s~ (dense launches); otherwise pt_i = e_i
// (a one-hot or extra-token draw needs no normaliser: its boundaries are
// relative to its own total).
template <int MODE, bool NORM>
__device__ __forceinline__ void group_masses(const float (&z)[kGroup], const float (&q)[kGroup], int32_t e0,
                                             const SurvArgs &X, unsigned long long (&pt2)[kGroup / 2],
                                             float (&w)[kGroup], float (&qp)[kGroup], float &ws, float &qs)
{
    const unsigned long long c2 = pack2(X.c, X.c), nmc2 = pack2(-X.mc, -X.mc), inv2 = pack2(X.inv_s, X.inv_s);
    const unsigned long long m1 = pack2(-1.0f, -1.0f);
    unsigned long long wsum = 0ull, qsum = 0ull; // packed (+0, +0)
#pragma unroll
    for (int h = 0; h < kGroup / 2; ++h) {
        const int k = 2 * h;
        float y0, y1;
        unpack2(fma2(pack2(z[k], z[k + 1]), c2, nmc2), y0, y1);
        pt2[h] = NORM ? mul2(pack2(ex2(y0), ex2(y1)), inv2) : pack2(ex2(y0), ex2(y1));
        if (MODE == kModeDense) {
            float d0, d1;
            unpack2(fma2(pack2(q[k], q[k + 1]), m1, pt2[h]), d0, d1); // pt - q
            w[k] = fmaxf(d0, 0.0f);
            w[k + 1] = fmaxf(d1, 0.0f);
            qp[k] = d0 > 0.0f ? q[k] : 0.0f;
            qp[k + 1] = d1 > 0.0f ? q[k + 1] : 0.0f;
            qsum = add2(qsum, pack2(qp[k], qp[k + 1]));
        } else {
            float p0, p1;
            unpack2(pt2[h], p0, p1);
            w[k] = (MODE == kModeOneHot && e0 + k == X.x) ? 0.0f : p0;
            w[k + 1] = (MODE == kModeOneHot && e0 + k + 1 == X.x) ? 0.0f : p1;
            qp[k] = qp[k + 1] = 0.0f;
        }
        wsum = add2(wsum, pack2(w[k], w[k + 1]));
    }
    float a0, a1;
    unpack2(wsum, a0, a1);
    ws = __fadd_rn(a0, a1);
    unpack2(qsum, a0, a1);
    qs = __fadd_rn(a0, a1);
}

// The correction term of the dense residual's boundaries, in 2^-fb units:
// (S' - 1) * Qp * 2^fb = delta * Qp with delta = E - 2^fb (E: the exact
// sum of pt in 2^-fb units), rounded to an integer.
__device__ __forceinline__ long long corr_of(float delta, float qp)
{
    return to_fixed(__fmul_rn(delta, qp), 0);
}


// The surviving row of sequence b (and its draft row, dense and rejected).
template <typename LT, bool DENSE>
__device__ __forceinline__ void seq_rows(const Params &P, int64_t b, const Verdict &v, const LT *&row,
                                         const float *&qrow)
{
    const int64_t V = P.V;
    row = static_cast<const LT *>(P.logits) + (b * (P.K + 1) + (v.jstar < 0 ? 0 : v.jstar)) * V;
    qrow = (DENSE && v.jstar >= 0 && v.jstar < P.K) ? P.q + (b * P.K + v.jstar) * V : nullptr;
}

__device__ __forceinline__ SurvArgs surv_args(const Params &P, const Verdict &v)
{
    SurvArgs X;
    X.c = P.c;
    X.mc = mc_of(v.m, P.c);
    X.inv_s = __frcp_rn(v.s);
    X.fb = P.fix_bits;
    X.x = v.x;
    return X;
}

// The masses of one lane's group for a launch: MODE kModeDense (q = 0 for an
// accepted sequence) or kModeOneHot (x = -1 for an accepted sequence).
template <bool DENSE>
struct LaunchMode {
    static constexpr int value = DENSE ? kModeDense : kModeOneHot;
};

// How a chunk of the draw stream is folded: the residual of a rejection
// with dense q, the one-hot residual, or p itself (every draft accepted; the
// same masses as the dense form with q = 0 and the one-hot form with no x).
// kFoldOneHotNoX: a chunk of a one-hot residual that does not hold the
// rejected draft id (every chunk but one): the masses are p itself.
enum { kFoldDense = 0, kFoldOneHot = 1, kFoldBonus = 2, kFoldOneHotNoX = 3 };

// Fold one group into the lane's running totals: the chunk's A (sum of the
// group masses in 2^-fb units) and Qs (sum of qp), and, for a dense
// rejection, the sequence's normaliser share (Ehi, Elo), an error-free
// (Fast2Sum) running sum of pt per id parity.  Only the group totals are
// formed; they equal group_masses' bit for bit (the same per-pair
// arithmetic, added in the same order).
template <int KIND, bool NORM>
__device__ __forceinline__ void fold_group(const float (&z)[kGroup], const float (&q)[kGroup], int32_t e0,
                                           const SurvArgs &X, unsigned long long &Ehi, unsigned long long &Elo,
                                           long long &A, float &Qs)
{
    const unsigned long long c2 = pack2(X.c, X.c), nmc2 = pack2(-X.mc, -X.mc), inv2 = pack2(X.inv_s, X.inv_s);
    const unsigned long long m1 = pack2(-1.0f, -1.0f);
    unsigned long long wsum = 0ull, qsum = 0ull; // packed (+0, +0)
    const bool xin = KIND == kFoldOneHot && static_cast<unsigned>(X.x - e0) < static_cast<unsigned>(kGroup);
#pragma unroll
    for (int h = 0; h < kGroup / 2; ++h) {
        const int k = 2 * h;
        float y0, y1;
        unpack2(fma2(pack2(z[k], z[k + 1]), c2, nmc2), y0, y1);
        const unsigned long long pt2 = NORM ? mul2(pack2(ex2(y0), ex2(y1)), inv2) : pack2(ex2(y0), ex2(y1));
        if (KIND == kFoldDense) { // |Ehi| >= 2 > every pt
            const unsigned long long s = add2(Ehi, pt2);
            const unsigned long long tt = fma2(Ehi, m1, s);       // s - Ehi
            Elo = add2(Elo, fma2(tt, m1, pt2));                  // + (pt - tt)
            Ehi = s;
            float d0, d1;
            unpack2(fma2(pack2(q[k], q[k + 1]), m1, pt2), d0, d1); // pt - q
            wsum = add2(wsum, pack2(fmaxf(d0, 0.0f), fmaxf(d1, 0.0f)));
            qsum = add2(qsum, pack2(d0 > 0.0f ? q[k] : 0.0f, d1 > 0.0f ? q[k + 1] : 0.0f));
        } else if (KIND == kFoldOneHotNoX) {
            wsum = add2(wsum, pt2);
        } else if (KIND == kFoldOneHot) {
            unsigned long long w2 = pt2;
            if (xin) { // the rejected draft's own id carries no residual mass
                float p0, p1;
                unpack2(pt2, p0, p1);
                w2 = pack2(e0 + k == X.x ? 0.0f : p0, e0 + k + 1 == X.x ? 0.0f : p1);
            }
            wsum = add2(wsum, w2);
        } else {
            wsum = add2(wsum, pt2);
        }
    }
    float a0, a1;
    unpack2(wsum, a0, a1);
    A += to_fixed(__fadd_rn(a0, a1), X.fb);
    if (KIND == kFoldDense) {
        unpack2(qsum, a0, a1);
        Qs = __fadd_rn(Qs, __fadd_rn(a0, a1));
    }
}

// The final draw of sequence b by the draw warp that completes its chunk
// count, staging the chosen chunk in ring stage `stage` (sv_final.cuh).
template <typename LT, bool DENSE, bool RING>
__device__ void final_inline(const Params &P, int64_t b, const Verdict &v, int lane, uint8_t *stage);

// What a ring stage's consumer needs about the chunk's sequence: written by
// the issue side (which computed the verdict) when it issues the chunk.
struct StageInfo {
    int32_t jstar; // -1: bad sequence (nothing to fold)
    float m, s;
    int32_t x;
};

// The chunks [c0, c1) of one warp.  RING: rows of whole, 16-byte aligned
// groups stream through the warp's ring, kDrawStages - 1 chunks ahead, a
// lane copying (and later reading) its own 4 groups of each chunk; otherwise
// each lane loads its groups directly.  The issue side meets each sequence
// first and computes its verdict (the warp that issues a sequence's chunk 0
// also writes the sequence's outputs); the consumer folds the chunks,
// writes one record per chunk and, per sequence, adds its share of the
// normaliser.
template <typename LT, bool DENSE, bool RING>
__device__ __forceinline__ void draw_range(const Params &P, int64_t c0, int64_t c1, int lane, uint8_t *ring,
                                           StageInfo *info)
{
    using Shape = DrawShape<LT, DENSE>;
    constexpr int LB = Shape::LB;
    const int32_t V = P.V, K = P.K, CPS = P.CPS;
    const int32_t ng = (V + kGroup - 1) / kGroup;
    const int64_t nchunks = c1 - c0;

    // ---- issue side: the chunk kDrawStages - 1 ahead of the consumer
    int64_t ib = divi(c0, CPS);
    int32_t icis = static_cast<int32_t>(c0 - ib * CPS);
    int ist = 0;       // ring stage of the next issued chunk
    int64_t iseq = -1; // sequence whose verdict iv holds
    Verdict iv = {-1, 0.0f, 1.0f, -1};
    const LT *irow = nullptr;
    const float *iq = nullptr;
    auto issue = [&](int64_t k) {
        if (k < nchunks) {
            if (ib != iseq) {
                iv = seq_verdict<LT, DENSE>(P, ib, lane, icis == 0);
                seq_rows<LT, DENSE>(P, ib, iv, irow, iq);
                iseq = ib;
            }
            if (lane == 0)
                info[ist] = StageInfo{iv.jstar, iv.m, iv.s, iv.x};
            if (RING && iv.jstar >= 0) {
                uint8_t *st = ring + ist * Shape::kChunkBytes;
                const int32_t g0 = icis * kChunkGroups + lane;
                const uint8_t *src = reinterpret_cast<const uint8_t *>(irow + static_cast<int64_t>(g0) * kGroup);
                const uint8_t *qsrc =
                    DENSE && iq ? reinterpret_cast<const uint8_t *>(iq + static_cast<int64_t>(g0) * kGroup) : nullptr;
                const bool full = (icis + 1) * kChunkGroups <= ng; // every group of the chunk in the row
#pragma unroll
                for (int t = 0; t < kChunkTiles; ++t) {
                    if (full || g0 + 32 * t < ng) {
                        const int gl = 32 * t + lane;
#pragma unroll
                        for (int h = 0; h < LB; h += 16)
                            cp_async16(st + gl * LB + h, src + 32 * t * LB + h);
                        if (DENSE && qsrc) {
                            cp_async16(st + kChunkGroups * LB + gl * 32, qsrc + 32 * t * 32);
                            cp_async16(st + kChunkGroups * LB + gl * 32 + 16, qsrc + 32 * t * 32 + 16);
                        }
                    }
                }
            }
            if (++icis == CPS) {
                icis = 0;
                ++ib;
            }
            ist = ist + 1 == kDrawStages ? 0 : ist + 1;
        }
        if (RING)
            cp_async_commit();
    };

    // ---- consumer side
    int64_t cb = divi(c0, CPS);
    int32_t ccis = static_cast<int32_t>(c0 - cb * CPS);
    int cst = 0;      // ring stage of chunk k
    int64_t cur = -1; // sequence whose totals are being accumulated
    SurvArgs X = {};
    Verdict cv = {-1, 0.0f, 1.0f, -1};
    int32_t ccount = 0; // chunks of `cur` folded by this warp
    bool cvalid = false, cdraft = false, cvec = false;
    const LT *crow = nullptr;
    const float *cq = nullptr;
    const unsigned long long E0 = DENSE ? pack2(2.0f, 2.0f) : 0ull;
    unsigned long long Ehi = E0, Elo = 0ull; // see fold_group
    auto flush = [&]() {
        // the dense rejection's share of its normaliser E = sum pt, in 2^-fb
        // units; read by the final draw
        if (DENSE) {
            float h0, h1, l0, l1;
            unpack2(Ehi, h0, h1);
            unpack2(Elo, l0, l1);
            const long long e = to_fixed(h0, X.fb) + to_fixed(h1, X.fb) + to_fixed(l0, X.fb) + to_fixed(l1, X.fb) -
                                2 * to_fixed(2.0f, X.fb);
            const long long E = warp_sum_ll(e);
            if (lane == 0 && cvalid && cdraft)
                atomicAdd(reinterpret_cast<unsigned long long *>(&P.seq_E[cur]), static_cast<unsigned long long>(E));
            Ehi = E0;
            Elo = 0ull;
        }
    };

#pragma unroll 1
    for (int s = 0; s < kDrawStages - 1; ++s)
        issue(s);
#pragma unroll 1
    for (int64_t k = 0; k < nchunks; ++k) {
        issue(k + kDrawStages - 1);
        if (RING)
            cp_async_wait<kDrawStages - 1>();
        if (cb != cur) {
            if (cur >= 0)
                flush();
            __syncwarp();
            const StageInfo si = info[cst];
            const Verdict v = {si.jstar, si.m, si.s, si.x};
            cv = v;
            seq_rows<LT, DENSE>(P, cb, v, crow, cq);
            X = surv_args(P, v);
            cvalid = v.jstar >= 0;
            cdraft = v.jstar >= 0 && v.jstar < K;
            cvec = (reinterpret_cast<uintptr_t>(crow) & 15u) == 0 &&
                   (cq == nullptr || (reinterpret_cast<uintptr_t>(cq) & 15u) == 0);
            cur = cb;
        }
        const uint8_t *st = ring + cst * Shape::kChunkBytes;
        const int32_t g0 = ccis * kChunkGroups + lane;
        const bool full = (ccis + 1) * kChunkGroups <= ng; // every group of the chunk in the row
        long long A = 0;
        float Qs = 0.0f;
        auto fold_chunk = [&](auto kind) {
            constexpr int KIND = decltype(kind)::value;
            constexpr bool WQ = KIND == kFoldDense;
#pragma unroll
            for (int t = 0; t < kChunkTiles; ++t) {
                const int32_t g = g0 + 32 * t;
                const bool in = cvalid && (full || g < ng);
                float z[kGroup], q[kGroup];
                if (RING)
                    load_group_smem<LT, WQ>(st, 32 * t + lane, in, z, q);
                else
                    load_group_any<LT, WQ>(crow, cq, in ? g : ng, ng, V, cvec, z, q);
                fold_group<KIND, DENSE>(z, q, g * kGroup, X, Ehi, Elo, A, Qs);
            }
        };
        if (DENSE && cdraft)
            fold_chunk(std::integral_constant<int, kFoldDense>{});
        else if (!DENSE && cdraft) {
            // the rejected draft's id lies in one chunk of its row
            if (static_cast<unsigned>(X.x - ccis * kChunkGroups * kGroup) < static_cast<unsigned>(kChunkGroups * kGroup))
                fold_chunk(std::integral_constant<int, kFoldOneHot>{});
            else
                fold_chunk(std::integral_constant<int, kFoldOneHotNoX>{});
        }
        else
            fold_chunk(std::integral_constant<int, kFoldBonus>{});
        // the chunk's record
        const long long at = static_cast<long long>(warp_sum_u64(static_cast<unsigned long long>(A)));
        const float qt = DENSE ? warp_sum_f(Qs) : 0.0f;
        if (lane == 0) {
            P.rec_a[cb * CPS + ccis] = at;
            P.rec_q[cb * CPS + ccis] = qt;
        }
        ++ccount;
        cst = cst + 1 == kDrawStages ? 0 : cst + 1;
        if (++ccis == CPS) {
            ccis = 0;
            ++cb;
        }
    }
    if (RING)
        cp_async_wait<0>();
    flush();
    if (P.inline_final) {
        // the range held chunks of one sequence only: count them in
        // (release: this warp's records and normaliser share first); the warp
        // completing the count (acquire: everyone else's) makes the draw,
        // staging its chunk in the now idle ring
        uint32_t last = 0;
        if (lane == 0) {
            const uint32_t old = atom_add_acq_rel(&P.seq_cnt[cur], static_cast<uint32_t>(ccount));
            last = old + static_cast<uint32_t>(ccount) == static_cast<uint32_t>(CPS);
        }
        if (__shfl_sync(0xFFFFFFFFu, last, 0)) {
            __syncwarp();
            final_inline<LT, DENSE, RING>(P, cur, cv, lane, ring);
        }
    }
}

// The draw stream.  Each warp takes a contiguous range of the call's chunks
// (within one sequence when there are at least as many warps as sequences).
// Launched behind the row pass with programmatic dependent launch: it waits
// in griddepcontrol.wait until the row pass has completed.
template <typename LT, bool DENSE>
__global__ void __launch_bounds__(kDrawWarps * 32, SV_MIN_CTAS) survivor_kernel(const Params P)
{
    extern __shared__ __align__(128) uint8_t smem[]; // DrawShape::kWarpBytes per warp
    __shared__ StageInfo info[kDrawWarps][kDrawStages];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    uint8_t *ring = smem + warp * DrawShape<LT, DENSE>::kWarpBytes;
    pdl_wait_primary();
    const int64_t W = static_cast<int64_t>(blockIdx.x) * kDrawWarps + warp;
    const int64_t NW = static_cast<int64_t>(gridDim.x) * kDrawWarps;
    int64_t c0, c1;
    if (NW >= P.B) {
        // every sequence its own group of warps (sequence b: warps
        // [ceil(b NW / B), ceil((b+1) NW / B))), its chunks split evenly
        // among them: no warp meets a second sequence and its verdict
        const int64_t b = divi(W * P.B, NW);
        const int64_t w0 = divi(b * NW + P.B - 1, P.B), w1 = divi((b + 1) * NW + P.B - 1, P.B);
        const int64_t i = W - w0, n = w1 - w0;
        c0 = b * P.CPS + divi(i * P.CPS, n);
        c1 = b * P.CPS + divi((i + 1) * P.CPS, n);
    } else {
        c0 = divi(W * P.NC, NW);
        c1 = divi((W + 1) * P.NC, NW);
    }
    if (c0 < c1) {
        if (P.ring_ok)
            draw_range<LT, DENSE, true>(P, c0, c1, lane, ring, info[warp]);
        else
            draw_range<LT, DENSE, false>(P, c0, c1, lane, ring, info[warp]);
    }
    pdl_launch_dependents();
}

} // namespace sv
