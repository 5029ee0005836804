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

#include "sv_device.cuh"

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
// group totals.
template <int MODE>
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
        pt2[h] = mul2(pack2(ex2(y0), ex2(y1)), inv2);
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

// Re-formed warp tile (this lane's group g, already loaded): look for the id
// whose boundary (A - delta * Qp in 2^-fb units, measured from the chunk
// start; `run` = the tiles before) first exceeds `rem`, i.e. the first id
// whose running mass passes the draw.  Returns the id, or -1 with `run`
// advanced by the tile; `last_pos` tracks the last id of positive mass seen.
template <int MODE>
__device__ __forceinline__ int32_t scan_group(const float (&z)[kGroup], const float (&q)[kGroup], int32_t g,
                                              const SurvArgs &X, float delta, long long rem, long long &run,
                                              int32_t &last_pos, int lane)
{
    unsigned long long pt2[kGroup / 2];
    float w[kGroup], qp[kGroup], ws, qs;
    group_masses<MODE>(z, q, g * kGroup, X, pt2, w, qp, ws, qs);
    int kpos = -1;
#pragma unroll
    for (int k = 0; k < kGroup; ++k)
        if (w[k] > 0.0f)
            kpos = k;
    const long long Lv = to_fixed(ws, X.fb) - corr_of(delta, qs);
    const long long incl = warp_incl_scan_ll(Lv, lane) + run;
    const unsigned pos = __ballot_sync(0xFFFFFFFFu, kpos >= 0);
    if (pos) {
        const int hl = 31 - __clz(pos);
        const int kk = __shfl_sync(0xFFFFFFFFu, kpos, hl);
        last_pos = (g - lane + hl) * kGroup + kk;
    }
    const unsigned hit = __ballot_sync(0xFFFFFFFFu, incl > rem);
    int32_t tok = -1;
    if (hit) {
        const int l = __ffs(hit) - 1;
        if (lane == l) {
            const long long excl = incl - Lv;
            tok = g * kGroup + (kpos >= 0 ? kpos : 0);
            // the id within the group: running sums in id order (the group's
            // last boundary is its total, so an id past rounding falls back
            // to the last id of positive mass)
            float cw = 0.0f, cq = 0.0f;
#pragma unroll
            for (int k = 0; k < kGroup; ++k) {
                cw = __fadd_rn(cw, w[k]);
                cq = __fadd_rn(cq, qp[k]);
                if (w[k] > 0.0f && excl + to_fixed(cw, X.fb) - corr_of(delta, cq) > rem) {
                    tok = g * kGroup + k;
                    break;
                }
            }
        }
        tok = __shfl_sync(0xFFFFFFFFu, tok, l);
    }
    run = __shfl_sync(0xFFFFFFFFu, incl, 31);
    return tok;
}

// What the draw learns about a sequence once the rows are done.
struct SeqView {
    int32_t jstar; // -1: bad sequence
    float m, s;
    int32_t x;     // rejected one-hot draft, else -1
};

template <bool DENSE>
__device__ __forceinline__ SeqView load_seq(const Params &P, int64_t b, int lane)
{
    SeqView sv = {-1, 0.0f, 1.0f, -1};
    if (lane == 0) {
        sv.jstar = __ldcg(&P.seq_jstar[b]);
        sv.m = __ldcg(&P.seq_m[b]);
        sv.s = __ldcg(&P.seq_s[b]);
        if (!DENSE && sv.jstar >= 0 && sv.jstar < P.K)
            sv.x = __ldg(&P.tokens[b * P.K + sv.jstar]);
    }
    sv.jstar = __shfl_sync(0xFFFFFFFFu, sv.jstar, 0);
    sv.m = __shfl_sync(0xFFFFFFFFu, sv.m, 0);
    sv.s = __shfl_sync(0xFFFFFFFFu, sv.s, 0);
    sv.x = __shfl_sync(0xFFFFFFFFu, sv.x, 0);
    return sv;
}

// The surviving row of sequence b (and its draft row, dense and rejected).
template <typename LT, bool DENSE>
__device__ __forceinline__ void seq_rows(const Params &P, int64_t b, const SeqView &sv, const LT *&row,
                                         const float *&qrow)
{
    const int64_t V = P.V;
    row = static_cast<const LT *>(P.logits) + (b * (P.K + 1) + (sv.jstar < 0 ? 0 : sv.jstar)) * V;
    qrow = (DENSE && sv.jstar >= 0 && sv.jstar < P.K) ? P.q + (b * P.K + sv.jstar) * V : nullptr;
}

__device__ __forceinline__ SurvArgs surv_args(const Params &P, const SeqView &sv)
{
    SurvArgs X;
    X.c = P.c;
    X.mc = mc_of(sv.m, P.c);
    X.inv_s = __frcp_rn(sv.s);
    X.fb = P.fix_bits;
    X.x = sv.x;
    return X;
}

// The masses of one lane's group for a launch: MODE kModeDense (q = 0 for an
// accepted sequence) or kModeOneHot (x = -1 for an accepted sequence).
template <bool DENSE>
struct LaunchMode {
    static constexpr int value = DENSE ? kModeDense : kModeOneHot;
};

// Fold one group into the lane's running totals of its chunk (A, Qs) and
// sequence: E2 = (Ehi, Elo) packed pairs, an error-free (Fast2Sum) running
// sum of pt per id parity (dense); E2's first pair alone, a plain sum of pt
// (one-hot).
template <bool DENSE>
__device__ __forceinline__ void fold_group(const float (&z)[kGroup], const float (&q)[kGroup], int32_t e0,
                                           const SurvArgs &X, unsigned long long &Ehi, unsigned long long &Elo,
                                           long long &A, float &Qs)
{
    constexpr int MODE = LaunchMode<DENSE>::value;
    unsigned long long pt2[kGroup / 2];
    float w[kGroup], qp[kGroup], ws, qs;
    group_masses<MODE>(z, q, e0, X, pt2, w, qp, ws, qs);
    const unsigned long long m1 = pack2(-1.0f, -1.0f);
#pragma unroll
    for (int h = 0; h < kGroup / 2; ++h) {
        if (DENSE) { // |Ehi| >= 2 > every pt
            const unsigned long long s = add2(Ehi, pt2[h]);
            const unsigned long long tt = fma2(Ehi, m1, s);       // s - Ehi
            Elo = add2(Elo, fma2(tt, m1, pt2[h]));               // + (pt - tt)
            Ehi = s;
        } else {
            Ehi = add2(Ehi, pt2[h]);
        }
    }
    A += to_fixed(ws, X.fb);
    Qs = __fadd_rn(Qs, qs);
}

// Scan the 4 tiles of chunk `ch` of a row (one warp, direct loads) for the id
// whose boundary first exceeds `rem` (measured from the chunk start).  Falls
// back to the chunk's last id of positive mass if rounding leaves none.
// Copy chunk ch of a row into ring stage `st` in the fold's layout (group gl
// at gl * LB, its draft probabilities after the chunk's logits); lane l
// copies groups 4l .. 4l+3.  Rows of whole aligned groups go by async copy;
// others by plain loads (ids past the row as -inf, q as 0).  Returns when
// the lane's own data has landed (each lane reads only what it copied).
template <typename LT, bool DENSE>
__device__ void stage_chunk(uint8_t *st, const LT *row, const float *qrow, int32_t ch, int32_t V, bool ring_ok,
                            bool vec_ok, int lane)
{
    constexpr int LB = DrawShape<LT, DENSE>::LB;
    constexpr int GL = kChunkGroups / 32;
    const int32_t ng = (V + kGroup - 1) / kGroup;
#pragma unroll 1
    for (int i = 0; i < GL; ++i) {
        const int gl = lane * GL + i;
        const int32_t g = ch * kChunkGroups + gl;
        uint8_t *zs = st + gl * LB;
        uint8_t *qs = st + kChunkGroups * LB + gl * 32;
        if (ring_ok) {
            if (g < ng) {
                const uint8_t *src = reinterpret_cast<const uint8_t *>(row + static_cast<int64_t>(g) * kGroup);
                for (int h = 0; h < LB; h += 16)
                    cp_async16(zs + h, src + h);
                if (DENSE && qrow) {
                    const uint8_t *qsrc = reinterpret_cast<const uint8_t *>(qrow + static_cast<int64_t>(g) * kGroup);
                    cp_async16(qs, qsrc);
                    cp_async16(qs + 16, qsrc + 16);
                }
            }
        } else {
            float z[kGroup], q[kGroup];
            load_group_any<LT, DENSE>(row, qrow, g, ng, V, vec_ok, z, q);
            for (int k = 0; k < kGroup; ++k) {
                if constexpr (sizeof(LT) == 2)
                    reinterpret_cast<uint16_t *>(zs)[k] = static_cast<uint16_t>(__float_as_uint(z[k]) >> 16);
                else
                    reinterpret_cast<float *>(zs)[k] = z[k];
                if (DENSE)
                    reinterpret_cast<float *>(qs)[k] = q[k];
            }
        }
    }
    cp_async_commit();
    cp_async_wait<0>();
}

// Scan chunk ch (staged in `st`) for the id whose boundary (A - delta * Qp
// in 2^-fb units, from the chunk start) first exceeds `rem`.  Lane l re-forms
// groups 4l .. 4l+3 with the fold's per-group arithmetic (so the same group
// totals); one warp scan over the lanes' sums finds the lane, a walk over its
// groups the group, and running sums in id order the id.  Falls back to the
// chunk's last id of positive mass if rounding leaves none.  Rolled loops:
// this runs once per sequence, from a cold instruction cache.
template <typename LT, bool DENSE>
__device__ int32_t scan_chunk(const uint8_t *st, bool has_q, int32_t ch, int32_t V, const SurvArgs &X, float delta,
                              long long rem, int lane)
{
    constexpr int MODE = LaunchMode<DENSE>::value;
    constexpr int GL = kChunkGroups / 32;
    const int32_t ng = (V + kGroup - 1) / kGroup;
    const int32_t gbase = ch * kChunkGroups + lane * GL;
    auto group = [&](int i, float (&w)[kGroup], float (&qp)[kGroup]) {
        float z[kGroup], q[kGroup];
        load_group_smem<LT, DENSE>(st, lane * GL + i, gbase + i < ng, z, q);
        if (!has_q)
            for (int k = 0; k < kGroup; ++k)
                q[k] = 0.0f;
        unsigned long long pt2[kGroup / 2];
        float ws, qs;
        group_masses<MODE>(z, q, (gbase + i) * kGroup, X, pt2, w, qp, ws, qs);
        return to_fixed(ws, X.fb) - corr_of(delta, qs);
    };
    long long Ll = 0;
    int lastg = -1, lastk = -1;
#pragma unroll 1
    for (int i = 0; i < GL; ++i) {
        float w[kGroup], qp[kGroup];
        Ll += group(i, w, qp);
        for (int k = 0; k < kGroup; ++k)
            if (w[k] > 0.0f) {
                lastg = i;
                lastk = k;
            }
    }
    const long long incl = warp_incl_scan_ll(Ll, lane);
    const unsigned pos = __ballot_sync(0xFFFFFFFFu, lastg >= 0);
    int32_t last_pos = -1;
    if (pos) {
        const int hl = 31 - __clz(pos);
        const int lg = __shfl_sync(0xFFFFFFFFu, lastg, hl), lk = __shfl_sync(0xFFFFFFFFu, lastk, hl);
        last_pos = (ch * kChunkGroups + hl * GL + lg) * kGroup + lk;
    }
    const unsigned hit = __ballot_sync(0xFFFFFFFFu, incl > rem);
    if (!hit)
        return last_pos;
    const int l = __ffs(hit) - 1;
    int32_t tok = -1;
    if (lane == l) {
        long long excl = incl - Ll;
#pragma unroll 1
        for (int i = 0; i < GL && tok < 0; ++i) {
            float w[kGroup], qp[kGroup];
            const long long Lg = group(i, w, qp);
            if (excl + Lg > rem) {
                // running sums in id order (the group's last boundary is its
                // total, so an id past rounding falls back to its last id of
                // positive mass)
                float cw = 0.0f, cq = 0.0f;
                int kpos = -1;
                for (int k = 0; k < kGroup; ++k) {
                    cw = __fadd_rn(cw, w[k]);
                    cq = __fadd_rn(cq, qp[k]);
                    if (w[k] > 0.0f) {
                        kpos = k;
                        if (excl + to_fixed(cw, X.fb) - corr_of(delta, cq) > rem) {
                            tok = (gbase + i) * kGroup + k;
                            break;
                        }
                    }
                }
                if (tok < 0)
                    tok = (gbase + i) * kGroup + (kpos >= 0 ? kpos : 0);
            }
            excl += Lg;
        }
        if (tok < 0)
            tok = last_pos;
    }
    return __shfl_sync(0xFFFFFFFFu, tok, l);
}

// A sequence's chunk records in batches of kRecBatch: lane l holds records
// base + 8l .. base + 8l + 7 (raw A and Qp; 0 past the end).
constexpr int kRecLane = 8;
constexpr int kRecBatch = 32 * kRecLane;

__device__ __forceinline__ void load_recs(const long long *ra, const float *rq, int32_t base, int32_t n, int lane,
                                          long long (&a)[kRecLane], float (&q)[kRecLane])
{
#pragma unroll
    for (int i = 0; i < kRecLane; ++i) {
        const int32_t c = base + lane * kRecLane + i;
        a[i] = c < n ? __ldcg(ra + c) : 0;
        q[i] = c < n ? __ldcg(rq + c) : 0.0f;
    }
}

// A record's boundary mass max(0, A - delta * Qp) in 2^-fb units.
__device__ __forceinline__ long long rec_value(long long a, float q, float delta)
{
    const long long v = a - corr_of(delta, q);
    return v > 0 ? v : 0;
}

// The accepted-draft draw from p of a row, for a rejection whose residual
// came out with no mass (impossible in exact arithmetic): two passes over
// the whole row with direct loads (total, then the scan).
template <typename LT>
__device__ int32_t draw_from_p(const LT *row, int32_t V, bool vec_ok, SurvArgs X, float u, int lane)
{
    X.x = -1;
    const int32_t ng = (V + kGroup - 1) / kGroup;
    float q[kGroup];
#pragma unroll
    for (int k = 0; k < kGroup; ++k)
        q[k] = 0.0f;
    long long A = 0;
    for (int32_t g0 = 0; g0 < ng; g0 += 32) {
        float z[kGroup], qq[kGroup];
        load_group<LT, false>(row, nullptr, g0 + lane, ng, V, vec_ok, z, qq);
        unsigned long long pt2[kGroup / 2];
        float w[kGroup], qp[kGroup], ws, qs;
        group_masses<kModeBonus>(z, q, (g0 + lane) * kGroup, X, pt2, w, qp, ws, qs);
        A += to_fixed(ws, X.fb);
    }
    const long long t = mul_floor(u, warp_sum_ll(A));
    long long run = 0;
    int32_t last_pos = -1;
    for (int32_t g0 = 0; g0 < ng; g0 += 32) {
        float z[kGroup], qq[kGroup];
        load_group<LT, false>(row, nullptr, g0 + lane, ng, V, vec_ok, z, qq);
        const int32_t tok = scan_group<kModeBonus>(z, q, g0 + lane, X, 0.0f, t, run, last_pos, lane);
        if (tok >= 0)
            return tok;
    }
    return last_pos;
}

// Combine the chunk records of sequence b, draw the token, clear the
// scratch.  One warp: the one that completed the sequence's last chunk; `st`
// is a free stage of its ring.  Two rounds of loads in the common case
// (V <= 262144): the sequence's scalars with its records, then the chosen
// chunk.
template <typename LT, bool DENSE>
__device__ __noinline__ void final_draw(const Params &P, int64_t b, int lane, uint8_t *st)
{
    __threadfence();
    const int32_t K = P.K, V = P.V, CPS = P.CPS;
    long long *ra = P.rec_a + b * CPS;
    float *rq = P.rec_q + b * CPS;
    // ---- round 1: scalars and the first batch of records, all in flight
    long long a0[kRecLane];
    float q0[kRecLane];
    load_recs(ra, rq, 0, CPS, lane, a0, q0);
    const SeqView sv = load_seq<DENSE>(P, b, lane);
    const long long Eraw = __ldcg(&P.seq_E[b]), Fraw = __ldcg(&P.seq_F[b]);
    const float u = __ldg(&P.u[b * (K + 1) + K]);
    if (sv.jstar >= 0) {
        const LT *row;
        const float *qrow;
        seq_rows<LT, DENSE>(P, b, sv, row, qrow);
        const SurvArgs X = surv_args(P, sv);
        const bool rejected = sv.jstar < K;
        const bool vec_ok = (reinterpret_cast<uintptr_t>(row) & 15u) == 0 &&
                            (qrow == nullptr || (reinterpret_cast<uintptr_t>(qrow) & 15u) == 0);
        // dense: delta = E - 2^fb = (S' - 1) 2^fb, S' the exact sum of pt;
        // one-hot: F = sum of pt in 2^-fb units (the residual's normaliser)
        const long long E = rejected && DENSE ? Eraw : 0, F = rejected && !DENSE ? Fraw : 0;
        const float delta = rejected && DENSE ? static_cast<float>(E - (1ll << P.fix_bits)) : 0.0f;
        const int nb = (CPS + kRecBatch - 1) / kRecBatch;
        // ---- the total Z (the first batch's values kept for the search)
        long long v0[kRecLane], Z = 0;
        for (int bt = 0; bt < nb; ++bt) {
            long long a[kRecLane];
            float q[kRecLane];
            if (bt > 0)
                load_recs(ra, rq, bt * kRecBatch, CPS, lane, a, q);
            long long s = 0;
#pragma unroll
            for (int i = 0; i < kRecLane; ++i) {
                const long long v = bt == 0 ? rec_value(a0[i], q0[i], delta) : rec_value(a[i], q[i], delta);
                if (bt == 0)
                    v0[i] = v;
                s += v;
            }
            Z += warp_sum_ll(s);
        }
        int32_t tok = -1;
        const bool degenerate = rejected && !(Z > 0);
        if (degenerate) {
            tok = draw_from_p<LT>(row, V, vec_ok, X, u, lane);
        } else {
            // the first id whose running mass exceeds floor(u * Z): u * Z < P
            // iff floor(u * Z) < P for an integer P
            const long long t = mul_floor(u, Z);
            long long run = 0, rem = 0;
            int32_t sel = -1, lastc = -1;
            for (int bt = 0; bt < nb && sel < 0; ++bt) {
                long long v[kRecLane], L = 0;
                if (bt == 0) {
#pragma unroll
                    for (int i = 0; i < kRecLane; ++i)
                        v[i] = v0[i];
                } else {
                    long long a[kRecLane];
                    float q[kRecLane];
                    load_recs(ra, rq, bt * kRecBatch, CPS, lane, a, q);
#pragma unroll
                    for (int i = 0; i < kRecLane; ++i)
                        v[i] = rec_value(a[i], q[i], delta);
                }
                int lp = -1;
#pragma unroll
                for (int i = 0; i < kRecLane; ++i) {
                    L += v[i];
                    if (v[i] > 0)
                        lp = i;
                }
                const long long incl = warp_incl_scan_ll(L, lane) + run;
                const unsigned pos = __ballot_sync(0xFFFFFFFFu, lp >= 0);
                if (pos) {
                    const int hl = 31 - __clz(pos);
                    lastc = bt * kRecBatch + hl * kRecLane + __shfl_sync(0xFFFFFFFFu, lp, hl);
                }
                const unsigned hit = __ballot_sync(0xFFFFFFFFu, incl > t);
                if (hit) {
                    const int l = __ffs(hit) - 1;
                    int32_t c = -1;
                    long long before = 0;
                    if (lane == l) {
                        long long acc = incl - L;
                        for (int i = 0; i < kRecLane; ++i) {
                            if (v[i] > 0 && acc + v[i] > t) {
                                c = bt * kRecBatch + lane * kRecLane + i;
                                before = acc;
                                break;
                            }
                            acc += v[i];
                        }
                        if (c < 0) { // not reached with exact integer sums
                            c = bt * kRecBatch + lane * kRecLane + (lp >= 0 ? lp : 0);
                            before = t;
                        }
                    }
                    sel = __shfl_sync(0xFFFFFFFFu, c, l);
                    rem = t - __shfl_sync(0xFFFFFFFFu, before, l);
                }
                run = __shfl_sync(0xFFFFFFFFu, incl, 31);
            }
            if (sel < 0) { // rounding put the draw past the last chunk: take its last id
                sel = lastc;
                rem = LLONG_MAX;
            }
            if (sel >= 0) {
                stage_chunk<LT, DENSE>(st, row, qrow, sel, V, P.ring_ok != 0, vec_ok, lane);
                tok = scan_chunk<LT, DENSE>(st, qrow != nullptr, sel, V, X, delta, rem, lane);
            }
        }
        if (lane == 0) {
            P.out_tokens[b * (K + 1) + sv.jstar] = tok;
            if (P.residual_mass) {
                // Z / 2^fb over the residual's normaliser (S' or F / 2^fb)
                const long long norm = DENSE ? E : F;
                P.residual_mass[b] = (rejected && !degenerate && norm > 0)
                                         ? __fdiv_rn(static_cast<float>(Z), static_cast<float>(norm))
                                         : 0.0f;
            }
            if (degenerate && P.status)
                atomicOr(P.status, kDegenerate);
        }
    }
    // every chunk of the sequence is done: return its scratch to zero
    for (int32_t i = lane; i < CPS; i += 32) {
        ra[i] = 0;
        rq[i] = 0.0f;
    }
    if (lane == 0) {
        P.surv_cnt[b] = 0u;
        P.seq_E[b] = 0;
        P.seq_F[b] = 0;
        P.seq_jstar[b] = 0;
        P.seq_m[b] = 0.0f;
        P.seq_s[b] = 0.0f;
    }
}

// The chunks [c0, c1) of one warp.  RING: rows of whole, 16-byte aligned
// groups stream through the warp's ring, kDrawStages - 1 chunks ahead, a
// lane copying (and later reading) its own 4 groups of each chunk; otherwise
// each lane loads its groups directly.
template <typename LT, bool DENSE, bool RING>
__device__ __forceinline__ void draw_range(const Params &P, int64_t c0, int64_t c1, int lane, uint8_t *ring)
{
    using Shape = DrawShape<LT, DENSE>;
    constexpr int LB = Shape::LB;
    const int32_t V = P.V, CPS = P.CPS;
    const int32_t ng = (V + kGroup - 1) / kGroup;
    const int64_t nchunks = c1 - c0;

    // ---- issue side (RING): the chunk kDrawStages - 1 ahead of the consumer
    int64_t ib = c0 / CPS;
    int32_t icis = static_cast<int32_t>(c0 - ib * CPS);
    int ist = 0;       // ring stage of the next issued chunk
    int64_t iseq = -1; // sequence whose rows irow / iq point into
    const LT *irow = nullptr;
    const float *iq = nullptr;
    bool ivalid = false;
    auto issue = [&](int64_t k) {
        if (RING && k < nchunks) {
            if (ib != iseq) {
                const SeqView sv = load_seq<DENSE>(P, ib, lane);
                seq_rows<LT, DENSE>(P, ib, sv, irow, iq);
                ivalid = sv.jstar >= 0;
                iseq = ib;
            }
            if (ivalid) {
                uint8_t *st = ring + ist * Shape::kChunkBytes;
                const int32_t g0 = icis * kChunkGroups + lane;
                const uint8_t *src = reinterpret_cast<const uint8_t *>(irow + static_cast<int64_t>(g0) * kGroup);
                const uint8_t *qsrc =
                    DENSE && iq ? reinterpret_cast<const uint8_t *>(iq + static_cast<int64_t>(g0) * kGroup) : nullptr;
#pragma unroll
                for (int t = 0; t < kChunkTiles; ++t) {
                    if (g0 + 32 * t < ng) {
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
    int64_t cb = c0 / CPS;
    int32_t ccis = static_cast<int32_t>(c0 - cb * CPS);
    int cst = 0;      // ring stage of chunk k
    int64_t cur = -1; // sequence whose totals are being accumulated
    SurvArgs X = {};
    bool cvalid = false, cdraft = false, cvec = false;
    const LT *crow = nullptr;
    const float *cq = nullptr;
    const unsigned long long E0 = DENSE ? pack2(2.0f, 2.0f) : 0ull;
    unsigned long long Ehi = E0, Elo = 0ull; // see fold_group
    int32_t nch = 0; // chunks of `cur` done
    auto flush = [&](uint8_t *free_stage) {
        // the sequence's normaliser share and its chunk count; the warp that
        // completes the sequence draws its token
        float h0, h1, l0, l1;
        unpack2(Ehi, h0, h1);
        unpack2(Elo, l0, l1);
        long long e = to_fixed(h0, X.fb) + to_fixed(h1, X.fb);
        if (DENSE)
            e += to_fixed(l0, X.fb) + to_fixed(l1, X.fb) - 2 * to_fixed(2.0f, X.fb);
        const long long E = warp_sum_ll(e);
        int last = 0;
        if (lane == 0) {
            if (cvalid && cdraft) {
                if (DENSE)
                    atomicAdd(reinterpret_cast<unsigned long long *>(&P.seq_E[cur]), static_cast<unsigned long long>(E));
                else
                    atomicAdd(reinterpret_cast<unsigned long long *>(&P.seq_F[cur]), static_cast<unsigned long long>(E));
            }
            __threadfence();
            last = atomicAdd(&P.surv_cnt[cur], static_cast<unsigned>(nch)) + static_cast<unsigned>(nch) ==
                   static_cast<unsigned>(CPS);
        }
        last = __shfl_sync(0xFFFFFFFFu, last, 0);
        if (last)
            final_draw<LT, DENSE>(P, cur, lane, free_stage);
        Ehi = E0;
        Elo = 0ull;
        nch = 0;
    };

#pragma unroll 1
    for (int s = 0; s < kDrawStages - 1; ++s)
        issue(s);
#pragma unroll 1
    for (int64_t k = 0; k < nchunks; ++k) {
        // a new sequence: close the last one while the stage about to take
        // chunk k + kDrawStages - 1 (chunk k - 1's) is still free
        if (cb != cur && cur >= 0)
            flush(ring + (cst + kDrawStages - 1) % kDrawStages * Shape::kChunkBytes);
        issue(k + kDrawStages - 1);
        if (RING)
            cp_async_wait<kDrawStages - 1>();
        if (cb != cur) {
            const SeqView sv = load_seq<DENSE>(P, cb, lane);
            seq_rows<LT, DENSE>(P, cb, sv, crow, cq);
            X = surv_args(P, sv);
            cvalid = sv.jstar >= 0;
            cdraft = sv.jstar >= 0 && sv.jstar < P.K;
            cvec = (reinterpret_cast<uintptr_t>(crow) & 15u) == 0 &&
                   (cq == nullptr || (reinterpret_cast<uintptr_t>(cq) & 15u) == 0);
            cur = cb;
        }
        const uint8_t *st = ring + cst * Shape::kChunkBytes;
        const int32_t g0 = ccis * kChunkGroups + lane;
        long long A = 0;
        float Qs = 0.0f;
#pragma unroll
        for (int t = 0; t < kChunkTiles; ++t) {
            const int32_t g = g0 + 32 * t;
            const bool in = cvalid && g < ng;
            float z[kGroup], q[kGroup];
            if (RING)
                load_group_smem<LT, DENSE>(st, 32 * t + lane, in, z, q);
            else
                load_group_any<LT, DENSE>(crow, cq, in ? g : ng, ng, V, cvec, z, q);
            if (DENSE && cq == nullptr) {
#pragma unroll
                for (int j = 0; j < kGroup; ++j)
                    q[j] = 0.0f;
            }
            fold_group<DENSE>(z, q, g * kGroup, X, Ehi, Elo, A, Qs);
        }
        // the chunk's record
        const long long at = warp_sum_ll(A);
        const float qt = DENSE ? warp_sum_f(Qs) : 0.0f;
        if (lane == 0) {
            P.rec_a[cb * CPS + ccis] = at;
            P.rec_q[cb * CPS + ccis] = qt;
        }
        ++nch;
        cst = cst + 1 == kDrawStages ? 0 : cst + 1;
        if (++ccis == CPS) {
            ccis = 0;
            ++cb;
        }
    }
    cp_async_wait<0>();
    flush(ring);
}

// The final draws.  Each warp takes a contiguous range of the call's chunks;
// the warp that completes a sequence's last chunk draws its token.  Launched
// behind the row pass with programmatic dependent launch: it waits in
// griddepcontrol.wait until the row pass has completed.
template <typename LT, bool DENSE>
__global__ void __launch_bounds__(kDrawWarps * 32, SV_MIN_CTAS) survivor_kernel(const Params P)
{
    extern __shared__ __align__(128) uint8_t smem[]; // DrawShape::kWarpBytes per warp
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    uint8_t *ring = smem + warp * DrawShape<LT, DENSE>::kWarpBytes;
    pdl_wait_primary();
    const int64_t W = static_cast<int64_t>(blockIdx.x) * kDrawWarps + warp;
    const int64_t NW = static_cast<int64_t>(gridDim.x) * kDrawWarps;
    const int64_t c0 = W * P.NC / NW, c1 = (W + 1) * P.NC / NW;
    if (c0 >= c1)
        return;
    if (P.ring_ok)
        draw_range<LT, DENSE, true>(P, c0, c1, lane, ring);
    else
        draw_range<LT, DENSE, false>(P, c0, c1, lane, ring);
}

} // namespace sv
