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
// The surviving row is cut into slices of 2048 ids, one warp each, streamed
// through the warp's async-copy ring.  A lane owns groups of 8 consecutive
// ids; a warp tile is 32 groups.  Per element:
//   e_i  = exp2(z_i * c - fl(m * c))          (m: the row maximum)
//   pt_i = e_i / s~                           (s~: the row pass's fp32 normaliser)
//   w_i  = max(0, pt_i - q_i) | pt_i | pt_i with x removed
// The 8 masses of a group are added in fp32 in id order and the group total
// is held as an integer multiple of 2^-fix_bits, so every sum over groups,
// tiles and slices is exact and order-independent; the draw re-forms groups
// with the same arithmetic, so its boundaries agree with the totals.
//
// The dense residual needs the exact normaliser, not s~: with
// S' = sum_i pt_i (accumulated error-free per element, Fast2Sum), the true
// residual is proportional to pt_i - S' q_i = w_i - (S' - 1) q_i on the ids
// where it is positive.  So each slice also carries Qp = sum of q_i over the
// ids with w_i > 0, and every boundary is taken as A - (S' - 1) * Qp.  (Ids
// within |S' - 1| q_i of the kink move by less than one fp32 ulp of their own
// mass.)  Each slice publishes its totals and one record per warp tile; the
// normalisers are integer sums, added atomically.  The warp that completes a
// sequence's last slice combines the slice totals, finds the slice, the warp
// tile and the id that hold u_K * Z, and clears the sequence's scratch.
#pragma once

#include "sv_device.cuh"

namespace sv {

enum { kModeBonus = 0, kModeDense = 1, kModeOneHot = 2 };

struct SurvArgs {
    float c, mc;   // log2(e)/T and fl(m*c) of the surviving row
    float inv_s;   // 1 / s~
    float scale;   // 2^fix_bits
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

// z (and q) of this lane's group from a ring stage: logits at lane * LB,
// q after the 32 lanes' logits.
template <typename LT, bool WANT_Q>
__device__ __forceinline__ void load_group_smem(const uint8_t *st, int lane, bool in, float (&z)[kGroup],
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
        const uint4 w = lds_v4(st + lane * LB);
        z[0] = bf16_lo(w.x); z[1] = bf16_hi(w.x);
        z[2] = bf16_lo(w.y); z[3] = bf16_hi(w.y);
        z[4] = bf16_lo(w.z); z[5] = bf16_hi(w.z);
        z[6] = bf16_lo(w.w); z[7] = bf16_hi(w.w);
    } else {
        const uint4 a = lds_v4(st + lane * LB), b = lds_v4(st + lane * LB + 16);
        z[0] = __uint_as_float(a.x); z[1] = __uint_as_float(a.y);
        z[2] = __uint_as_float(a.z); z[3] = __uint_as_float(a.w);
        z[4] = __uint_as_float(b.x); z[5] = __uint_as_float(b.y);
        z[6] = __uint_as_float(b.z); z[7] = __uint_as_float(b.w);
    }
    if constexpr (WANT_Q) {
        const uint8_t *qs = st + 32 * LB + lane * 32;
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

// The masses of one group, in id order.  pt: e_i / s~; w: the mass the draw
// uses; qp: q_i where w > 0 (dense), else 0.  The same code forms the slice
// totals and the final scan, so both see identical values.
template <int MODE>
__device__ __forceinline__ void group_masses(const float (&z)[kGroup], const float (&q)[kGroup], int32_t e0,
                                             const SurvArgs &X, float (&pt)[kGroup], float (&w)[kGroup],
                                             float (&qp)[kGroup])
{
#pragma unroll
    for (int k = 0; k < kGroup; ++k) {
        pt[k] = __fmul_rn(term(z[k], X.c, X.mc), X.inv_s);
        if (MODE == kModeDense) {
            const float d = __fsub_rn(pt[k], q[k]);
            w[k] = fmaxf(d, 0.0f);
            qp[k] = d > 0.0f ? q[k] : 0.0f;
        } else if (MODE == kModeOneHot) {
            w[k] = (e0 + k == X.x) ? 0.0f : pt[k];
            qp[k] = 0.0f;
        } else {
            w[k] = pt[k];
            qp[k] = 0.0f;
        }
    }
}

// Totals of one slice (lane-uniform after the warp reductions).
struct SliceTotals {
    long long A;   // sum of group masses, units of 2^-fix_bits (exact)
    long long E;   // sum of pt, units of 2^-fix_bits, error-free (dense)
    double Qp;     // sum over the slice's tiles of the tile's fp32 Qp (dense)
    double Ef;     // sum of pt, fp32 per lane then 2^-fix_bits units (one-hot)
};

// Fold the masses of this lane's group of one warp tile into the totals and
// record the tile's own totals (rec_a / rec_q, written by lane 0).
template <int MODE>
__device__ __forceinline__ void fold_group(const float (&z)[kGroup], const float (&q)[kGroup], int32_t e0,
                                           const SurvArgs &X, float &Ehi, float &Elo, float &Ef, long long &A,
                                           double &Q, long long *rec_a, float *rec_q, int lane)
{
    float pt[kGroup], w[kGroup], qp[kGroup];
    group_masses<MODE>(z, q, e0, X, pt, w, qp);
    float ws = 0.0f, qs = 0.0f;
#pragma unroll
    for (int k = 0; k < kGroup; ++k) {
        ws = __fadd_rn(ws, w[k]);
        qs = __fadd_rn(qs, qp[k]);
        if (MODE == kModeDense) { // error-free running sum of pt
            const float s = __fadd_rn(Ehi, pt[k]);
            const float tt = __fsub_rn(s, Ehi);
            Elo = __fadd_rn(Elo, __fsub_rn(pt[k], tt));
            Ehi = s;
        } else if (MODE == kModeOneHot) {
            Ef = __fadd_rn(Ef, pt[k]);
        }
    }
    const long long at = warp_sum_ll(to_fixed(ws, X.scale));
    const float qt = MODE == kModeDense ? warp_sum_f(qs) : 0.0f;
    if (lane == 0) {
        *rec_a = at;
        *rec_q = qt;
    }
    A += at;
    Q += static_cast<double>(qt);
}

// One slice: groups [gs, ge) of the row; warp tile t = groups gs + 32t + lane.
// With `use_ring` (16-byte aligned rows of whole groups) the tiles stream
// through the warp's async-copy ring, three tiles ahead; otherwise each
// lane loads its group directly.
template <typename LT, int MODE>
__device__ __forceinline__ SliceTotals slice_totals(const LT *row, const float *qrow, int32_t gs, int32_t ge,
                                                    int32_t V, bool vec_ok, bool use_ring, const SurvArgs &X,
                                                    int lane, uint8_t *ring, long long *rec_a, float *rec_q)
{
    constexpr bool WQ = MODE == kModeDense;
    constexpr int LB = kGroup * sizeof(LT);
    float Ehi = 2.0f, Elo = 0.0f, Ef = 0.0f; // Fast2Sum pair: |Ehi| >= 2 > every pt
    long long A = 0;
    double Q = 0.0;
    const int ntiles = (ge - gs + 31) / 32;
    if (use_ring) {
        auto issue = [&](int t) {
            const int32_t g = gs + 32 * t + lane;
            if (t < ntiles && g < ge) {
                uint8_t *st = ring + (t % kStages) * kStageBytes;
                const uint8_t *src = reinterpret_cast<const uint8_t *>(row + static_cast<int64_t>(g) * kGroup);
#pragma unroll
                for (int h = 0; h < LB; h += 16)
                    cp_async16(st + lane * LB + h, src + h);
                if (WQ) {
                    const uint8_t *qsrc = reinterpret_cast<const uint8_t *>(qrow + static_cast<int64_t>(g) * kGroup);
                    cp_async16(st + 32 * LB + lane * 32, qsrc);
                    cp_async16(st + 32 * LB + lane * 32 + 16, qsrc + 16);
                }
            }
            cp_async_commit();
        };
#pragma unroll
        for (int t = 0; t < kStages - 1; ++t)
            issue(t);
        for (int t = 0; t < ntiles; ++t) {
            issue(t + kStages - 1);
            cp_async_wait<kStages - 1>();
            const int32_t g = gs + 32 * t + lane;
            float z[kGroup], q[kGroup];
            load_group_smem<LT, WQ>(ring + (t % kStages) * kStageBytes, lane, g < ge, z, q);
            fold_group<MODE>(z, q, g * kGroup, X, Ehi, Elo, Ef, A, Q, rec_a + t, rec_q + t, lane);
        }
    } else {
        for (int t = 0; t < ntiles; ++t) {
            const int32_t g = gs + 32 * t + lane;
            float z[kGroup], q[kGroup];
            load_group<LT, WQ>(row, qrow, g, ge, V, vec_ok, z, q);
            fold_group<MODE>(z, q, g * kGroup, X, Ehi, Elo, Ef, A, Q, rec_a + t, rec_q + t, lane);
        }
    }
    SliceTotals T;
    T.A = A;
    T.Qp = Q;
    T.E = MODE == kModeDense
              ? warp_sum_ll(to_fixed(Ehi, X.scale) - to_fixed(2.0f, X.scale) + to_fixed(Elo, X.scale))
              : 0;
    T.Ef = MODE == kModeOneHot ? static_cast<double>(warp_sum_ll(to_fixed(Ef, X.scale))) : 0.0;
    return T;
}

template <typename LT, bool DENSE>
__device__ __forceinline__ SliceTotals slice_totals_mode(int mode, const LT *row, const float *qrow, int32_t gs,
                                                         int32_t ge, int32_t V, bool vec_ok, bool use_ring,
                                                         const SurvArgs &X, int lane, uint8_t *ring,
                                                         long long *rec_a, float *rec_q)
{
    // a dense-q launch meets the dense residual and the extra token, a
    // one-hot launch the one-hot residual and the extra token
    if (DENSE && mode == kModeDense)
        return slice_totals<LT, kModeDense>(row, qrow, gs, ge, V, vec_ok, use_ring, X, lane, ring, rec_a, rec_q);
    if (!DENSE && mode == kModeOneHot)
        return slice_totals<LT, kModeOneHot>(row, qrow, gs, ge, V, vec_ok, use_ring, X, lane, ring, rec_a, rec_q);
    return slice_totals<LT, kModeBonus>(row, qrow, gs, ge, V, vec_ok, use_ring, X, lane, ring, rec_a, rec_q);
}

// Re-formed warp tile (this lane's group g, already loaded): look for the id
// whose boundary (A - dfix * Qp, measured from the slice start; `run` = the
// tiles before) first exceeds `rem`.  Returns the id, or -1 with `run`
// advanced by the tile; `last_pos` tracks the last id of positive mass seen.
template <int MODE>
__device__ __forceinline__ int32_t scan_group(const float (&z)[kGroup], const float (&q)[kGroup], int32_t g,
                                              const SurvArgs &X, double dfix, double rem, double &run,
                                              int32_t &last_pos, int lane)
{
    float pt[kGroup], w[kGroup], qp[kGroup];
    group_masses<MODE>(z, q, g * kGroup, X, pt, w, qp);
    float cw[kGroup], cq[kGroup];
    float ws = 0.0f, qs = 0.0f;
    int kpos = -1;
#pragma unroll
    for (int k = 0; k < kGroup; ++k) {
        ws = __fadd_rn(ws, w[k]);
        qs = __fadd_rn(qs, qp[k]);
        cw[k] = ws;
        cq[k] = qs;
        if (w[k] > 0.0f)
            kpos = k;
    }
    const double Lv = static_cast<double>(to_fixed(ws, X.scale)) - dfix * static_cast<double>(qs);
    const double incl = warp_incl_scan_d(Lv, lane) + run;
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
            const double excl = incl - Lv;
            tok = g * kGroup + (kpos >= 0 ? kpos : 0);
#pragma unroll
            for (int k = 0; k < kGroup; ++k) {
                const double v = static_cast<double>(to_fixed(cw[k], X.scale)) - dfix * static_cast<double>(cq[k]);
                if (excl + v > rem) {
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

// Re-form warp tile [g0, ...) of the row (one warp) and find the id holding
// `rem` (measured from the tile start).  Falls back to the tile's last id of
// positive mass if rounding leaves none.
template <typename LT, int MODE>
__device__ __forceinline__ int32_t scan_tile(const LT *row, const float *qrow, int32_t g0, int32_t ge, int32_t V,
                                             bool vec_ok, const SurvArgs &X, double dfix, double rem, int lane)
{
    constexpr bool WQ = MODE == kModeDense;
    float z[kGroup], q[kGroup];
    load_group<LT, WQ>(row, qrow, g0 + lane, ge, V, vec_ok, z, q);
    double run = 0.0;
    int32_t last_pos = -1;
    const int32_t tok = scan_group<MODE>(z, q, g0 + lane, X, dfix, rem, run, last_pos, lane);
    return tok >= 0 ? tok : last_pos;
}

template <typename LT, bool DENSE>
__device__ __forceinline__ int32_t scan_tile_mode(int mode, const LT *row, const float *qrow, int32_t g0,
                                                  int32_t ge, int32_t V, bool vec_ok, const SurvArgs &X,
                                                  double dfix, double rem, int lane)
{
    if (DENSE && mode == kModeDense)
        return scan_tile<LT, kModeDense>(row, qrow, g0, ge, V, vec_ok, X, dfix, rem, lane);
    if (!DENSE && mode == kModeOneHot)
        return scan_tile<LT, kModeOneHot>(row, qrow, g0, ge, V, vec_ok, X, dfix, rem, lane);
    return scan_tile<LT, kModeBonus>(row, qrow, g0, ge, V, vec_ok, X, dfix, rem, lane);
}

// Inclusive scan of `v` over `n` entries (lane-strided chunks of 32): the
// first index whose running sum exceeds `t`, with the sum before it.
// Returns -1 (and the total in *before) if none does; `last` receives the
// last index with v > 0.
template <typename F>
__device__ __forceinline__ int32_t find_first_over(int32_t n, double t, F value, double *before, int32_t *last,
                                                   int lane)
{
    double run = 0.0;
    int32_t lastp = -1;
    for (int32_t s0 = 0; s0 < n; s0 += 32) {
        const int32_t s = s0 + lane;
        const double v = s < n ? value(s) : 0.0;
        const double incl = warp_incl_scan_d(v, lane) + run;
        const unsigned pos = __ballot_sync(0xFFFFFFFFu, v > 0.0);
        if (pos)
            lastp = s0 + 31 - __clz(pos);
        const unsigned hit = __ballot_sync(0xFFFFFFFFu, s < n && incl > t);
        if (hit) {
            const int l = __ffs(hit) - 1;
            *before = __shfl_sync(0xFFFFFFFFu, incl, l) - __shfl_sync(0xFFFFFFFFu, v, l);
            *last = lastp;
            return s0 + l;
        }
        run = __shfl_sync(0xFFFFFFFFu, incl, 31);
    }
    *before = run;
    *last = lastp;
    return -1;
}

// What a slice item learns about its sequence once the rows are done.
struct SeqView {
    int32_t jstar; // -1: bad sequence (or a wait that ran out)
    float m, s;
    int32_t x;     // rejected one-hot draft
};

template <typename LT, bool DENSE>
__device__ __forceinline__ void seq_setup(const Params &P, int64_t b, const SeqView &sv, SurvArgs &X, int &mode,
                                          const LT *&row, const float *&qrow, bool &vec_ok, bool &use_ring)
{
    const int32_t K = P.K, V = P.V;
    const bool rejected = sv.jstar < K;
    row = static_cast<const LT *>(P.logits) + (b * (K + 1) + sv.jstar) * static_cast<int64_t>(V);
    qrow = (DENSE && rejected) ? P.q + (b * K + sv.jstar) * static_cast<int64_t>(V) : nullptr;
    X.c = P.c;
    X.mc = mc_of(sv.m, P.c);
    X.inv_s = __frcp_rn(sv.s);
    X.scale = __int_as_float((127 + P.fix_bits) << 23);
    X.x = sv.x;
    mode = !rejected ? kModeBonus : (DENSE ? kModeDense : kModeOneHot);
    vec_ok = (reinterpret_cast<uintptr_t>(row) & 15u) == 0 &&
             (qrow == nullptr || (reinterpret_cast<uintptr_t>(qrow) & 15u) == 0);
    use_ring = vec_ok && (V % kGroup) == 0; // whole, aligned groups only
}

// Combine the slice totals of sequence b, draw the token, clear the scratch.
// One warp: the one that completed the last slice.  Three dependent rounds
// of loads: slice totals, the chosen slice's tile records, the chosen tile.
template <typename LT, bool DENSE>
__device__ void final_draw(const Params &P, int64_t b, const SeqView &sv, int lane, uint8_t *ring)
{
    __threadfence();
    const int32_t K = P.K, V = P.V, NSL = P.NSL;
    long long *tot = P.slice_tot + b * NSL * 2;
    long long *ra = P.rec_a + b * NSL * kSliceTiles;
    float *rq = P.rec_q + b * NSL * kSliceTiles;
    if (sv.jstar >= 0) {
        SurvArgs X;
        int mode;
        const LT *row;
        const float *qrow;
        bool vec_ok, use_ring;
        seq_setup<LT, DENSE>(P, b, sv, X, mode, row, qrow, vec_ok, use_ring);
        const bool rejected = sv.jstar < K;
        const int32_t ngroups = (V + kGroup - 1) / kGroup;
        const double two_fb = ldexp(1.0, P.fix_bits);
        bool degenerate = false;
        double d = 0.0, Z = 0.0, norm = 0.0;
        for (int attempt = 0; attempt < 2; ++attempt) {
            const double Sp = static_cast<double>(__ldcg(&P.seq_E[b])) / two_fb; // exact sum of pt
            d = mode == kModeDense ? (Sp - 1.0) * two_fb : 0.0;
            norm = mode == kModeDense ? Sp
                                      : (mode == kModeOneHot ? static_cast<double>(__ldcg(&P.seq_F[b])) / two_fb
                                                             : 0.0);
            double before;
            int32_t lastz;
            (void)find_first_over(NSL, INFINITY, [&](int32_t s) {
                return fmax(0.0, static_cast<double>(__ldcg(&tot[2 * s])) -
                                     d * __longlong_as_double(__ldcg(&tot[2 * s + 1])));
            }, &before, &lastz, lane);
            Z = before;
            if (!(mode != kModeBonus && !(Z > 0.0)))
                break;
            // residual of zero mass after a rejection (impossible in exact
            // arithmetic): draw from p of the same row instead
            mode = kModeBonus;
            degenerate = true;
            for (int32_t s = 0; s < NSL; ++s) {
                const SliceTotals T = slice_totals<LT, kModeBonus>(
                    row, qrow, s * kSliceGroups, min(ngroups, (s + 1) * kSliceGroups), V, vec_ok, use_ring, X, lane,
                    ring, ra + s * kSliceTiles, rq + s * kSliceTiles);
                if (lane == 0) {
                    tot[2 * s] = T.A;
                    tot[2 * s + 1] = __double_as_longlong(0.0);
                }
            }
            __syncwarp();
            __threadfence();
        }
        const double t = static_cast<double>(__ldg(&P.u[b * (K + 1) + K])) * Z;

        // ---- the slice, then the warp tile, holding the draw
        double before = 0.0;
        int32_t last_s = -1;
        int32_t sel = find_first_over(NSL, t, [&](int32_t s) {
            return fmax(0.0, static_cast<double>(__ldcg(&tot[2 * s])) -
                                 d * __longlong_as_double(__ldcg(&tot[2 * s + 1])));
        }, &before, &last_s, lane);
        double rem = t - before;
        if (sel < 0) { // rounding put the draw past the last slice: take its last id
            sel = last_s;
            rem = INFINITY;
        }
        int32_t tok = -1;
        if (sel >= 0) {
            const int32_t gs = sel * kSliceGroups, ge = min(ngroups, gs + kSliceGroups);
            const int32_t ntiles = (ge - gs + 31) / 32;
            double tb = 0.0;
            int32_t last_t = -1;
            int32_t tsel = find_first_over(ntiles, rem, [&](int32_t tt) {
                return static_cast<double>(__ldcg(&ra[sel * kSliceTiles + tt])) -
                       d * static_cast<double>(__ldcg(&rq[sel * kSliceTiles + tt]));
            }, &tb, &last_t, lane);
            double rem2 = rem - tb;
            if (tsel < 0) {
                tsel = last_t >= 0 ? last_t : ntiles - 1;
                rem2 = INFINITY;
            }
            tok = scan_tile_mode<LT, DENSE>(mode, row, qrow, gs + 32 * tsel, ge, V, vec_ok, X, d, rem2, lane);
        }
        if (lane == 0) {
            P.out_tokens[b * (K + 1) + sv.jstar] = tok;
            if (P.residual_mass)
                P.residual_mass[b] = (rejected && !degenerate && norm > 0.0)
                                         ? static_cast<float>(Z / two_fb / norm)
                                         : 0.0f;
            if (degenerate && P.status)
                atomicOr(P.status, kDegenerate);
        }
    }
    // every slice of the sequence is done: return its scratch to zero
    for (int32_t i = lane; i < NSL * 2; i += 32)
        tot[i] = 0;
    for (int32_t i = lane; i < NSL * kSliceTiles; i += 32) {
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

// One slice ticket (a warp): ticket t is slice t % NSL of sequence t / NSL.
template <typename LT, bool DENSE>
__device__ void slice_item(const Params &P, unsigned long long ticket, int lane, uint8_t *ring)
{
    const int32_t K = P.K, V = P.V, NSL = P.NSL;
    const int64_t b = divi(static_cast<int64_t>(ticket), NSL);
    const int32_t slice = static_cast<int32_t>(static_cast<int64_t>(ticket) - b * NSL);
    SeqView sv = {-1, 0.0f, 1.0f, -1};
    if (lane == 0) {
        sv.jstar = __ldcg(&P.seq_jstar[b]);
        sv.m = __ldcg(&P.seq_m[b]);
        sv.s = __ldcg(&P.seq_s[b]);
        if (!DENSE && sv.jstar >= 0 && sv.jstar < K)
            sv.x = __ldg(&P.tokens[b * K + sv.jstar]);
    }
    sv.jstar = __shfl_sync(0xFFFFFFFFu, sv.jstar, 0);
    sv.m = __shfl_sync(0xFFFFFFFFu, sv.m, 0);
    sv.s = __shfl_sync(0xFFFFFFFFu, sv.s, 0);
    sv.x = __shfl_sync(0xFFFFFFFFu, sv.x, 0);

    if (sv.jstar >= 0) {
        SurvArgs X;
        int mode;
        const LT *row;
        const float *qrow;
        bool vec_ok, use_ring;
        seq_setup<LT, DENSE>(P, b, sv, X, mode, row, qrow, vec_ok, use_ring);
        const int32_t ngroups = (V + kGroup - 1) / kGroup;
        const int32_t gs = slice * kSliceGroups, ge = min(ngroups, gs + kSliceGroups);
        const SliceTotals T = slice_totals_mode<LT, DENSE>(mode, row, qrow, gs, ge, V, vec_ok, use_ring, X, lane,
                                                           ring, P.rec_a + (b * NSL + slice) * kSliceTiles,
                                                           P.rec_q + (b * NSL + slice) * kSliceTiles);
        if (lane == 0) {
            long long *tot = P.slice_tot + (b * NSL + slice) * 2;
            tot[0] = T.A;
            tot[1] = __double_as_longlong(T.Qp);
            if (mode == kModeDense)
                atomicAdd(reinterpret_cast<unsigned long long *>(&P.seq_E[b]), static_cast<unsigned long long>(T.E));
            if (mode == kModeOneHot)
                atomicAdd(reinterpret_cast<unsigned long long *>(&P.seq_F[b]),
                          static_cast<unsigned long long>(static_cast<long long>(T.Ef)));
        }
    }
    int last = 0;
    if (lane == 0) {
        __threadfence();
        last = atomicAdd(&P.surv_cnt[b], 1u) == static_cast<unsigned>(NSL - 1);
    }
    last = __shfl_sync(0xFFFFFFFFu, last, 0);
    if (last)
        final_draw<LT, DENSE>(P, b, sv, lane, ring);
}

// The final draws.  Persistent warps take slice tickets from a counter; the
// warp that completes a sequence's last slice draws its token.  Launched
// behind the row pass with programmatic dependent launch: it waits in
// griddepcontrol.wait until the row pass has completed.
template <typename LT, bool DENSE>
__global__ void __launch_bounds__(kThreads, SV_MIN_CTAS) survivor_kernel(const Params P)
{
    extern __shared__ __align__(128) uint8_t smem[]; // kWarpSmem per warp
    const int lane = threadIdx.x & 31;
    uint8_t *ring = smem + (threadIdx.x >> 5) * kWarpSmem;
    pdl_wait_primary();
    const unsigned long long n = static_cast<unsigned long long>(P.B) * P.NSL;
    unsigned long long t = 0;
    if (lane == 0)
        t = atomicAdd(&P.ctr[0], 1ull);
    t = __shfl_sync(0xFFFFFFFFu, t, 0);
    while (t < n) {
        unsigned long long tn = 0;
        if (lane == 0) // the next ticket arrives while this one runs
            tn = atomicAdd(&P.ctr[0], 1ull);
        slice_item<LT, DENSE>(P, t, lane, ring);
        t = __shfl_sync(0xFFFFFFFFu, tn, 0);
    }
    // the last warp to finish returns the counters to zero
    if (lane == 0 && atomicAdd(&P.ctr[1], 1ull) == P.n_warps - 1) {
        P.ctr[0] = 0ull;
        P.ctr[1] = 0ull;
    }
}

} // namespace sv
