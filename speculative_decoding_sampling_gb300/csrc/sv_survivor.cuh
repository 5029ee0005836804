// sv_survivor.cuh -- the final draw of each sequence.
//
// After the row pass, every sequence has one surviving row j*: the row of
// its first rejection, or row K when every draft passed.  One thread-block
// cluster (up to 8 CTAs, each a contiguous slice of the vocabulary) draws the
// final token from
//   rejected, dense q:  r_i = max(0, p_i - q_i)   (p = softmax(z_{j*} / T))
//   rejected, one-hot:  r_i = p_i for i != x, r_x = 0
//   all accepted:       p_i of row K
// by inverse CDF with the final uniform u_K: the smallest id i with
// u_K * sum(r) < r_0 + ... + r_i ("推测解码：草稿、验证与实际加速", sections
// 接受与拒绝怎样保住分布 (equation for r(x)) and 算完三个 token 的全部概率
// (the replay's sampler and its final draw)).
//
// Exactness: every mass is formed in fp32 from the unnormalised term
// e_i = exp2(z_i * c - fl(m * c)) (m the row maximum) and then held as an
// integer multiple of 2^-fix_bits, so every sum, prefix and the product
// floor(u_K * Z) are exact and independent of the reduction order.  The
// softmax normaliser s = sum_i e_i that the dense residual needs is itself
// such an exact sum, taken over the cluster before the residual is formed,
// and enters the residual as a two-float pair; no rounding of s or of any
// running sum can move a CDF boundary.
//
// Cluster protocol (no flag waits, only hardware cluster barriers):
//   dense rejected: pass A (exact s) -> exchange -> pass B (residual tiles)
//   otherwise:      pass B (masses and, for one-hot, s)
//   exchange of the slice totals -> the CTA whose slice holds floor(u_K * Z)
//   re-forms that one tile and scans it.
#pragma once

#include "sv_device.cuh"

namespace sv {

enum { kModeBonus = 0, kModeDense = 1, kModeOneHot = 2 };

template <typename LT>
__device__ __forceinline__ void load_group_z(const LT *row, int32_t g, int32_t V, bool vec_ok, float (&z)[kGroup])
{
    const int32_t e0 = g * kGroup;
    if (vec_ok && e0 + kGroup <= V) {
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
    } else {
#pragma unroll
        for (int k = 0; k < kGroup; ++k)
            z[k] = e0 + k < V ? load_elem<LT>(row + e0 + k) : -INFINITY;
    }
}

__device__ __forceinline__ void load_group_q(const float *qrow, int32_t g, int32_t V, bool vec_ok, float (&q)[kGroup])
{
    const int32_t e0 = g * kGroup;
    if (vec_ok && e0 + kGroup <= V) {
        const uint4 a = ld_stream_v4(qrow + e0), b = ld_stream_v4(qrow + e0 + 4);
        q[0] = __uint_as_float(a.x); q[1] = __uint_as_float(a.y);
        q[2] = __uint_as_float(a.z); q[3] = __uint_as_float(a.w);
        q[4] = __uint_as_float(b.x); q[5] = __uint_as_float(b.y);
        q[6] = __uint_as_float(b.z); q[7] = __uint_as_float(b.w);
    } else {
#pragma unroll
        for (int k = 0; k < kGroup; ++k)
            q[k] = e0 + k < V ? __ldg(qrow + e0 + k) : 0.0f;
    }
}

struct SurvCtx {
    float c, mc;     // log2(e)/T and fl(m*c) of the surviving row
    float s_hi, s_lo;// exact normaliser as a two-float pair (dense mode)
    float scale;     // 2^fix_bits
    int32_t x;       // rejected one-hot draft
    int mode;
};

// Fixed-point masses of the 8 elements of group g (and, in one-hot mode, of
// the unnormalised terms, for the normaliser).
template <typename LT>
__device__ __forceinline__ void group_masses(const LT *row, const float *qrow, int32_t g, int32_t V,
                                             bool vec_ok, const SurvCtx &X, long long (&f)[kGroup],
                                             long long &fe)
{
    float z[kGroup];
    load_group_z<LT>(row, g, V, vec_ok, z);
    float qv[kGroup];
    if (X.mode == kModeDense)
        load_group_q(qrow, g, V, vec_ok, qv);
    fe = 0;
#pragma unroll
    for (int k = 0; k < kGroup; ++k) {
        const float e = term(z[k], X.c, X.mc);
        float w = e;
        if (X.mode == kModeDense) {
            float d = __fmaf_rn(-X.s_hi, qv[k], e);
            d = __fmaf_rn(-X.s_lo, qv[k], d);
            w = fminf(fmaxf(d, 0.0f), 2.0f);
        } else if (X.mode == kModeOneHot) {
            w = (g * kGroup + k == X.x) ? 0.0f : e;
            fe += to_fixed(e, X.scale);
        }
        f[k] = to_fixed(w, X.scale);
    }
}

template <typename LT, bool DENSE>
__global__ void __launch_bounds__(kSurvThreads) survivor_kernel(const Params P)
{
    constexpr int NT = kSurvThreads, NW = NT / 32;
    __shared__ long long s_tile[kMaxTiles];
    __shared__ long long s_red[2][NW];
    __shared__ long long s_xch[2]; // [0] mass of this slice, [1] normaliser part
    __shared__ long long s_scan[NW];
    __shared__ int32_t s_sel_tile;
    __shared__ long long s_sel_rem;

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const uint32_t CL = static_cast<uint32_t>(P.CL);
    const uint32_t rank = cluster_ctarank();
    const int64_t b = blockIdx.x / CL;
    const int32_t jstar = __ldcg(&P.seq_jstar[b]);
    const float m_row = __ldcg(&P.seq_m[b]);
    if (jstar < 0) {
        // bad sequence: the same decision in every CTA of the cluster
        cluster_sync_all();
        if (rank == 0 && tid == 0)
            P.seq_jstar[b] = 0;
        return;
    }

    const int32_t K = P.K, V = P.V;
    const bool rejected = jstar < K;
    const int64_t r = b * (K + 1) + jstar;
    const LT *row = static_cast<const LT *>(P.logits) + r * static_cast<int64_t>(V);
    const float *qrow = (DENSE && rejected) ? P.q + (b * K + jstar) * static_cast<int64_t>(V) : nullptr;

    SurvCtx X;
    X.c = P.c;
    X.mc = mc_of(m_row, P.c);
    X.s_hi = 0.0f;
    X.s_lo = 0.0f;
    X.scale = __int_as_float((127 + P.fix_bits) << 23);
    X.x = (!DENSE && rejected) ? P.tokens[b * K + jstar] : -1;
    X.mode = !rejected ? kModeBonus : (DENSE ? kModeDense : kModeOneHot);

    const bool vec_ok = (reinterpret_cast<uintptr_t>(row) & 15u) == 0 &&
                        (qrow == nullptr || (reinterpret_cast<uintptr_t>(qrow) & 15u) == 0);
    const int32_t ngroups = (V + kGroup - 1) / kGroup;
    const int32_t g0 = static_cast<int32_t>(static_cast<int64_t>(ngroups) * rank / CL);
    const int32_t g1 = static_cast<int32_t>(static_cast<int64_t>(ngroups) * (rank + 1) / CL);
    const int32_t ntiles = (g1 - g0 + NT - 1) / NT;

    long long S_fixed = 0; // exact normaliser sum_i e_i, in units of 2^-fix_bits

    // ---- pass A (dense residual only): the exact normaliser over the cluster
    if (X.mode == kModeDense) {
        long long part = 0;
        for (int32_t g = g0 + tid; g < g1; g += NT) {
            float z[kGroup];
            load_group_z<LT>(row, g, V, vec_ok, z);
#pragma unroll
            for (int k = 0; k < kGroup; ++k)
                part += to_fixed(term(z[k], X.c, X.mc), X.scale);
        }
        part = warp_sum_ll(part);
        if (lane == 0)
            s_red[0][warp] = part;
        __syncthreads();
        if (tid == 0) {
            long long t = 0;
            for (int w = 0; w < NW; ++w)
                t += s_red[0][w];
            s_xch[1] = t;
        }
        cluster_sync_all();
        for (uint32_t k = 0; k < CL; ++k)
            S_fixed += ld_cluster_ll(&s_xch[1], k);
        const double s = ldexp(static_cast<double>(S_fixed), -P.fix_bits);
        X.s_hi = static_cast<float>(s);
        X.s_lo = static_cast<float>(s - static_cast<double>(X.s_hi));
        __syncthreads(); // s_red[0] is reused below
    }

    // ---- pass B: masses per tile, slice totals over the cluster
    long long Z = 0, prefix = 0, own = 0;
    bool degenerate = false;
    for (int attempt = 0; attempt < 2; ++attempt) {
        long long fe_part = 0;
        own = 0;
        for (int32_t t = 0; t < ntiles; ++t) {
            const int32_t g = g0 + t * NT + tid;
            long long ts = 0;
            if (g < g1) {
                long long f[kGroup], fe;
                group_masses<LT>(row, qrow, g, V, vec_ok, X, f, fe);
#pragma unroll
                for (int k = 0; k < kGroup; ++k)
                    ts += f[k];
                fe_part += fe;
            }
            ts = warp_sum_ll(ts);
            if (lane == 0)
                s_red[t & 1][warp] = ts;
            __syncthreads();
            if (tid == 0) {
                long long s = 0;
                for (int w = 0; w < NW; ++w)
                    s += s_red[t & 1][w];
                s_tile[t] = s;
                own += s;
            }
        }
        if (X.mode == kModeOneHot) {
            fe_part = warp_sum_ll(fe_part);
            __syncthreads();
            if (lane == 0)
                s_scan[warp] = fe_part;
            __syncthreads();
            if (tid == 0) {
                long long s = 0;
                for (int w = 0; w < NW; ++w)
                    s += s_scan[w];
                s_xch[1] = s;
            }
        }
        if (tid == 0)
            s_xch[0] = own;
        cluster_sync_all(); // slice totals visible cluster-wide
        Z = 0;
        prefix = 0;
        long long Sx = 0;
        for (uint32_t k = 0; k < CL; ++k) {
            const long long v = ld_cluster_ll(&s_xch[0], k);
            if (k < rank)
                prefix += v;
            Z += v;
            if (X.mode == kModeOneHot)
                Sx += ld_cluster_ll(&s_xch[1], k);
        }
        if (X.mode == kModeOneHot)
            S_fixed = Sx;
        cluster_sync_all(); // every remote read done before s_xch is reused or the CTA exits
        if (!(X.mode != kModeBonus && Z == 0))
            break;
        // residual of zero mass after a rejection (impossible in exact
        // arithmetic): draw from p of the same row instead
        X.mode = kModeBonus;
        degenerate = true;
    }
    // every CTA has read the per-sequence slots: return them to zero
    if (rank == 0 && tid == 0) {
        P.seq_jstar[b] = 0;
        P.seq_m[b] = 0.0f;
    }
    // the slice total was accumulated by thread 0 only
    if (tid == 0)
        s_scan[0] = own;
    __syncthreads();
    own = s_scan[0];
    __syncthreads();

    const float uK = P.u[b * (K + 1) + K];
    const long long t_abs = static_cast<long long>(floor_mul(uK, static_cast<unsigned long long>(Z)));
    if (!(t_abs >= prefix && t_abs < prefix + own))
        return; // another CTA of the cluster holds the draw
    const long long t_loc = t_abs - prefix;

    // ---- the tile holding the draw (warp 0 scans the tile totals)
    if (warp == 0) {
        long long run = 0;
        int32_t sel = -1;
        long long rem = 0;
        for (int32_t base = 0; base < ntiles && sel < 0; base += 32) {
            const int32_t t = base + lane;
            const long long v = t < ntiles ? s_tile[t] : 0;
            const long long incl = warp_incl_scan_ll(v, lane) + run;
            const unsigned m = __ballot_sync(0xFFFFFFFFu, t < ntiles && incl > t_loc);
            if (m) {
                const int l = __ffs(m) - 1;
                const long long incl_l = __shfl_sync(0xFFFFFFFFu, incl, l);
                const long long v_l = __shfl_sync(0xFFFFFFFFu, v, l);
                sel = base + l;
                rem = t_loc - (incl_l - v_l);
            }
            run = __shfl_sync(0xFFFFFFFFu, incl, 31);
        }
        if (lane == 0) {
            s_sel_tile = sel;
            s_sel_rem = rem;
        }
    }
    __syncthreads();
    const int32_t tsel = s_sel_tile;
    const long long rem = s_sel_rem;
    if (tsel < 0)
        return; // unreachable: the slice total covers t_loc

    // ---- re-form the selected tile and scan it
    const int32_t g = g0 + tsel * NT + tid;
    long long f[kGroup];
    long long ts = 0;
    if (g < g1) {
        long long fe;
        group_masses<LT>(row, qrow, g, V, vec_ok, X, f, fe);
#pragma unroll
        for (int k = 0; k < kGroup; ++k)
            ts += f[k];
    } else {
#pragma unroll
        for (int k = 0; k < kGroup; ++k)
            f[k] = 0;
    }
    const long long incl = warp_incl_scan_ll(ts, lane);
    if (lane == 31)
        s_scan[warp] = incl;
    __syncthreads();
    long long wbase = 0;
    for (int w = 0; w < warp; ++w)
        wbase += s_scan[w];
    const long long excl = wbase + incl - ts;
    if (rem >= excl && rem < excl + ts) {
        long long acc = excl;
        int32_t tok = g * kGroup + kGroup - 1;
#pragma unroll
        for (int k = 0; k < kGroup; ++k) {
            acc += f[k];
            if (rem < acc) {
                tok = g * kGroup + k;
                break;
            }
        }
        P.out_tokens[b * (K + 1) + jstar] = tok;
        if (P.residual_mass) {
            const float rm = (rejected && !degenerate && S_fixed > 0)
                                 ? static_cast<float>(static_cast<double>(Z) / static_cast<double>(S_fixed))
                                 : 0.0f;
            P.residual_mass[b] = rm;
        }
        if (degenerate && P.status)
            atomicOr(P.status, kDegenerate);
    }
}

} // namespace sv
