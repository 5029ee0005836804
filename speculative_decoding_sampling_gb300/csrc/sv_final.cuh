// sv_final.cuh -- the final draw of each sequence: one CTA per sequence.
//
// Once the draw stream has completed (the kernel boundary), every chunk of
// every surviving row has its record (A, Qp) and every sequence its
// normaliser (E or F).  The final token is the first id whose running
// residual mass exceeds u_K * Z, Z the row's total (inverse CDF in id order,
// "推测解码：草稿、验证与实际加速", section 算完三个 token 的全部概率, the replay's
// sampler and its final draw): a block scan over the records finds the chunk,
// a block scan over the chunk's 128 groups (one per thread, re-formed with
// the fold's arithmetic) finds the group, and running sums in id order the
// id.  All boundaries are exact integers in 2^-fb units: u * Z is taken as
// floor(u * Z) from a 96-bit product, so u * Z < P iff floor(u * Z) < P.
#pragma once

#include <climits>

#include "sv_survivor.cuh"

namespace sv {

constexpr int kFinalThreads = 128;
constexpr int kFinalWarps = kFinalThreads / 32;

// A chunk record's boundary mass max(0, A - delta * Qp) in 2^-fb units.
__device__ __forceinline__ long long rec_value(long long a, float q, float delta)
{
    const long long v = a - corr_of(delta, q);
    return v > 0 ? v : 0;
}

// Block-wide inclusive scan of one int64 per thread, in thread order; the
// block total in `tot`.  `sw` holds kFinalWarps values of scratch.
__device__ __forceinline__ long long block_incl_scan_ll(long long v, long long *sw, long long &tot)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const long long incl = warp_incl_scan_ll(v, lane);
    if (lane == 31)
        sw[warp] = incl;
    __syncthreads();
    long long off = 0;
    tot = 0;
#pragma unroll
    for (int w = 0; w < kFinalWarps; ++w) {
        const long long x = sw[w];
        if (w < warp)
            off += x;
        tot += x;
    }
    __syncthreads();
    return incl + off;
}

// The smallest thread index with `pred`, or kFinalThreads.
__device__ __forceinline__ int block_first(bool pred, int *si)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const unsigned m = __ballot_sync(0xFFFFFFFFu, pred);
    if (lane == 0)
        si[warp] = m ? warp * 32 + __ffs(m) - 1 : kFinalThreads;
    __syncthreads();
    int f = kFinalThreads;
#pragma unroll
    for (int w = 0; w < kFinalWarps; ++w)
        f = min(f, si[w]);
    __syncthreads();
    return f;
}

// The largest value over the block.
__device__ __forceinline__ int block_max(int v, int *si)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    v = __reduce_max_sync(0xFFFFFFFFu, v);
    if (lane == 0)
        si[warp] = v;
    __syncthreads();
    int r = INT_MIN;
#pragma unroll
    for (int w = 0; w < kFinalWarps; ++w)
        r = max(r, si[w]);
    __syncthreads();
    return r;
}

// Block-wide inclusive scan of one int64 per thread (thread order) fused
// with the search for the first thread whose prefix exceeds a threshold and
// the maximum of `mx` over the block: two barriers.  The threshold is `thr`,
// or floor(u * total) when `u` is not negative.  With `s_excl`, every
// thread's exclusive prefix is left there, visible after the call.  Each call site passes its
// own scratch, so no barrier is needed after the call.
struct ScanFirst {
    long long incl, tot, thr;
    int first, mx;
};

__device__ __forceinline__ ScanFirst block_scan_first(long long v, long long thr, float u, int mx, long long *s_tot,
                                                      int *s_mx, int *s_first, long long *s_excl = nullptr)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    ScanFirst r;
    r.incl = warp_incl_scan_ll(v, lane);
    const int wmx = __reduce_max_sync(0xFFFFFFFFu, mx);
    if (lane == 31)
        s_tot[warp] = r.incl;
    if (lane == 0)
        s_mx[warp] = wmx;
    __syncthreads();
    long long off = 0;
    r.tot = 0;
    r.mx = INT_MIN;
#pragma unroll
    for (int w = 0; w < kFinalWarps; ++w) {
        const long long x = s_tot[w];
        if (w < warp)
            off += x;
        r.tot += x;
        r.mx = max(r.mx, s_mx[w]);
    }
    r.incl += off;
    if (s_excl) // each thread's exclusive prefix, for the search after the call
        s_excl[threadIdx.x] = r.incl - v;
    r.thr = u >= 0.0f ? mul_floor(u, r.tot) : thr;
    const unsigned m = __ballot_sync(0xFFFFFFFFu, r.incl > r.thr);
    if (lane == 0)
        s_first[warp] = m ? warp * 32 + __ffs(m) - 1 : kFinalThreads;
    __syncthreads();
    r.first = kFinalThreads;
#pragma unroll
    for (int w = 0; w < kFinalWarps; ++w)
        r.first = min(r.first, s_first[w]);
    return r;
}

// One round of the id scan: groups g0 .. g0 + 127 of a row, one per thread.
// Looks for the first id whose boundary (carry + running group values, then
// running sums in id order within the group) exceeds `rem`; returns it, or
// -1 with `carry` advanced by the round.  `last_pos` tracks the last id of
// positive mass seen.  Block-collective.
template <typename LT, bool DENSE, int MODE>
__device__ int32_t scan_round(const LT *row, const float *qrow, int32_t g0, int32_t V, bool vec_ok,
                              const SurvArgs &X, float delta, long long rem, long long &carry, int32_t &last_pos,
                              long long *sw, int *si)
{
    const int tid = threadIdx.x;
    const int32_t ng = (V + kGroup - 1) / kGroup;
    const int32_t g = g0 + tid;
    float z[kGroup], q[kGroup];
    load_group_any<LT, DENSE>(row, qrow, g, ng, V, vec_ok, z, q);
    unsigned long long pt2[kGroup / 2];
    float w[kGroup], qp[kGroup], ws, qs;
    group_masses<MODE, DENSE>(z, q, g * kGroup, X, pt2, w, qp, ws, qs);
    const long long Lg = to_fixed(ws, X.fb) - corr_of(delta, qs);
    int kpos = -1;
#pragma unroll
    for (int k = 0; k < kGroup; ++k)
        if (w[k] > 0.0f)
            kpos = k;
    long long tot;
    const long long incl = block_incl_scan_ll(Lg, sw, tot) + carry;
    const int lp = block_max(kpos >= 0 ? g * kGroup + kpos : -1, si);
    if (lp >= 0)
        last_pos = lp;
    const int f = block_first(incl > rem, si);
    if (f == kFinalThreads) {
        carry += tot;
        return -1;
    }
    if (tid == f) {
        // running sums in id order (the group's last boundary is its total,
        // so an id past rounding falls back to its last id of positive mass)
        const long long excl = incl - Lg;
        int32_t tok = g * kGroup + (kpos >= 0 ? kpos : 0);
        float cw = 0.0f, cq = 0.0f;
        for (int k = 0; k < kGroup; ++k) {
            cw = __fadd_rn(cw, w[k]);
            cq = __fadd_rn(cq, qp[k]);
            if (w[k] > 0.0f && excl + to_fixed(cw, X.fb) - corr_of(delta, cq) > rem) {
                tok = g * kGroup + k;
                break;
            }
        }
        si[0] = tok;
    }
    __syncthreads();
    const int32_t tok = si[0];
    __syncthreads();
    return tok;
}

// Scratch of the final kernel's block-wide steps.
struct FinalSmem {
    long long sw[kFinalWarps];
    int si[kFinalWarps];
    long long tot[2][kFinalWarps];
    int mx[2][kFinalWarps];
    int first[2][kFinalWarps];
    long long excl[kFinalThreads];
};

// The final draw of sequence b and the return of its scratch to zero.
// Two rounds of loads: the sequence's verdict, normaliser, uniform and
// chunk records together; then the chosen chunk (one group per thread).
template <typename LT, bool DENSE>
__device__ void final_sequence(const Params &P, int64_t b, FinalSmem &sm, long long *s_v)
{
    const int tid = threadIdx.x;
    const int32_t K = P.K, V = P.V, CPS = P.CPS;
    long long *ra = P.rec_a + b * CPS;
    float *rq = P.rec_q + b * CPS;
    // ---- first load round, all in flight together
    const int4 info = __ldcg(&P.seq_info[b]);
    const long long Eraw = DENSE ? __ldcg(&P.seq_E[b]) : 0;
    const float u = __ldg(&P.u[b * (K + 1) + K]);
    const int R = (CPS + kFinalThreads - 1) / kFinalThreads; // thread t holds chunks [t*R, (t+1)*R)
    for (int i = 0; i < R; ++i) {
        const int c = tid * R + i;
        if (c < CPS) {
            const long long a = __ldcg(&ra[c]);
            const float q = __ldcg(&rq[c]);
            s_v[c] = a; // raw; turned into boundary masses below
            reinterpret_cast<float *>(s_v + CPS)[c] = q;
            ra[c] = 0; // the scratch goes back to zero as soon as it is read
            rq[c] = 0.0f;
        }
    }
    const int64_t r0 = b * (static_cast<int64_t>(K) + 1);
    for (int64_t i = tid; i < (static_cast<int64_t>(K) + 1) * P.PM; i += kFinalThreads)
        P.row_part[r0 * P.PM + i] = make_float2(0.0f, 0.0f); // not read here
    const int32_t jstar = info.x;
    if (jstar >= 0) {
        const bool rejected = jstar < K;
        Verdict v;
        v.jstar = jstar;
        v.m = __int_as_float(info.y);
        v.s = __int_as_float(info.z);
        v.x = info.w;
        const LT *row;
        const float *qrow;
        seq_rows<LT, DENSE>(P, b, v, row, qrow);
        const SurvArgs X = surv_args(P, v);
        const bool vec_ok = (reinterpret_cast<uintptr_t>(row) & 15u) == 0 &&
                            (qrow == nullptr || (reinterpret_cast<uintptr_t>(qrow) & 15u) == 0);
        // dense: delta = E - 2^fb = (S' - 1) 2^fb, S' the exact sum of pt;
        // one-hot: the residual's mass is 1 - p(x), p(x) as the accept test
        // took it (z(x) from the row pass's side data)
        const long long E = rejected && DENSE ? Eraw : 0;
        const float zx = rejected && !DENSE ? __ldcg(&P.row_side[b * (K + 1) + jstar]).y : 0.0f;
        const float delta = rejected && DENSE ? static_cast<float>(E - (1ll << P.fix_bits)) : 0.0f;
        // ---- the chunk: block scan over the threads' record sums, the
        // first thread whose running sum passes floor(u * Z)
        long long T = 0;
        int lastc = -1;
        for (int i = 0; i < R; ++i) {
            const int c = tid * R + i;
            if (c < CPS) {
                const long long vc = rec_value(s_v[c], reinterpret_cast<const float *>(s_v + CPS)[c], delta);
                s_v[c] = vc;
                T += vc;
                if (vc > 0)
                    lastc = c;
            }
        }
        const ScanFirst sr = block_scan_first(T, 0, u, lastc, sm.tot[0], sm.mx[0], sm.first[0], sm.excl);
        const long long Z = sr.tot;
        // every thread has read the sequence's info, normaliser and side
        // data before the scan's barriers
        for (int32_t j = tid; j <= K; j += kFinalThreads)
            P.row_side[r0 + j] = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
        if (tid == 0) {
            P.seq_E[b] = 0;
            P.seq_info[b] = make_int4(0, 0, 0, 0);
        }
        int32_t tok = -1;
        const bool degenerate = rejected && !(Z > 0);
        if (degenerate) {
            // residual of zero mass after a rejection (impossible in exact
            // arithmetic): draw from p of the same row instead
            SurvArgs Xb = X;
            Xb.x = -1;
            long long A = 0;
            const int32_t ng = (V + kGroup - 1) / kGroup;
            for (int32_t g0 = 0; g0 < ng; g0 += kFinalThreads) {
                float z[kGroup], q[kGroup];
                load_group_any<LT, false>(row, nullptr, g0 + tid, ng, V, vec_ok, z, q);
                unsigned long long pt2[kGroup / 2];
                float w[kGroup], qp[kGroup], ws, qs;
                group_masses<kModeBonus, false>(z, q, (g0 + tid) * kGroup, Xb, pt2, w, qp, ws, qs);
                A += to_fixed(ws, Xb.fb);
            }
            long long Zp;
            (void)block_incl_scan_ll(A, sm.sw, Zp);
            const long long t = mul_floor(u, Zp);
            long long carry = 0;
            int32_t last_pos = -1;
            for (int32_t g0 = 0; g0 < ng && tok < 0; g0 += kFinalThreads)
                tok = scan_round<LT, false, kModeBonus>(row, nullptr, g0, V, vec_ok, Xb, 0.0f, t, carry, last_pos,
                                                        sm.sw, sm.si);
            if (tok < 0)
                tok = last_pos;
        } else {
            const long long t = sr.thr;
            // every thread walks the chosen thread's chunks itself (the
            // records and the prefixes are in shared memory): no barrier
            int32_t sel = -1;
            long long acc = 0;
            if (sr.first < kFinalThreads) {
                acc = sm.excl[sr.first];
                for (int i = 0; i < R && sel < 0; ++i) {
                    const int c = sr.first * R + i;
                    if (c < CPS) {
                        const long long vc = s_v[c];
                        if (vc > 0 && acc + vc > t)
                            sel = c;
                        else
                            acc += vc;
                    }
                }
            }
            long long rem = t - acc;
            if (sel < 0) { // rounding put the draw past the last chunk: take its last id
                sel = sr.mx;
                rem = LLONG_MAX;
            }
            if (sel >= 0) {
                // ---- second load round: the chunk's 128 groups, one per thread
                constexpr int MODE = LaunchMode<DENSE>::value;
                const int32_t ng = (V + kGroup - 1) / kGroup;
                const int32_t g = sel * kChunkGroups + tid;
                float z[kGroup], q[kGroup];
                load_group_any<LT, DENSE>(row, qrow, g, ng, V, vec_ok, z, q);
                unsigned long long pt2[kGroup / 2];
                float w[kGroup], qp[kGroup], ws, qs;
                group_masses<MODE, DENSE>(z, q, g * kGroup, X, pt2, w, qp, ws, qs);
                const long long Lg = to_fixed(ws, X.fb) - corr_of(delta, qs);
                int kpos = -1;
#pragma unroll
                for (int k = 0; k < kGroup; ++k)
                    if (w[k] > 0.0f)
                        kpos = k;
                const ScanFirst gr = block_scan_first(Lg, rem, -1.0f, kpos >= 0 ? g * kGroup + kpos : -1,
                                                      sm.tot[1], sm.mx[1], sm.first[1]);
                if (tid == gr.first) {
                    // running sums in id order (the group's last boundary is
                    // its total, so an id past rounding falls back to its last
                    // id of positive mass)
                    // (all 8 boundaries formed independently, the first
                    // passing one taken)
                    const long long excl = gr.incl - Lg;
                    float cw = 0.0f, cq = 0.0f;
                    unsigned hit = 0u;
#pragma unroll
                    for (int k = 0; k < kGroup; ++k) {
                        cw = __fadd_rn(cw, w[k]);
                        cq = __fadd_rn(cq, qp[k]);
                        if (w[k] > 0.0f && excl + to_fixed(cw, X.fb) - corr_of(delta, cq) > rem)
                            hit |= 1u << k;
                    }
                    P.out_tokens[b * (K + 1) + jstar] =
                        g * kGroup + (hit ? __ffs(hit) - 1 : (kpos >= 0 ? kpos : 0));
                } else if (gr.first == kFinalThreads && tid == 0) {
                    P.out_tokens[b * (K + 1) + jstar] = gr.mx; // the chunk's last id of positive mass
                }
                tok = -2; // written above
            }
        }
        if (tid == 0) {
            if (tok != -2)
                P.out_tokens[b * (K + 1) + jstar] = tok;
            if (P.residual_mass) {
                float rm = 0.0f;
                if (rejected && !degenerate) {
                    if (DENSE) // Z / 2^fb over the residual's normaliser S'
                        rm = E > 0 ? __fdiv_rn(static_cast<float>(Z), static_cast<float>(E)) : 0.0f;
                    else
                        rm = __fsub_rn(1.0f, __fdiv_rn(term(zx, X.c, X.mc), v.s));
                }
                P.residual_mass[b] = rm;
            }
            if (degenerate && P.status)
                atomicOr(P.status, kDegenerate);
        }
    } else {
        // a sequence with bad data: nothing to draw, only scratch to clear
        __syncthreads(); // every thread has read the info
        for (int32_t j = tid; j <= K; j += kFinalThreads)
            P.row_side[r0 + j] = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
        if (tid == 0) {
            P.seq_E[b] = 0;
            P.seq_info[b] = make_int4(0, 0, 0, 0);
        }
    }
    __syncthreads(); // the block's scratch is reused by the next sequence
}

// The final draws: one CTA per sequence (grid-stride beyond the grid size).
// Dynamic shared memory: CPS chunk records (8 + 4 bytes each).
template <typename LT, bool DENSE>
__global__ void __launch_bounds__(kFinalThreads) final_kernel(const Params P)
{
    __shared__ FinalSmem sm;
    extern __shared__ __align__(16) long long s_v[];
    pdl_wait_primary();
    for (int64_t b = blockIdx.x; b < P.B; b += gridDim.x)
        final_sequence<LT, DENSE>(P, b, sm, s_v);
}

} // namespace sv
