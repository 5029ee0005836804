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

// ---------------------------------------------------------------------------
// The final draw inside the draw stream.  When every sequence has its own
// group of draw warps, the warp that completes a sequence's chunk count
// draws its token: a warp scan over the chunk records (each lane a
// contiguous run of chunks) picks the chunk, the chunk is staged in the
// warp's idle ring (each lane its own groups 32 t + lane, as in the stream),
// and a warp scan over its groups, tile by tile, picks the group and then the
// id -- the same exact boundaries as the final kernel.

// The chunk of a row holding boundary floor(u * Z) among the chunk masses
// `mass(c)`, each lane a contiguous run of chunks (up to 8 kept in
// registers): sets sel (the row's last chunk of positive mass, with before =
// LLONG_MIN, when rounding puts the boundary past the last chunk; -1 when
// every mass is 0), the mass before it and the boundary; returns the total Z.
// Warp-collective.
template <typename Mass>
__device__ long long chunk_select(int32_t nc, float u, Mass mass, int lane, int32_t &sel, long long &before,
                                  long long &thr)
{
    constexpr int kRegs = 8;
    const int32_t R = (nc + 31) / 32;
    const int32_t c_lo = min(nc, lane * R), c_hi = min(nc, c_lo + R);
    long long vr[kRegs];
#pragma unroll
    for (int i = 0; i < kRegs; ++i)
        vr[i] = c_lo + i < c_hi ? mass(c_lo + i) : 0;
    long long T = 0;
    int32_t lastc = -1;
#pragma unroll
    for (int i = 0; i < kRegs; ++i) {
        T += vr[i];
        if (vr[i] > 0)
            lastc = c_lo + i;
    }
    for (int32_t c = c_lo + kRegs; c < c_hi; ++c) {
        const long long vc = mass(c);
        T += vc;
        if (vc > 0)
            lastc = c;
    }
    const long long incl = warp_incl_scan_ll(T, lane);
    const long long Z = __shfl_sync(0xFFFFFFFFu, incl, 31);
    thr = mul_floor(u, Z);
    const unsigned hit = __ballot_sync(0xFFFFFFFFu, incl > thr);
    const int32_t last_all = __reduce_max_sync(0xFFFFFFFFu, lastc);
    if (!hit) {
        sel = last_all;
        before = LLONG_MIN;
        return Z;
    }
    const int src = __ffs(hit) - 1;
    int32_t s = -1;
    long long acc = incl - T;
#pragma unroll
    for (int i = 0; i < kRegs; ++i) {
        if (s < 0 && c_lo + i < c_hi) {
            if (vr[i] > 0 && acc + vr[i] > thr)
                s = c_lo + i;
            else
                acc += vr[i];
        }
    }
    if (lane == src) {
        for (int32_t c = c_lo + kRegs; s < 0 && c < c_hi; ++c) {
            const long long vc = mass(c);
            if (vc > 0 && acc + vc > thr)
                s = c;
            else
                acc += vc;
        }
    }
    sel = __shfl_sync(0xFFFFFFFFu, s, src);
    before = __shfl_sync(0xFFFFFFFFu, acc, src);
    if (sel < 0) { // not reached with exact running sums; kept as the final kernel's fallback
        sel = last_all;
        before = LLONG_MIN;
    }
    return Z;
}

// Stage chunk `sel` of a row (and of its draft row, WANT_Q) in ring stage
// `st`, in the stream's layout; lane l fetches (and later reads) groups
// 32 t + l.  RING: 16-byte async copies; otherwise element loads and shared
// stores.
template <typename LT, bool WANT_Q, bool RING>
__device__ __forceinline__ void fetch_chunk(const LT *row, const float *qrow, int32_t sel, int32_t V, bool vec_ok,
                                            int lane, uint8_t *st)
{
    constexpr int LB = kGroup * static_cast<int>(sizeof(LT));
    const int32_t ng = (V + kGroup - 1) / kGroup;
#pragma unroll
    for (int t = 0; t < kChunkTiles; ++t) {
        const int gl = 32 * t + lane;
        const int32_t g = sel * kChunkGroups + gl;
        if (g < ng) {
            if constexpr (RING) {
                const uint8_t *src = reinterpret_cast<const uint8_t *>(row + static_cast<int64_t>(g) * kGroup);
#pragma unroll
                for (int h = 0; h < LB; h += 16)
                    cp_async16(st + gl * LB + h, src + h);
                if (WANT_Q) {
                    const uint8_t *qsrc = reinterpret_cast<const uint8_t *>(qrow + static_cast<int64_t>(g) * kGroup);
                    cp_async16(st + kChunkGroups * LB + gl * 32, qsrc);
                    cp_async16(st + kChunkGroups * LB + gl * 32 + 16, qsrc + 16);
                }
            } else {
                float z[kGroup], q[kGroup];
                load_group<LT, WANT_Q>(row, qrow, g, ng, V, vec_ok, z, q);
#pragma unroll
                for (int k = 0; k < kGroup; ++k) {
                    if constexpr (sizeof(LT) == 2)
                        reinterpret_cast<uint16_t *>(st + gl * LB)[k] =
                            static_cast<uint16_t>(__float_as_uint(z[k]) >> 16); // exact: z came from bf16
                    else
                        reinterpret_cast<float *>(st + gl * LB)[k] = z[k];
                    if (WANT_Q)
                        reinterpret_cast<float *>(st + kChunkGroups * LB + gl * 32)[k] = q[k];
                }
            }
        }
    }
    if constexpr (RING) {
        cp_async_commit();
        cp_async_wait<0>();
    }
    __syncwarp(); // the scan reads other lanes' groups
}

// The id of the staged chunk `sel` whose boundary first exceeds `rem`
// (boundaries relative to the chunk's start), or the chunk's last id of
// positive mass when none does.  Each lane forms the group values of its own
// groups 32 t + lane into `sL` (128 entries of shared scratch), then takes
// four consecutive ones, 4 lane .. 4 lane + 3, for a single warp scan; the
// lane holding the first group whose running sum passes `rem` searches its
// ids.  Warp-collective.
template <typename LT, bool WANT_Q, int MODE, bool NORM>
__device__ int32_t chunk_id_scan_stage(const uint8_t *st, int32_t sel, int32_t V, const SurvArgs &X, float delta,
                                       long long rem, int lane, long long *sL)
{
    const int32_t ng = (V + kGroup - 1) / kGroup;
    const int32_t gbase = sel * kChunkGroups;
    int lastid = -1;
#pragma unroll 1
    for (int t = 0; t < kChunkTiles; ++t) {
        const int gl = 32 * t + lane;
        const int32_t g = gbase + gl;
        float z[kGroup], q[kGroup];
        load_group_smem<LT, WANT_Q>(st, gl, g < ng, z, q);
        unsigned long long pt2[kGroup / 2];
        float w[kGroup], qp[kGroup], ws, qs;
        group_masses<MODE, NORM>(z, q, g * kGroup, X, pt2, w, qp, ws, qs);
        sL[gl] = to_fixed(ws, X.fb) - corr_of(delta, qs);
#pragma unroll
        for (int k = 0; k < kGroup; ++k)
            if (w[k] > 0.0f)
                lastid = g * kGroup + k;
    }
    __syncwarp();
    static_assert(kChunkGroups == 4 * 32, "four consecutive groups per lane");
    long long L[4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
        L[i] = sL[4 * lane + i];
    const long long T = (L[0] + L[1]) + (L[2] + L[3]);
    const long long incl = warp_incl_scan_ll(T, lane);
    // the first of the lane's groups whose running sum passes rem
    long long run = incl - T;
    int hit_i = -1;
    long long excl_hit = 0;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        if (hit_i < 0 && run + L[i] > rem) {
            hit_i = i;
            excl_hit = run;
        }
        run += L[i];
    }
    const unsigned m = __ballot_sync(0xFFFFFFFFu, hit_i >= 0);
    if (!m)
        return __reduce_max_sync(0xFFFFFFFFu, lastid);
    const int hl = __ffs(m) - 1;
    int32_t tok = -1;
    if (lane == hl) {
        // running sums in id order (the group's last boundary is its total,
        // so an id past rounding falls back to its last id of positive mass)
        const int gl = 4 * lane + hit_i;
        const int32_t g = gbase + gl;
        float z[kGroup], q[kGroup];
        load_group_smem<LT, WANT_Q>(st, gl, g < ng, z, q);
        unsigned long long pt2[kGroup / 2];
        float w[kGroup], qp[kGroup], ws, qs;
        group_masses<MODE, NORM>(z, q, g * kGroup, X, pt2, w, qp, ws, qs);
        int kpos = 0;
        float cw = 0.0f, cq = 0.0f;
        unsigned hitk = 0u;
#pragma unroll
        for (int k = 0; k < kGroup; ++k) {
            if (w[k] > 0.0f)
                kpos = k;
            cw = __fadd_rn(cw, w[k]);
            cq = __fadd_rn(cq, qp[k]);
            if (w[k] > 0.0f && excl_hit + to_fixed(cw, X.fb) - corr_of(delta, cq) > rem)
                hitk |= 1u << k;
        }
        tok = g * kGroup + (hitk ? __ffs(hitk) - 1 : kpos);
    }
    return __shfl_sync(0xFFFFFFFFu, tok, hl);
}

template <typename LT, bool DENSE, bool RING>
__device__ void final_inline(const Params &P, int64_t b, const Verdict &v, int lane, uint8_t *stage)
{
    const int32_t K = P.K, V = P.V, CPS = P.CPS;
    long long *ra = P.rec_a + b * CPS;
    float *rq = P.rec_q + b * CPS;
    // the group values of the chosen chunk: in the ring's second stage
    long long *sL = reinterpret_cast<long long *>(stage + DrawShape<LT, DENSE>::kChunkBytes);
    // the sequence's scratch goes back to zero once it has been read (every
    // lane's loads of it have been consumed by the warp's shuffles first)
    auto zero_scratch = [&]() {
        __syncwarp();
        for (int32_t c = lane; c < CPS; c += 32) {
            ra[c] = 0;
            rq[c] = 0.0f;
        }
        const int64_t r0 = b * (static_cast<int64_t>(K) + 1);
        for (int64_t i = lane; i < (static_cast<int64_t>(K) + 1) * P.PM; i += 32)
            P.row_part[r0 * P.PM + i] = make_float2(0.0f, 0.0f);
        for (int32_t j = lane; j <= K; j += 32)
            P.row_side[r0 + j] = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
        if (lane == 0) {
            P.seq_E[b] = 0;
            P.seq_info[b] = make_int4(0, 0, 0, 0);
            P.seq_cnt[b] = 0u;
        }
    };
    const int32_t jstar = v.jstar;
    if (jstar < 0) { // a sequence with bad data: nothing to draw
        zero_scratch();
        return;
    }
    const bool rejected = jstar < K;
    const LT *row;
    const float *qrow;
    seq_rows<LT, DENSE>(P, b, v, row, qrow);
    const SurvArgs X = surv_args(P, v);
    const bool vec_ok = (reinterpret_cast<uintptr_t>(row) & 15u) == 0 &&
                        (qrow == nullptr || (reinterpret_cast<uintptr_t>(qrow) & 15u) == 0);
    const float u = __ldg(&P.u[b * (K + 1) + K]);
    // dense: delta = E - 2^fb = (S' - 1) 2^fb, S' the exact sum of pt;
    // one-hot: the residual's mass is 1 - p(x), p(x) as the accept test
    // took it (z(x) from the row pass's side data)
    const long long E = rejected && DENSE ? static_cast<long long>(__ldcg(&P.seq_E[b])) : 0;
    const float zx = rejected && !DENSE && lane == 0 ? __ldcg(&P.row_side[b * (K + 1) + jstar]).y : 0.0f;
    const float delta = rejected && DENSE ? static_cast<float>(E - (1ll << P.fix_bits)) : 0.0f;
    int32_t sel;
    long long before, thr;
    const long long Z = chunk_select(
        CPS, u, [&](int32_t c) { return rec_value(__ldcg(&ra[c]), __ldcg(&rq[c]), delta); }, lane, sel, before, thr);
    const bool degenerate = rejected && !(Z > 0);
    if (lane == 0) {
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
    zero_scratch();
    int32_t tok = -1;
    constexpr int MODE = LaunchMode<DENSE>::value;
    if (degenerate) {
        // residual of zero mass after a rejection (impossible in exact
        // arithmetic): draw from p of the same row instead -- the chunk
        // masses of p one chunk at a time, then the chosen chunk's ids
        SurvArgs Xb = X;
        Xb.x = -1;
        const int32_t ng = (V + kGroup - 1) / kGroup;
        auto chunk_mass = [&](int32_t c) {
            fetch_chunk<LT, false, RING>(row, nullptr, c, V, vec_ok, lane, stage);
            long long A = 0;
#pragma unroll 1
            for (int t = 0; t < kChunkTiles; ++t) {
                const int gl = 32 * t + lane;
                const int32_t g = c * kChunkGroups + gl;
                float z[kGroup], q[kGroup];
                load_group_smem<LT, false>(stage, gl, g < ng, z, q);
                unsigned long long pt2[kGroup / 2];
                float w[kGroup], qp[kGroup], ws, qs;
                group_masses<kModeBonus, false>(z, q, g * kGroup, Xb, pt2, w, qp, ws, qs);
                A += to_fixed(ws, Xb.fb);
            }
            return warp_sum_ll(A);
        };
        long long Zp = 0;
        for (int32_t c = 0; c < CPS; ++c)
            Zp += chunk_mass(c);
        const long long t = mul_floor(u, Zp);
        long long acc = 0;
        int32_t c = 0;
        for (; c < CPS - 1; ++c) {
            const long long m = chunk_mass(c);
            if (m > 0 && acc + m > t)
                break;
            acc += m;
        }
        fetch_chunk<LT, false, RING>(row, nullptr, c, V, vec_ok, lane, stage);
        tok = chunk_id_scan_stage<LT, false, kModeBonus, false>(stage, c, V, Xb, 0.0f, t - acc, lane, sL);
    } else if (sel >= 0) {
        const long long rem = before == LLONG_MIN ? LLONG_MAX : thr - before;
        if (DENSE && qrow != nullptr) {
            fetch_chunk<LT, true, RING>(row, qrow, sel, V, vec_ok, lane, stage);
            tok = chunk_id_scan_stage<LT, true, MODE, DENSE>(stage, sel, V, X, delta, rem, lane, sL);
        } else {
            fetch_chunk<LT, false, RING>(row, nullptr, sel, V, vec_ok, lane, stage);
            tok = chunk_id_scan_stage<LT, false, MODE, DENSE>(stage, sel, V, X, delta, rem, lane, sL);
        }
    }
    if (lane == 0)
        P.out_tokens[b * (K + 1) + jstar] = tok;
}

} // namespace sv
