// sv_filter.cuh -- top-k / top-p filtering of target logit rows.
//
// The target distribution the accept test uses already carries the
// target's own sampling processing: temperature, top-k and top-p
// ("推测解码：草稿、验证与实际加速", section 接受与拒绝怎样保住分布).  The pages
// name these steps without defining them; the reading implemented here:
// the ids of a row are ordered by p = softmax(z / T) descending, equal p by
// ascending id; top-k keeps the first min(k, #finite) ids; top-p keeps the
// shortest prefix of that set whose mass reaches top_p times the set's mass
// (the crossing id is kept); every other logit becomes -inf, kept logits
// are copied unchanged, so softmax(z' / T) is the renormalised filtered p.
//
// One CTA per row (a persistent grid over the rows).  The first pass reads
// the row with an L2 evict-last hint and the output is stored evict-first,
// so the later passes find the rows in L2.  Masses are the
// verification's own: e_i = exp2(z_i c - fl(m c)) as an integer multiple of
// 2^-fb, so every sum is exact and order-independent.  Per row:
//   1. one pass: the maximum, the finite count, NaN / +inf detection (the
//      only pass that has to come from HBM; the rest find the row in L2);
//   2. one pass: counts in kYBins bins of y = z c - fl(m c) (bin 0 holds
//      the largest values; the last bin everything whose mass rounds to
//      zero), the exact masses of the top kTopBins bins, and the exact total
//      mass, summed in registers; the bin where the top-k count / top-p mass
//      is reached, by a scan from bin 0 (when the cut lies below the top
//      bins -- a large top-k, a flat row -- one more pass forms the masses
//      of the bins down to a limit that counts times each bin's smallest
//      mass sets);
//   3. inside that bin, the exact element.  A bin is a contiguous range of
//      the order key of z (an unsigned integer that sorts like z).  A bin of
//      at most kCollect ids is collected into shared memory in one pass,
//      sorted (bitonic, by key then id) and walked with a block scan.  A
//      larger bin is narrowed radix digit by radix digit (8 bits per pass,
//      starting below the bits all its keys share) to one value, and among
//      the ids holding that value the j-th in id order is found by an
//      ordered block scan;
//   4. one pass writes the row: z where (z, id) ranks at or before the cut,
//      -inf elsewhere.
// With both filters, top-k is resolved first (its cut bounds the elements
// top-p may keep, and its exact mass sets the top-p target).
#pragma once

#include "sv_device.cuh"

namespace sv {

constexpr int kFilterThreads = 256; // 4 CTAs per SM: rows spread over more CTA slots (384 rows of the
                                      // top-p workload: 608 slots instead of 304, so no partial second wave)
constexpr int kFilterWarps = kFilterThreads / 32;
constexpr int kYBins = 512;       // coarse bins of y
constexpr int kTieIds = 8;        // consecutive ids a thread owns in the ordered scan
constexpr int kCollect = 2048;    // ids of a bin resolved by a sort in shared memory
constexpr int kTopBins = 200;     // bins whose exact masses the binning pass forms (y >= -200/yscale)

struct FilterParams {
    const void *in;
    void *out;
    int64_t rows;
    int32_t V;
    float c;          // log2(e) / T
    int32_t top_k;    // <= 0: off
    float top_p;      // >= 1: off
    int fb;           // fractional bits of the masses
    float yscale;     // bins per unit of -y: kYBins / (fb + 2), so the last
                      // bin only holds ids whose mass rounds to zero
    int vec;          // rows are 16-byte aligned groups: vector loads
    int32_t *kept;    // [rows] or nullptr
    int32_t *status;  // or nullptr
};

// The element type's raw bits, value, order key and -inf pattern.
template <typename LT> struct FilterElem;
template <> struct FilterElem<uint16_t> {
    static constexpr int kPerVec = 8;
    __device__ static float value(uint32_t h) { return __uint_as_float(h << 16); }
    __device__ static bool finite(uint32_t h) { return (h & 0x7F80u) != 0x7F80u; }
    __device__ static bool nan_or_pinf(uint32_t h) { return (h & 0x7F80u) == 0x7F80u && h != 0xFF80u; }
    // -0 sorts as +0: they are the same logit
    __device__ static uint32_t key(uint32_t h)
    {
        h = h == 0x8000u ? 0u : h;
        return (h & 0x8000u) ? (~h & 0xFFFFu) : (h | 0x8000u);
    }
    __device__ static uint32_t bits_of_key(uint32_t k) { return (k & 0x8000u) ? (k & 0x7FFFu) : (~k & 0xFFFFu); }
    static constexpr uint32_t kNegInf = 0xFF80u;
    static constexpr uint32_t kKeyMin = 0x0080u, kKeyMax = 0xFF7Fu; // keys of the finite values
};
template <> struct FilterElem<float> {
    static constexpr int kPerVec = 4;
    __device__ static float value(uint32_t u) { return __uint_as_float(u); }
    __device__ static bool finite(uint32_t u) { return (u & 0x7F800000u) != 0x7F800000u; }
    __device__ static bool nan_or_pinf(uint32_t u) { return (u & 0x7F800000u) == 0x7F800000u && u != 0xFF800000u; }
    __device__ static uint32_t key(uint32_t u)
    {
        u = u == 0x80000000u ? 0u : u;
        return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
    }
    __device__ static uint32_t bits_of_key(uint32_t k) { return (k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k; }
    static constexpr uint32_t kNegInf = 0xFF800000u;
    static constexpr uint32_t kKeyMin = 0x00800000u, kKeyMax = 0xFF7FFFFFu;
};

// Raw bits of element i (plain loads: the output may be the input).
template <typename LT>
__device__ __forceinline__ uint32_t filter_bits(const LT *row, int64_t i)
{
    if constexpr (sizeof(LT) == 2)
        return reinterpret_cast<const unsigned short *>(row)[i];
    else
        return __float_as_uint(row[i]);
}

// 16-byte load keeping the line in L2 with priority (the later passes over
// the row find it there)
__device__ __forceinline__ uint4 ld_v4_keep(const void *p, uint64_t pol)
{
    uint4 r;
    asm volatile("ld.global.L2::cache_hint.v4.u32 {%0,%1,%2,%3}, [%4], %5;"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "l"(p), "l"(pol));
    return r;
}

// 16-byte store evicted from L2 first (the output is not read again here)
__device__ __forceinline__ void st_v4_stream(void *p, uint4 v, uint64_t pol)
{
    asm volatile("st.global.L2::cache_hint.v4.u32 [%0], {%1,%2,%3,%4}, %5;" ::"l"(p), "r"(v.x), "r"(v.y), "r"(v.z),
                 "r"(v.w), "l"(pol)
                 : "memory");
}

__device__ __forceinline__ uint64_t l2_policy_evict_last()
{
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
    return p;
}

__device__ __forceinline__ uint64_t l2_policy_evict_first()
{
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}

// Visit every element (id, raw bits) of a row; thread t takes vectors (or
// elements) t, t + blockDim, ...; the next U vectors are requested before
// the current ones are visited.  KEEP: loads carry an L2 evict-last hint.
template <typename LT, bool KEEP = false, typename F>
__device__ __forceinline__ void filter_visit(const LT *row, int32_t V, bool vec, F &&f)
{
    if (vec) {
        constexpr int PV = FilterElem<LT>::kPerVec;
        constexpr int U = 4; // vectors a thread has in flight
        const int32_t nv = V / PV;
        const uint4 *rv = reinterpret_cast<const uint4 *>(row);
        const uint64_t pol = KEEP ? l2_policy_evict_last() : 0ull;
        auto load = [&](int32_t v) { return KEEP ? ld_v4_keep(rv + v, pol) : rv[v]; };
        auto visit_vec = [&](int32_t v, const uint4 w) {
            const uint32_t u[4] = {w.x, w.y, w.z, w.w};
            if constexpr (PV == 8) {
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    f(v * 8 + 2 * k, u[k] & 0xFFFFu);
                    f(v * 8 + 2 * k + 1, u[k] >> 16);
                }
            } else {
#pragma unroll
                for (int k = 0; k < 4; ++k)
                    f(v * 4 + k, u[k]);
            }
        };
        constexpr int32_t STEP = U * kFilterThreads;
        const int32_t nfull = nv / STEP * STEP; // vectors in whole steps
        int32_t v = threadIdx.x;
        if (nfull > 0) {
            uint4 w[U], nx[U];
#pragma unroll
            for (int t = 0; t < U; ++t)
                w[t] = load(v + t * kFilterThreads);
            for (; v < nfull; v += STEP) {
                const bool more = v + STEP < nfull;
#pragma unroll
                for (int t = 0; t < U; ++t)
                    nx[t] = more ? load(v + STEP + t * kFilterThreads) : w[t];
#pragma unroll
                for (int t = 0; t < U; ++t)
                    visit_vec(v + t * kFilterThreads, w[t]);
#pragma unroll
                for (int t = 0; t < U; ++t)
                    w[t] = nx[t];
            }
        }
        for (; v < nv; v += kFilterThreads)
            visit_vec(v, load(v));
    } else {
        for (int32_t i = threadIdx.x; i < V; i += kFilterThreads)
            f(i, filter_bits<LT>(row, i));
    }
}

struct FilterShared {
    unsigned int cnt[kYBins];
    unsigned long long mass[kYBins];
    unsigned int dcnt[256];
    unsigned long long dmass[256];
    float redf[kFilterWarps];
    long long redl[kFilterWarps];
    union {
        struct {
            uint32_t ckey[kCollect]; // a bin's collected ids: keys, then sorted with them
            int32_t cid[kCollect];
        };
        unsigned int wcnt[kFilterWarps][kYBins]; // the binning pass: each warp's own counts
    };
    unsigned long long wmass[kFilterWarps][kTopBins]; // and its own top-bin masses
    unsigned int ncol;
    unsigned int kmin, kmax;
    int bad;
    int found;
    int32_t found_id;
};

__device__ __forceinline__ float block_max_f(float v, FilterShared &S)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
        v = fmaxf(v, __shfl_xor_sync(0xFFFFFFFFu, v, o));
    __syncthreads();
    if (lane == 0)
        S.redf[warp] = v;
    __syncthreads();
    float r = S.redf[0];
#pragma unroll
    for (int w = 1; w < kFilterWarps; ++w)
        r = fmaxf(r, S.redf[w]);
    return r;
}

__device__ __forceinline__ long long block_sum_l(long long v, FilterShared &S)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    v = warp_sum_ll(v);
    __syncthreads();
    if (lane == 0)
        S.redl[warp] = v;
    __syncthreads();
    long long r = 0;
#pragma unroll
    for (int w = 0; w < kFilterWarps; ++w)
        r += S.redl[w];
    return r;
}

// The per-row constants every pass forms masses and bins with.
struct FilterRow {
    float c, mc, yscale;
    int fb;
    __device__ float y(float z) const { return __fmaf_rn(z, c, -mc); }
    __device__ long long w(float yv) const { return to_fixed(ex2(yv), fb); }
    __device__ int bin(float yv) const
    {
        const float t = fmaxf(__fmul_rn(-yv, yscale), 0.0f);
        return t < static_cast<float>(kYBins - 1) ? static_cast<int>(t) : kYBins - 1;
    }
};

// The keys of coarse bin b: [klo, khi].  The bin of a value never grows
// with its key (y is a rounded fma of z with c > 0, the bin a rounded
// scaling of -y), so a bin is a contiguous range of keys, found by binary
// search over the finite keys (every thread computes the same range).
template <typename LT>
__device__ __forceinline__ void bin_keys(const FilterRow &R, int b, uint32_t &klo, uint32_t &khi)
{
    using E = FilterElem<LT>;
    auto first_at_most = [&](int bb) { // smallest finite key whose bin is <= bb
        uint64_t lo = E::kKeyMin, hi = static_cast<uint64_t>(E::kKeyMax) + 1;
        while (lo < hi) {
            const uint64_t mid = (lo + hi) >> 1;
            if (R.bin(R.y(E::value(E::bits_of_key(static_cast<uint32_t>(mid))))) <= bb)
                hi = mid;
            else
                lo = mid + 1;
        }
        return lo;
    };
    klo = static_cast<uint32_t>(first_at_most(b));
    khi = b == 0 ? E::kKeyMax : static_cast<uint32_t>(first_at_most(b - 1) - 1);
}

// Ranks first in the filter order: the larger key, then the smaller id.
__device__ __forceinline__ bool ranks_first(uint32_t ka, int32_t ia, uint32_t kb, int32_t ib)
{
    return ka > kb || (ka == kb && ia < ib);
}

// k >> s, 0 for s >= 32 (a bin's keys may differ in all 32 bits)
__device__ __forceinline__ uint32_t shr32(uint32_t k, int s) { return s >= 32 ? 0u : k >> s; }

// A cut in the order: (key, id).  Element (k, i) ranks at or before it iff
// k > key or (k == key and i <= id).
struct Cut {
    uint32_t key;
    int32_t id;
    __device__ bool covers(uint32_t k, int32_t i) const { return k > key || (k == key && i <= id); }
};

// Inside coarse bin `b`, among the finite elements at or before `bound`
// (when `bounded`), the element at which the running count reaches
// `target` (MASS = false) or the running mass reaches `target` (MASS = true),
// in the filter order.  Returns the cut at that element and adds the mass
// of the elements up to and including it to *mass_upto.
template <typename LT, bool MASS>
__device__ Cut filter_resolve(const LT *row, int32_t V, bool vec, const FilterRow &R, int b, bool bounded,
                              Cut bound, long long target, long long *mass_upto, FilterShared &S)
{
    using E = FilterElem<LT>;
    uint32_t klo, khi;
    bin_keys<LT>(R, b, klo, khi);
    auto member = [&](int32_t i, uint32_t bits, uint32_t &k) {
        k = E::key(bits); // non-finite keys lie outside every bin's range
        return k >= klo && k <= khi && (!bounded || bound.covers(k, i));
    };
    auto considered = [&](int32_t i, uint32_t bits, uint32_t &k, long long &w) {
        if (!member(i, bits, k))
            return false;
        w = R.w(R.y(E::value(bits)));
        return true;
    };
    if (S.cnt[b] <= static_cast<unsigned>(kCollect)) {
        // the bin fits in shared memory: collect it, sort it, walk it
        if (threadIdx.x == 0)
            S.ncol = 0u;
        __syncthreads();
        filter_visit<LT>(row, V, vec, [&](int32_t i, uint32_t bits) {
            uint32_t k;
            if (member(i, bits, k)) {
                const unsigned slot = atomicAdd(&S.ncol, 1u);
                if (slot < static_cast<unsigned>(kCollect)) { // the bin's count bounds it; kept in bounds regardless
                    S.ckey[slot] = k;
                    S.cid[slot] = i;
                }
            }
        });
        __syncthreads();
        const int n = S.ncol < static_cast<unsigned>(kCollect) ? static_cast<int>(S.ncol) : kCollect;
        int n2 = 1;
        while (n2 < n)
            n2 <<= 1;
        for (int i = n + threadIdx.x; i < n2; i += kFilterThreads) { // padding ranks last
            S.ckey[i] = 0u;
            S.cid[i] = 0x7FFFFFFF;
        }
        __syncthreads();
        for (int k = 2; k <= n2; k <<= 1) { // bitonic sort into the filter order
            for (int j = k >> 1; j > 0; j >>= 1) {
                for (int i = threadIdx.x; i < n2; i += kFilterThreads) {
                    const int l = i ^ j;
                    if (l > i) {
                        const bool first = (i & k) == 0; // this pair sorts into filter order
                        const bool swap = first ? ranks_first(S.ckey[l], S.cid[l], S.ckey[i], S.cid[i])
                                                : ranks_first(S.ckey[i], S.cid[i], S.ckey[l], S.cid[l]);
                        if (swap) {
                            const uint32_t tk = S.ckey[i];
                            const int32_t ti = S.cid[i];
                            S.ckey[i] = S.ckey[l];
                            S.cid[i] = S.cid[l];
                            S.ckey[l] = tk;
                            S.cid[l] = ti;
                        }
                    }
                }
                __syncthreads();
            }
        }
        // running masses in that order: thread t owns entries 4t .. 4t+3
        constexpr int PT = kCollect / kFilterThreads;
        const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
        long long pre[PT];
        long long run = 0;
#pragma unroll
        for (int e = 0; e < PT; ++e) {
            const int i = threadIdx.x * PT + e;
            run += i < n ? R.w(R.y(E::value(E::bits_of_key(S.ckey[i])))) : 0;
            pre[e] = run;
        }
        const long long incl = warp_incl_scan_ll(run, lane);
        __syncthreads();
        if (lane == 31)
            S.redl[warp] = incl;
        if (threadIdx.x == 0)
            S.found_id = 0x7FFFFFFF;
        __syncthreads();
        long long off = incl - run;
        for (int w = 0; w < warp; ++w)
            off += S.redl[w];
#pragma unroll
        for (int e = 0; e < PT; ++e) {
            const int i = threadIdx.x * PT + e;
            pre[e] += off;
            const bool hit = MASS ? (i < n && pre[e] >= target) : (i == target - 1);
            if (hit)
                atomicMin(&S.found_id, i);
        }
        __syncthreads();
        const int ci = S.found_id < n ? S.found_id : n - 1;
        if (ci >= threadIdx.x * PT && ci < threadIdx.x * PT + PT)
            S.redl[0] = pre[ci - threadIdx.x * PT]; // running mass through the cut
        __syncthreads();
        const Cut cut = {S.ckey[ci], S.cid[ci]};
        *mass_upto += S.redl[0];
        __syncthreads();
        return cut;
    }
    // the key bits every considered element shares
    if (threadIdx.x == 0) {
        S.kmin = 0xFFFFFFFFu;
        S.kmax = 0u;
    }
    __syncthreads();
    filter_visit<LT>(row, V, vec, [&](int32_t i, uint32_t bits) {
        uint32_t k;
        long long w;
        if (considered(i, bits, k, w)) {
            atomicMin(&S.kmin, k);
            atomicMax(&S.kmax, k);
        }
    });
    __syncthreads();
    const uint32_t kx = S.kmin ^ S.kmax;
    int hi = kx ? 32 - __clz(kx) : 0; // the low `hi` bits still differ
    uint32_t prefix = shr32(S.kmax, hi);
    long long rem = target;
    long long acc_mass = 0;
    while (hi > 0) {
        const int lo = hi > 8 ? hi - 8 : 0;
        const int nd = 1 << (hi - lo);
        __syncthreads();
        for (int d = threadIdx.x; d < nd; d += kFilterThreads) {
            S.dcnt[d] = 0u;
            S.dmass[d] = 0ull;
        }
        __syncthreads();
        filter_visit<LT>(row, V, vec, [&](int32_t i, uint32_t bits) {
            uint32_t k;
            long long w;
            if (considered(i, bits, k, w) && shr32(k, hi) == prefix) {
                const uint32_t d = (k >> lo) & static_cast<uint32_t>(nd - 1);
                atomicAdd(&S.dcnt[d], 1u);
                if (w)
                    atomicAdd(&S.dmass[d], static_cast<unsigned long long>(w));
            }
        });
        __syncthreads();
        // every thread scans the (at most 256) digits from the top: the same
        // answer everywhere, no broadcast needed
        int d = nd - 1;
        for (; d > 0; --d) {
            const long long have = MASS ? static_cast<long long>(S.dmass[d]) : static_cast<long long>(S.dcnt[d]);
            if (have >= rem)
                break;
            rem -= have;
            acc_mass += static_cast<long long>(S.dmass[d]);
        }
        prefix = (prefix << (hi - lo)) | static_cast<uint32_t>(d);
        hi = lo;
    }
    // one value left: its ids in id order, the j-th of them is the cut
    const uint32_t kcut = prefix;
    const float ycut = R.y(E::value(E::bits_of_key(kcut)));
    const long long wcut = R.w(ycut);
    long long j = rem; // count target
    if (MASS)
        j = wcut > 0 ? (rem + wcut - 1) / wcut : 1;
    if (j < 1)
        j = 1;
    *mass_upto += acc_mass + j * wcut;
    // ordered scan: thread t owns ids [t0 + t * kTieIds, t0 + (t+1) * kTieIds)
    if (threadIdx.x == 0) {
        S.found = 0;
        S.found_id = -1;
    }
    __syncthreads();
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    for (int64_t t0 = 0; t0 < V; t0 += static_cast<int64_t>(kFilterThreads) * kTieIds) {
        const int64_t i0 = t0 + static_cast<int64_t>(threadIdx.x) * kTieIds;
        uint32_t hits = 0; // bit m: id i0 + m holds the value (and is considered)
#pragma unroll
        for (int m = 0; m < kTieIds; ++m) {
            const int64_t i = i0 + m;
            if (i < V) {
                const uint32_t bits = filter_bits<LT>(row, i);
                if (E::finite(bits) && E::key(bits) == kcut &&
                    (!bounded || bound.covers(kcut, static_cast<int32_t>(i))))
                    hits |= 1u << m;
            }
        }
        const long long n = __popc(hits);
        // block exclusive scan of n in thread (= id) order
        long long incl = warp_incl_scan_ll(n, lane);
        __syncthreads();
        if (lane == 31)
            S.redl[warp] = incl;
        __syncthreads();
        long long before = incl - n;
        long long total = 0;
#pragma unroll
        for (int w = 0; w < kFilterWarps; ++w) {
            const long long s = S.redl[w];
            if (w < warp)
                before += s;
            total += s;
        }
        if (before < j && j <= before + n) {
            uint32_t h = hits;
            for (long long r = j - before; r > 1; --r)
                h &= h - 1; // drop the lowest set bit
            S.found_id = static_cast<int32_t>(i0 + (__ffs(h) - 1));
            S.found = 1;
        }
        __syncthreads();
        if (S.found)
            break;
        j -= total;
    }
    __syncthreads();
    const Cut cut = {kcut, S.found_id};
    __syncthreads();
    return cut;
}

template <typename LT>
__global__ void __launch_bounds__(kFilterThreads, 4) filter_kernel(const FilterParams P)
{
    using E = FilterElem<LT>;
    __shared__ FilterShared S;
    const int32_t V = P.V;
    for (int64_t r = blockIdx.x; r < P.rows; r += gridDim.x) {
        const LT *row = static_cast<const LT *>(P.in) + r * V;
        LT *orow = static_cast<LT *>(P.out) + r * V;
        // 1. maximum, finite count, bad entries
        float m = -INFINITY;
        long long nfin = 0;
        int bad = 0;
        filter_visit<LT, true>(row, V, P.vec, [&](int32_t, uint32_t bits) {
            if (E::finite(bits)) {
                m = fmaxf(m, E::value(bits));
                ++nfin;
            } else if (E::nan_or_pinf(bits)) {
                bad = 1;
            }
        });
        if (threadIdx.x == 0)
            S.bad = 0;
        __syncthreads();
        if (bad)
            S.bad = 1;
        m = block_max_f(m, S);
        nfin = block_sum_l(nfin, S);
        if (S.bad || nfin == 0) {
            // a row the verification rejects anyway: copied unchanged
            if (P.out != P.in)
                for (int32_t i = threadIdx.x; i < V; i += kFilterThreads)
                    orow[i] = row[i];
            if (threadIdx.x == 0) {
                if (P.kept)
                    P.kept[r] = 0;
                if (P.status)
                    atomicOr(P.status, kBadRow);
            }
            __syncthreads();
            continue;
        }
        const FilterRow R = {P.c, mc_of(m, P.c), P.yscale, P.fb};

        // 2. coarse bins of y: counts only, and the exact total mass in
        // registers (the last bin's ids have zero mass and are only counted)
        // each warp counts into its own bins (no contention between warps);
        // they are added up after the pass
        unsigned int *wc = S.wcnt[threadIdx.x >> 5];
        unsigned long long *wm = S.wmass[threadIdx.x >> 5];
        for (int i = threadIdx.x & 31; i < kYBins; i += 32)
            wc[i] = 0u;
        for (int i = threadIdx.x & 31; i < kTopBins; i += 32)
            wm[i] = 0ull;
        for (int i = threadIdx.x; i < kYBins; i += kFilterThreads) {
            S.cnt[i] = 0u;
            S.mass[i] = 0ull;
        }
        __syncthreads();
        long long Stot = 0;
        unsigned int nlast = 0; // the last bin (zero mass) is the crowded one: counted in a register
        filter_visit<LT>(row, V, P.vec, [&](int32_t, uint32_t bits) {
            const bool fin = E::finite(bits);
            const float yv = fin ? R.y(E::value(bits)) : 0.0f;
            const int b = fin ? R.bin(yv) : -1;
            if (b == kYBins - 1) {
                ++nlast;
            } else if (b >= 0) {
                atomicAdd(&wc[b], 1u);
                const long long w = R.w(yv);
                Stot += w;
                if (b < kTopBins && w) // the top bins' exact masses: the cuts lie there for most rows
                    atomicAdd(&wm[b], static_cast<unsigned long long>(w));
            }
        });
        if (nlast)
            atomicAdd(&wc[kYBins - 1], nlast);
        Stot = block_sum_l(Stot, S); // (its barriers also end every warp's binning)
        for (int i = threadIdx.x; i < kYBins; i += kFilterThreads) {
            unsigned int c = 0u;
#pragma unroll
            for (int w = 0; w < kFilterWarps; ++w)
                c += S.wcnt[w][i];
            S.cnt[i] = c;
            if (i < kTopBins) {
                unsigned long long m2 = 0ull;
#pragma unroll
                for (int w = 0; w < kFilterWarps; ++w)
                    m2 += S.wmass[w][i];
                S.mass[i] = m2;
            }
        }
        __syncthreads();

        // 3. the cuts.  Exact bin masses are needed only above the cut: for
        // the bins before the top-k bin, or, for top-p alone, down to the
        // first bin where a lower bound of the running mass (counts times the
        // smallest mass a bin holds) reaches the target; they are formed in
        // one more pass over the ids of those bins only.
        const bool use_k = P.top_k >= 1 && static_cast<long long>(P.top_k) < nfin;
        const bool use_p = P.top_p < 1.0f;
        bool have_cut = false;
        Cut cut = {0u, -1};
        long long Sk = Stot; // mass of the top-k set
        int bk = kYBins - 1;
        long long acck = 0;
        if (use_k) {
            for (bk = 0; bk < kYBins - 1; ++bk) {
                if (acck + static_cast<long long>(S.cnt[bk]) >= P.top_k)
                    break;
                acck += S.cnt[bk];
            }
        }
        int b3 = -1; // exact masses of bins 0 .. b3
        if (use_p) {
            if (use_k) {
                b3 = bk - 1;
            } else {
                // below the top bins, a lower bound of the running mass
                // (counts times each bin's smallest mass) limits the bins
                // the threshold may lie in
                long long tau0 = static_cast<long long>(ceil(static_cast<double>(P.top_p) * static_cast<double>(Stot)));
                tau0 = tau0 < 1 ? 1 : tau0;
                long long top = 0; // the top bins' exact masses first: usually they reach the target
                for (b3 = 0; b3 < kTopBins; ++b3) {
                    top += static_cast<long long>(S.mass[b3]);
                    if (top >= tau0)
                        break;
                }
                long long lower = 0;
                if (b3 == kTopBins)
                    b3 = 0;
                else
                    lower = tau0; // found: the loop below stops at once
                for (; b3 < kYBins - 1; ++b3) {
                    if (lower >= tau0)
                        break;
                    // the smallest mass an id of bin b3 can have, taken a
                    // little below the bin's edge in y (an id's bin comes
                    // from a rounded product): a lower bound
                    const long long wlo = R.w(-(static_cast<float>(b3) + 1.01f) / R.yscale) - 1;
                    lower += static_cast<long long>(S.cnt[b3]) * (wlo > 0 ? wlo : 0);
                    if (lower >= tau0)
                        break;
                }
            }
            if (b3 >= kTopBins) { // masses below the top bins: one more pass, rarely needed
                filter_visit<LT>(row, V, P.vec, [&](int32_t, uint32_t bits) {
                    if (E::finite(bits)) {
                        const float yv = R.y(E::value(bits));
                        const int b = R.bin(yv);
                        if (b >= kTopBins && b <= b3) {
                            const long long w = R.w(yv);
                            if (w)
                                atomicAdd(&S.mass[b], static_cast<unsigned long long>(w));
                        }
                    }
                });
                __syncthreads();
            }
        }
        if (use_k) {
            long long accm = 0;
            for (int b = 0; b < bk; ++b)
                accm += static_cast<long long>(S.mass[b]); // exact when top-p needs them, unused otherwise
            Sk = accm;
            cut = filter_resolve<LT, false>(row, V, P.vec, R, bk, false, cut, P.top_k - acck, &Sk, S);
            have_cut = true;
        }
        if (use_p) {
            long long tau = static_cast<long long>(ceil(static_cast<double>(P.top_p) * static_cast<double>(Sk)));
            if (tau < 1)
                tau = 1;
            long long accm = 0;
            int b = 0;
            const int blim = use_k ? bk : b3;
            for (; b < blim; ++b) {
                if (accm + static_cast<long long>(S.mass[b]) >= tau)
                    break;
                accm += static_cast<long long>(S.mass[b]);
            }
            long long upto = accm;
            cut = filter_resolve<LT, true>(row, V, P.vec, R, b, have_cut && b == bk, cut, tau - accm, &upto, S);
            have_cut = true;
        }

        // 4. write the row
        long long kept = 0;
        const bool vec = P.vec;
        auto keep_of = [&](int32_t i, uint32_t bits) {
            return E::finite(bits) && (!have_cut || cut.covers(E::key(bits), i));
        };
        if (vec) {
            constexpr int PV = E::kPerVec;
            const int32_t nv = V / PV;
            const uint4 *rv = reinterpret_cast<const uint4 *>(row);
            uint4 *ov = reinterpret_cast<uint4 *>(orow);
            const uint64_t wpol = l2_policy_evict_first();
            for (int32_t v = threadIdx.x; v < nv; v += kFilterThreads) {
                const uint4 w = rv[v];
                uint32_t u[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    if constexpr (PV == 8) {
                        uint32_t lo = u[k] & 0xFFFFu, hi = u[k] >> 16;
                        const bool kl = keep_of(v * 8 + 2 * k, lo), kh = keep_of(v * 8 + 2 * k + 1, hi);
                        kept += kl + kh;
                        lo = kl ? lo : E::kNegInf;
                        hi = kh ? hi : E::kNegInf;
                        u[k] = lo | (hi << 16);
                    } else {
                        const bool kk = keep_of(v * 4 + k, u[k]);
                        kept += kk;
                        u[k] = kk ? u[k] : E::kNegInf;
                    }
                }
                st_v4_stream(ov + v, make_uint4(u[0], u[1], u[2], u[3]), wpol);
            }
        } else {
            for (int32_t i = threadIdx.x; i < V; i += kFilterThreads) {
                const uint32_t bits = filter_bits<LT>(row, i);
                const bool kk = keep_of(i, bits);
                kept += kk;
                const uint32_t o = kk ? bits : E::kNegInf;
                if constexpr (sizeof(LT) == 2)
                    reinterpret_cast<unsigned short *>(orow)[i] = static_cast<unsigned short>(o);
                else
                    reinterpret_cast<uint32_t *>(orow)[i] = o;
            }
        }
        kept = block_sum_l(kept, S);
        if (threadIdx.x == 0 && P.kept)
            P.kept[r] = static_cast<int32_t>(kept);
        __syncthreads();
    }
}

} // namespace sv
