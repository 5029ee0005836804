// sv_tree.cuh -- verification of a candidate tree (several drafts per node).
//
// The rule is multi-step speculative sampling (SpecInfer, Miao et al.,
// ASPLOS 2024): the pages require that a tree commits one contiguous path
// and keeps the target distribution, and that the chain's single-candidate
// correction is not applied to a tree as it stands ("推测解码：草稿、验证与
// 实际加速", section 链、树与自推测), but give no rule of their own.
//
// Sequence b has N nodes; node 0 is the committed prefix, node i >= 1 holds
// a draft token and parent[i] < i.  Row i of the logits gives p_i, the
// target's next-token distribution after node i's path; row i of q is the
// draft distribution node i's children were drawn from (i.i.d.).  From
// v = 0: the children of v, in index order, are tested against a running
// target r (first r = p_v): child c with token x is accepted iff
// u[c] < min(1, r(x) / q_v(x)); after a rejection r becomes
// max(0, r - q_v) normalised.  That residual has a closed form: after k
// rejections r = max(0, p_v - C_k q_v) / W_k with C_1 = 1,
// W_k = sum max(0, p_v - C_k q_v) and C_{k+1} = C_k + W_k, so each
// rejection is one pass over row v (p and q) for W_k.  When every child is
// rejected the final token is drawn from the last residual with u[0]; at a
// leaf it is drawn from p_v with u[0] (inverse CDF in id order).
//
// The row pass (rows_kernel over all B*N rows) supplies each row's
// (max, normaliser) partials; this kernel, a cluster of two CTAs per
// sequence, merges them, checks the inputs and walks the tree.  Masses in the passes are
// exact integer multiples of 2^-fix_bits (to_fixed), so sums are
// order-independent and the draw's boundaries agree with its totals.
#pragma once

#include "sv_rows.cuh"

namespace sv {

constexpr int kTreeThreads = 1024;
constexpr int kTreeWarps = kTreeThreads / 32;
constexpr int kTreeChunk = 256;     // ids per warp chunk: one group of 8 per lane
constexpr int kTreeMaxNodes = 256;   // nodes of one tree (the C ABI's SV_MAX_TREE_NODES)
constexpr int32_t kBadTree = 64;

struct TreeArgs {
    const int32_t *parent;  // [B, N]
    const int32_t *tokens;  // [B, N]
    const float *q;         // [B, N, V]
    const float *u;         // [B, N]
    int32_t N;
    int32_t *out_tokens;    // [B, N]
    int32_t *out_nodes;     // [B, N] or nullptr
    int32_t *num_emitted;   // [B]
    float *accept_prob;     // [B, N] or nullptr
    int32_t *status;        // or nullptr
};

struct TreeRow {
    const void *z;   // logits row (LT)
    const float *q;  // draft row
    float c, mc, inv_s;
    bool zvec, qvec; // rows 16-byte aligned: whole groups load as vectors
};

// The weights of the 8 ids of group g (ids past V weigh 0): p_i (bonus) or
// max(0, p_i - C q_i), p_i = exp2(z_i c - mc) / s in fp32.
template <typename LT>
__device__ __forceinline__ void tree_group(const TreeRow &R, int32_t g, int32_t V, bool resid, float C, float (&w)[8])
{
    const int32_t i0 = g * 8;
    float z[8], q[8];
    const LT *zr = static_cast<const LT *>(R.z) + i0;
    if (R.zvec && i0 + 8 <= V) {
        if constexpr (sizeof(LT) == 2) {
            const uint4 v = ld_stream_v4(zr);
            z[0] = bf16_lo(v.x); z[1] = bf16_hi(v.x); z[2] = bf16_lo(v.y); z[3] = bf16_hi(v.y);
            z[4] = bf16_lo(v.z); z[5] = bf16_hi(v.z); z[6] = bf16_lo(v.w); z[7] = bf16_hi(v.w);
        } else {
            const uint4 v0 = ld_stream_v4(zr), v1 = ld_stream_v4(zr + 4);
            z[0] = __uint_as_float(v0.x); z[1] = __uint_as_float(v0.y); z[2] = __uint_as_float(v0.z);
            z[3] = __uint_as_float(v0.w); z[4] = __uint_as_float(v1.x); z[5] = __uint_as_float(v1.y);
            z[6] = __uint_as_float(v1.z); z[7] = __uint_as_float(v1.w);
        }
    } else {
#pragma unroll
        for (int k = 0; k < 8; ++k)
            z[k] = i0 + k < V ? load_elem<LT>(zr + k) : -INFINITY;
    }
    if (resid) {
        const float *qr = R.q + i0;
        if (R.qvec && i0 + 8 <= V) {
            const uint4 v0 = ld_stream_v4(qr), v1 = ld_stream_v4(qr + 4);
            q[0] = __uint_as_float(v0.x); q[1] = __uint_as_float(v0.y); q[2] = __uint_as_float(v0.z);
            q[3] = __uint_as_float(v0.w); q[4] = __uint_as_float(v1.x); q[5] = __uint_as_float(v1.y);
            q[6] = __uint_as_float(v1.z); q[7] = __uint_as_float(v1.w);
        } else {
#pragma unroll
            for (int k = 0; k < 8; ++k)
                q[k] = i0 + k < V ? __ldg(qr + k) : 0.0f;
        }
    }
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        const float p = __fmul_rn(term(z[k], R.c, R.mc), R.inv_s);
        w[k] = resid ? fmaxf(__fmaf_rn(-C, q[k], p), 0.0f) : p;
    }
}

// The raw bits of group g of a 16-bit logits row and of its draft row (ids
// past V: -inf and 0), loaded before any is used, so a warp can have two
// groups in flight.  tree_raw_weights turns them into the weights
// tree_group gives, with the same arithmetic.
struct TreeRaw {
    uint4 z;      // 8 logits (bf16 bits)
    uint4 q0, q1; // 8 draft probabilities (fp32 bits), resid only
};

__device__ __forceinline__ TreeRaw tree_raw_load(const TreeRow &R, int32_t g, int32_t V, bool resid)
{
    TreeRaw t;
    const int32_t i0 = g * 8;
    const unsigned short *zr = static_cast<const unsigned short *>(R.z) + i0;
    if (R.zvec && i0 + 8 <= V) {
        t.z = ld_stream_v4(zr);
    } else {
        uint32_t h[8];
#pragma unroll
        for (int k = 0; k < 8; ++k)
            h[k] = i0 + k < V ? zr[k] : 0xFF80u;
        t.z = make_uint4(h[0] | h[1] << 16, h[2] | h[3] << 16, h[4] | h[5] << 16, h[6] | h[7] << 16);
    }
    t.q0 = t.q1 = make_uint4(0u, 0u, 0u, 0u);
    if (resid) {
        const float *qr = R.q + i0;
        if (R.qvec && i0 + 8 <= V) {
            t.q0 = ld_stream_v4(qr);
            t.q1 = ld_stream_v4(qr + 4);
        } else {
            uint32_t u[8];
#pragma unroll
            for (int k = 0; k < 8; ++k)
                u[k] = i0 + k < V ? __float_as_uint(__ldg(qr + k)) : 0u;
            t.q0 = make_uint4(u[0], u[1], u[2], u[3]);
            t.q1 = make_uint4(u[4], u[5], u[6], u[7]);
        }
    }
    return t;
}

__device__ __forceinline__ void tree_raw_weights(const TreeRaw &t, const TreeRow &R, bool resid, float C, float (&w)[8])
{
    const float z[8] = {bf16_lo(t.z.x), bf16_hi(t.z.x), bf16_lo(t.z.y), bf16_hi(t.z.y),
                        bf16_lo(t.z.z), bf16_hi(t.z.z), bf16_lo(t.z.w), bf16_hi(t.z.w)};
    const uint32_t qb[8] = {t.q0.x, t.q0.y, t.q0.z, t.q0.w, t.q1.x, t.q1.y, t.q1.z, t.q1.w};
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        const float p = __fmul_rn(term(z[k], R.c, R.mc), R.inv_s);
        w[k] = resid ? fmaxf(__fmaf_rn(-C, __uint_as_float(qb[k]), p), 0.0f) : p;
    }
}

// A group's mass: its 8 weights added in fp32 in id order, as a fixed-point
// integer.  The draw re-forms the same sums, so its boundaries agree.
__device__ __forceinline__ long long tree_group_fixed(const float (&w)[8], int fb)
{
    float s = w[0];
#pragma unroll
    for (int k = 1; k < 8; ++k)
        s = __fadd_rn(s, w[k]);
    return to_fixed(s, fb);
}

// A sequence is walked by a cluster of two CTAs (one per SM), which take the
// same decisions from the same data and split each pass over the row.
constexpr int kTreeCtas = 2;

__device__ __forceinline__ uint32_t tree_rank()
{
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

__device__ __forceinline__ void tree_cluster_sync()
{
    asm volatile("barrier.cluster.arrive.release;\n\tbarrier.cluster.wait.acquire;" ::: "memory");
}

// A 64-bit store into the same shared-memory location of CTA `rank`.
__device__ __forceinline__ void tree_st_peer(long long *p, uint32_t rank, long long v)
{
    uint32_t a;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(a) : "r"(smem_addr(p)), "r"(rank));
    asm volatile("st.shared::cluster.u64 [%0], %1;" ::"r"(a), "l"(v) : "memory");
}

// Bulk prefetches into L2 (cp.async.bulk.prefetch.L2): fire and forget,
// nothing waits for them.  Only the whole 16-byte units inside [p, p + n)
// are requested (the instruction's granule), so a prefetch never reaches
// outside the range it is given.
__device__ __forceinline__ void prefetch_l2_units(uintptr_t a, uintptr_t e)
{
    if (a < e)
        asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(a), "r"(static_cast<uint32_t>(e - a))
                     : "memory");
}

// [p, p + n) cut into one request per lane of the calling warp.
__device__ __forceinline__ void prefetch_l2_lanes(const void *p, int64_t n, int lane)
{
    const uintptr_t a = (reinterpret_cast<uintptr_t>(p) + 15u) & ~uintptr_t{15};
    const uintptr_t e = (reinterpret_cast<uintptr_t>(p) + static_cast<uintptr_t>(n)) & ~uintptr_t{15};
    if (e <= a)
        return;
    const uintptr_t piece = (((e - a + 31u) / 32u) + 15u) & ~uintptr_t{15};
    const uintptr_t b0 = a + static_cast<uintptr_t>(lane) * piece;
    prefetch_l2_units(b0, b0 + piece < e ? b0 + piece : e);
}

// One pass over the row: per-chunk totals into chunk[] (in both CTAs) and
// the row total (returned to every thread of both).  This CTA takes the
// chunks [c0, c1) of its half; warp w of it takes chunks c0 + w, c0 + w + 32,
// ...; lane l group 32 ch + l of chunk ch.  Its chunk totals are also
// written into the other CTA's chunk[], and its half of the row total into
// slot npass mod 2 of both CTAs' half[], all before the one cluster barrier
// that ends the pass.  No barrier is needed before the writes: the two CTAs
// take the same decisions, nothing reads chunk[] between passes (only the
// final draw, after the last pass), and a CTA can reuse a half[] slot only
// after the other has passed the next pass's barrier, that is, after it has
// read the slot.
template <typename LT>
__device__ long long tree_pass(const TreeRow &R, int32_t V, bool resid, float C, int fb, long long *chunk,
                               long long *red, long long (*half)[kTreeCtas], int &npass)
{
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int32_t nch = (V + kTreeChunk - 1) / kTreeChunk;
    const uint32_t rank = tree_rank(), peer = rank ^ 1u;
    const int32_t halfc = (nch + 1) / 2;
    const int32_t c0 = rank ? halfc : 0, c1 = rank ? nch : halfc;
    if (warp == 0 && c0 < c1) {
        // this CTA's half of the row (and of the draft row) into L2 at the
        // copy bandwidth, so the warps' group loads below find it there
        const int64_t i0 = static_cast<int64_t>(c0) * kTreeChunk;
        const int64_t i1 = min(static_cast<int64_t>(c1) * kTreeChunk, static_cast<int64_t>(V));
        prefetch_l2_lanes(static_cast<const LT *>(R.z) + i0, (i1 - i0) * static_cast<int64_t>(sizeof(LT)), lane);
        if (resid)
            prefetch_l2_lanes(R.q + i0, (i1 - i0) * static_cast<int64_t>(sizeof(float)), lane);
    }
    long long wsum = 0; // this warp's chunk totals (the same in every lane)
    auto publish = [&](int32_t ch, const float (&w)[8]) {
        // a chunk's total: 256 masses of at most 2^fb each (fb <= 40), so
        // below 2^48, and non-negative
        const long long s = static_cast<long long>(warp_sum_u64(static_cast<unsigned long long>(tree_group_fixed(w, fb))));
        if (lane == 0) {
            chunk[ch] = s;
            tree_st_peer(&chunk[ch], peer, s);
        }
        wsum += s;
    };
    if constexpr (sizeof(LT) == 2) {
        // two chunks a warp: both groups' loads issued before either is used
        for (int32_t ch = c0 + warp; ch < c1; ch += 2 * kTreeWarps) {
            const int32_t ch2 = ch + kTreeWarps;
            const TreeRaw t1 = tree_raw_load(R, ch * 32 + lane, V, resid);
            TreeRaw t2;
            if (ch2 < c1)
                t2 = tree_raw_load(R, ch2 * 32 + lane, V, resid);
            float w[8];
            tree_raw_weights(t1, R, resid, C, w);
            publish(ch, w);
            if (ch2 < c1) {
                tree_raw_weights(t2, R, resid, C, w);
                publish(ch2, w);
            }
        }
    } else {
        for (int32_t ch = c0 + warp; ch < c1; ch += kTreeWarps) {
            float w[8];
            tree_group<LT>(R, ch * 32 + lane, V, resid, C, w);
            publish(ch, w);
        }
    }
    // this CTA's half of the total, into both CTAs' slot of this pass
    if (lane == 0)
        red[warp] = wsum;
    __syncthreads();
    const int slot = npass & 1;
    ++npass;
    if (threadIdx.x == 0) {
        long long h = 0;
#pragma unroll 8
        for (int w = 0; w < kTreeWarps; ++w)
            h += red[w];
        half[slot][rank] = h;
        tree_st_peer(&half[slot][rank], peer, h);
    }
    tree_cluster_sync();
    return half[slot][0] + half[slot][1];
}

// Hand-off slots of tree_find (shared memory).
struct TreeSel {
    long long base; // cumulative weight before the chosen chunk
    int32_t chunk;  // the chunk holding t, or -1
    int32_t id;     // the id found, or -1
};

// First id whose cumulative weight exceeds t (0 <= t < total), from the
// chunk totals of the last pass over the same weights; every thread gets
// it.  Within a group the boundaries are the fixed-point values of its fp32
// partial sums in id order (the last one is the group's mass).  If rounding
// leaves no id, the last id of positive weight.
template <typename LT>
__device__ int32_t tree_find(const TreeRow &R, int32_t V, bool resid, float C, int fb, long long t,
                             const long long *chunk, long long *red, TreeSel *sel)
{
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int32_t nch = (V + kTreeChunk - 1) / kTreeChunk;
    // thread j owns chunks [j*per, (j+1)*per): their total, an exclusive
    // block scan, and the one thread whose range holds t finds the chunk
    const int32_t per = (nch + kTreeThreads - 1) / kTreeThreads;
    const int32_t c0 = threadIdx.x * per;
    long long own = 0;
    for (int32_t k = 0; k < per && c0 + k < nch; ++k)
        own += chunk[c0 + k];
    long long inc = own; // inclusive warp scan
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const long long y = __shfl_up_sync(0xFFFFFFFFu, inc, o);
        if (lane >= o)
            inc += y;
    }
    if (lane == 31)
        red[warp] = inc;
    if (threadIdx.x == 0) {
        sel->chunk = -1;
        sel->id = -1;
    }
    __syncthreads();
    long long before = inc - own;
    for (int w = 0; w < warp; ++w)
        before += red[w];
    if (own > 0 && before <= t && t < before + own) {
        long long acc = before;
        for (int32_t k = 0; k < per && c0 + k < nch; ++k) {
            if (t < acc + chunk[c0 + k]) {
                sel->chunk = c0 + k;
                sel->base = acc;
                break;
            }
            acc += chunk[c0 + k];
        }
    }
    __syncthreads();
    const int32_t ch = sel->chunk;
    if (ch >= 0 && warp == 0) {
        // the chunk: group masses, exclusive scan, then the group's ids
        float w[8];
        tree_group<LT>(R, ch * 32 + lane, V, resid, C, w);
        const long long s = tree_group_fixed(w, fb);
        long long inc2 = s;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const long long y = __shfl_up_sync(0xFFFFFFFFu, inc2, o);
            if (lane >= o)
                inc2 += y;
        }
        const long long g0 = sel->base + inc2 - s;
        int32_t id = -1;
        if (s > 0 && g0 <= t && t < g0 + s) {
            float part = w[0];
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                if (k > 0)
                    part = __fadd_rn(part, w[k]);
                if (id < 0 && t < g0 + to_fixed(part, fb))
                    id = (ch * 32 + lane) * 8 + k;
            }
        }
        const unsigned m = __ballot_sync(0xFFFFFFFFu, id >= 0);
        const int32_t first = __shfl_sync(0xFFFFFFFFu, id, m ? __ffs(m) - 1 : 0);
        if (lane == 0)
            sel->id = m ? first : -1;
    }
    __syncthreads();
    if (sel->id < 0) { // rounding left no id below t: the last id of positive weight
        __syncthreads();
        if (threadIdx.x == 0) {
            int32_t last = 0;
            for (int32_t g = (V + 7) / 8 - 1; g >= 0 && last == 0; --g) {
                float w[8];
                tree_group<LT>(R, g, V, resid, C, w);
                for (int k = 7; k >= 0; --k)
                    if (g * 8 + k < V && w[k] > 0.0f) {
                        last = g * 8 + k;
                        break;
                    }
            }
            sel->id = last;
        }
        __syncthreads();
    }
    const int32_t id = sel->id;
    __syncthreads(); // sel is reused
    return id;
}

template <typename LT>
__global__ void __launch_bounds__(kTreeThreads) tree_kernel(const Params P, const TreeArgs A)
{
    extern __shared__ long long tree_chunk[]; // [ceil(V / 256)] chunk totals of the last pass
    __shared__ int32_t s_par[kTreeMaxNodes], s_tok[kTreeMaxNodes];
    __shared__ float s_u[kTreeMaxNodes], s_M[kTreeMaxNodes], s_S[kTreeMaxNodes];
    __shared__ float s_zx[kTreeMaxNodes], s_qx[kTreeMaxNodes]; // node i's token under its parent's rows
    __shared__ long long s_red[kTreeWarps];
    __shared__ long long s_half[2][kTreeCtas]; // the passes' half totals, by pass parity and CTA
    int npass = 0;
    __shared__ TreeSel s_sel;
    __shared__ int32_t s_bad;
    const int64_t b = blockIdx.x / kTreeCtas;
    const bool writer = tree_rank() == 0; // the even CTA writes the outputs
    const int32_t N = A.N, V = static_cast<int32_t>(P.V);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const float c = P.c;

    if (threadIdx.x == 0)
        s_bad = 0;
    for (int32_t i = threadIdx.x; i < N; i += kTreeThreads) {
        s_par[i] = A.parent[b * N + i];
        s_tok[i] = A.tokens[b * N + i];
        s_u[i] = A.u[b * N + i];
    }
    __syncthreads();
    // the inputs: u in [0, 1), parents before their nodes, tokens in range
    // with positive draft probability; and the child tests' two values,
    // gathered for every node at once.  None of this reads what the row pass
    // writes, so it runs while the row pass drains (programmatic dependent
    // launch).
    for (int32_t i = threadIdx.x; i < N; i += kTreeThreads) {
        int32_t bad = 0;
        if (!(s_u[i] >= 0.0f && s_u[i] < 1.0f))
            bad |= kBadU;
        if (i >= 1) {
            const int32_t pa = s_par[i], x = s_tok[i];
            if (pa < 0 || pa >= i) {
                bad |= kBadTree;
            } else if (x < 0 || x >= V) {
                bad |= kBadToken;
            } else {
                const float qx = __ldg(A.q + (b * N + pa) * static_cast<int64_t>(V) + x);
                s_qx[i] = qx;
                s_zx[i] = load_elem<LT>(static_cast<const LT *>(P.logits) + (b * N + pa) * static_cast<int64_t>(V) + x);
                if (!(qx > 0.0f && isfinite(qx)))
                    bad |= kBadQ;
            }
        }
        if (bad)
            atomicOr(&s_bad, bad);
    }
    pdl_wait_primary(); // the row pass has completed: its partials are all written
    // each row's (max, normaliser): the merge of its row-pass partials
    for (int32_t i = warp; i < N; i += kTreeWarps) {
        const int64_t r = b * N + i;
        int64_t first;
        int n;
        row_ctas<LT>(P, r, first, n);
        float M = -INFINITY, S = 0.0f;
        for (int k = lane; k < n; k += 32) {
            const float2 pr = __ldcg(&P.row_part[r * P.PM + k]);
            merge_ms(M, S, pr.x, pr.y, c);
        }
        warp_merge_ms(M, S, c);
        if (lane == 0) {
            s_M[i] = M;
            s_S[i] = S;
            if (!(isfinite(M) && isfinite(S)))
                atomicOr(&s_bad, kBadRow);
        }
    }
    __syncthreads();
    tree_cluster_sync(); // both CTAs have read the row pass's partials
    // the row pass's scratch of this sequence goes back to zero once read
    // (the workspace is shared with spec_verify, which expects it zeroed)
    if (writer) {
        for (int64_t i = threadIdx.x; i < static_cast<int64_t>(N) * P.PM; i += kTreeThreads)
            P.row_part[b * N * P.PM + i] = make_float2(0.0f, 0.0f);
        for (int32_t i = threadIdx.x; i < N; i += kTreeThreads)
            P.row_side[b * N + i] = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
    }
    __syncthreads();
    const int32_t bad = s_bad;
    if (bad) {
        if (!writer)
            return;
        for (int32_t i = threadIdx.x; i < N; i += kTreeThreads) {
            A.out_tokens[b * N + i] = -1;
            if (A.out_nodes) A.out_nodes[b * N + i] = -1;
            if (A.accept_prob) A.accept_prob[b * N + i] = -1.0f;
        }
        if (threadIdx.x == 0) {
            A.num_emitted[b] = 0;
            if (A.status) atomicOr(A.status, bad);
        }
        return;
    }
    if (A.accept_prob && writer)
        for (int32_t i = threadIdx.x; i < N; i += kTreeThreads)
            A.accept_prob[b * N + i] = -1.0f;

    const int fb = P.fix_bits;
    int32_t v = 0, len = 0, y = 0, status = 0;
    for (;;) {
        TreeRow R;
        R.z = static_cast<const LT *>(P.logits) + (b * N + v) * static_cast<int64_t>(V);
        R.q = A.q + (b * N + v) * static_cast<int64_t>(V);
        R.c = c;
        R.mc = mc_of(s_M[v], c);
        R.inv_s = __frcp_rn(s_S[v]);
        R.zvec = (reinterpret_cast<uintptr_t>(R.z) & 15u) == 0;
        R.qvec = (reinterpret_cast<uintptr_t>(R.q) & 15u) == 0;
        int32_t nrej = 0, next = -1;
        float C = 1.0f, W = 0.0f; // the residual max(0, p - C q) / W after nrej rejections
        long long Wfix = 0;
        bool degenerate = false;
        for (int32_t ch = v + 1; ch < N; ++ch) {
            if (s_par[ch] != v)
                continue;
            // every thread takes the same decision from the same values (C
            // and W come from the pass totals every thread holds), so none
            // has to wait for another's
            const float px = __fmul_rn(term(s_zx[ch], c, R.mc), R.inv_s);
            const float qx = s_qx[ch];
            const float rx = nrej == 0 ? px : __fdiv_rn(fmaxf(__fmaf_rn(-C, qx, px), 0.0f), W);
            const float a = fminf(1.0f, __fdiv_rn(rx, qx));
            if (threadIdx.x == 0 && A.accept_prob && writer)
                A.accept_prob[b * N + ch] = a;
            const bool acc = s_u[ch] < a;
            if (acc) {
                next = ch;
                break;
            }
            // rejected: the next residual's constant and normaliser
            C = nrej == 0 ? 1.0f : __fadd_rn(C, W);
            ++nrej;
            Wfix = tree_pass<LT>(R, V, true, C, fb, tree_chunk, s_red, s_half, npass);
            W = ldexpf(static_cast<float>(Wfix), -fb);
            if (Wfix <= 0) {
                degenerate = true;
                break;
            }
        }
        if (next >= 0) {
            if (threadIdx.x == 0 && writer) {
                A.out_tokens[b * N + len] = s_tok[next];
                if (A.out_nodes) A.out_nodes[b * N + len] = next;
            }
            ++len;
            v = next;
            continue;
        }
        // the final draw, with u[0]: from the residual after the last
        // rejection, else (a leaf, or a residual with no mass) from p_v
        const bool resid = nrej > 0 && !degenerate;
        long long tot = Wfix;
        if (!resid)
            tot = tree_pass<LT>(R, V, false, 0.0f, fb, tree_chunk, s_red, s_half, npass);
        if (degenerate)
            status |= kDegenerate;
        const long long t = mul_floor(s_u[0], tot);
        y = tree_find<LT>(R, V, resid, C, fb, t, tree_chunk, s_red, &s_sel);
        break;
    }
    if (!writer)
        return;
    if (threadIdx.x == 0) {
        A.out_tokens[b * N + len] = y;
        A.num_emitted[b] = len + 1;
        if (status && A.status)
            atomicOr(A.status, status);
    }
    for (int32_t i = len + threadIdx.x; i < N; i += kTreeThreads) {
        if (i > len)
            A.out_tokens[b * N + i] = -1;
        if (A.out_nodes)
            A.out_nodes[b * N + i] = -1;
    }
}

} // namespace sv
