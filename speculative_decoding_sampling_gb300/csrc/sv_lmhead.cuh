// sv_lmhead.cuh -- the target's LM head fused with the row pass.
//
// logits = h W^T for the K+1 verified positions of every sequence: h bf16
// [M, d] (M = B (K+1) hidden states), W bf16 [V, d] (the output embedding),
// fp32 accumulation on the fifth-generation tensor cores.  Operator fusion
// of the verification into the target's last layer is named by
// "推测解码采样验证优化策略 —— 深度调研报告", part 1 section 6 (扩展性与安全性,
// 算子融合).  The logits are rounded to bf16 and stored (the surviving row is
// read again by the draw stream), and the epilogue also forms, from the
// rounded values, each row's (max, normaliser) of softmax(z / T) over the
// tile's 256 vocabulary ids -- the row pass's statistics -- so the logits are
// never streamed back in for them.
//
// Persistent, on pairs of SMs: a cluster of two CTAs (one per SM of a
// pair) walks the 256 x 256 output tiles, rows fastest, so the pairs
// running at one time share a few tiles of W and find them in L2.  The
// pair's MMA is one tcgen05.mma of M 256 (128 rows in each CTA's tensor
// memory), N 256, K 16, issued by the even CTA; each CTA loads its own 128
// rows of h and its half (128 ids) of the tile of W, so a stage holds
// 32 KiB per SM and the ring has 6 stages.
// Warp 0: the producer, 2-D tensor-memory-accelerator loads of 64-wide K
// slices (128-byte swizzle), both CTAs' copies completing on the even CTA's
// "full" barrier.  Warp 1: allocates all 512 tensor-memory columns of both
// SMs (two fp32 accumulators of 256 columns, one lane per row); in the even
// CTA one thread issues the MMAs, each stage's MMAs committed to both CTAs'
// "empty" barriers and each finished tile to both CTAs' accumulator "full"
// barriers.  Warps 2..5 of each CTA: the epilogue of its 128 rows,
// tcgen05.ld of the accumulator (warp w reads lanes 32 (w mod 4) .. +31),
// bf16 rounding, stores, the tile statistics; they hand the accumulator back
// (to the even CTA's "empty" barrier) while the next tile's MMAs already run
// in the other one.
// Every mbarrier wait is bounded in time; a wait that runs out sets
// SV_INTERNAL_TIMEOUT, the CTA stops issuing, gives the copies and MMAs in
// flight time to complete (the even CTA waits for its MMAs, bounded), and
// both CTAs free their tensor memory and return together.
#pragma once

#include <cuda.h>

#include "sv_rows.cuh"

namespace sv {

constexpr int kLmBM = 128;                       // rows of h per CTA (256 per pair)
constexpr int kLmBN = 256;                       // vocabulary ids per tile (128 loaded by each CTA)
constexpr int kLmBK = 64;                        // hidden dims per stage: one 128-byte swizzle row
constexpr int kLmStages = 6;
constexpr int kLmABytes = kLmBM * kLmBK * 2;     // 16 KiB
constexpr int kLmBBytes = kLmBN / 2 * kLmBK * 2; // 16 KiB: this CTA's half of the tile of W
constexpr int kLmStageBytes = kLmABytes + kLmBBytes;
constexpr int kLmThreads = 192;                  // producer, MMA, 4 epilogue warps
constexpr int kLmEpiWarps = 4;
constexpr int kLmSmem = kLmStages * kLmStageBytes + 1024; // + alignment of the swizzled tiles
constexpr uint32_t kLmTmemCols = 2 * kLmBN;     // two fp32 accumulators: all 512 columns

struct LmParams {
    int32_t M, N, Kd;  // rows of h, vocabulary, hidden size
    int32_t MT;        // 256-row tiles along M
    uint16_t *logits;  // [M, N] bf16 out
    float2 *part;      // [M, NT] (max, normaliser relative to fl(max c)) per 256-id tile, or nullptr
    int32_t NT;        // tiles along N
    float c;           // log2(e) / T
    int32_t vec;       // N % 8 == 0 and 16-byte aligned logits: vector stores
    int32_t *status;
    uint64_t wait_ns;
};

// ------------------------------------------------------------- primitives

__device__ __forceinline__ uint64_t lm_ns()
{
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ uint32_t lm_cluster_rank()
{
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

// the shared::cluster address of the same shared-memory location in CTA `rank`
__device__ __forceinline__ uint32_t lm_mapa(uint32_t saddr, uint32_t rank)
{
    uint32_t d;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(d) : "r"(saddr), "r"(rank));
    return d;
}

__device__ __forceinline__ void lm_cluster_sync()
{
    asm volatile("barrier.cluster.arrive.release;\n\tbarrier.cluster.wait.acquire;" ::: "memory");
}

__device__ __forceinline__ void lm_mbar_init(uint32_t bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void lm_mbar_expect(uint32_t bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}

// one arrival on a barrier of either CTA of the cluster
__device__ __forceinline__ void lm_mbar_arrive_cluster(uint32_t cluster_bar)
{
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_bar) : "memory");
}

__device__ __forceinline__ bool lm_mbar_test(uint32_t bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile("{\n\t.reg .pred p;\n\t"
                 "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
                 "selp.u32 %0, 1, 0, p;\n\t}"
                 : "=r"(ok)
                 : "r"(bar), "r"(parity)
                 : "memory");
    return ok != 0;
}

// Wait for phase `parity` of `bar`; false after limit_ns or once *stop is set.
__device__ __forceinline__ bool lm_wait(uint32_t bar, uint32_t parity, const volatile int *stop, uint64_t limit_ns)
{
    if (lm_mbar_test(bar, parity))
        return true;
    const uint64_t t0 = lm_ns();
    for (;;) {
#pragma unroll 1
        for (int i = 0; i < 16; ++i)
            if (lm_mbar_test(bar, parity))
                return true;
        if ((stop && *stop) || lm_ns() - t0 > limit_ns)
            return false;
    }
}

// 2-D tiled tensor load (box from the map) into this CTA's shared memory at
// `dst`, completing on `cluster_bar` (a barrier of either CTA of the pair);
// c0 (the inner, hidden coordinate) is a multiple of 64 elements.
__device__ __forceinline__ void lm_tma_2d(uint32_t dst, const CUtensorMap *map, int32_t c0, int32_t c1,
                                          uint32_t cluster_bar)
{
    asm volatile("cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes"
                 " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
                 "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(cluster_bar)
                 : "memory");
}

// tensor memory of both CTAs of the pair; each CTA's warp takes part
__device__ __forceinline__ void lm_tmem_alloc(uint32_t dst_smem, uint32_t ncols)
{
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem), "r"(ncols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void lm_tmem_dealloc(uint32_t taddr, uint32_t ncols)
{
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

__device__ __forceinline__ void lm_tc_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void lm_tc_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// The pair's D[tmem] (+)= A[smem] B[smem]^T, both K-major: A's 256 rows are
// the two CTAs' 128, B's 256 rows the two CTAs' halves; the descriptors'
// addresses are taken in both CTAs' shared memory.
__device__ __forceinline__ void lm_mma(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc, uint32_t acc)
{
    asm volatile("{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
                 "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
                 "l"(adesc), "l"(bdesc), "r"(idesc), "r"(acc)
                 : "memory");
}

// The barrier at this shared-memory offset in both CTAs gets one arrival
// once every MMA this thread issued before is done.
__device__ __forceinline__ void lm_commit_both(uint32_t bar)
{
    asm volatile("tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::
                     "r"(bar), "h"(static_cast<uint16_t>(3))
                 : "memory");
}

// the same, for a barrier of this CTA only
__device__ __forceinline__ void lm_commit_local(uint32_t bar)
{
    asm volatile("tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar) : "memory");
}

// 32 consecutive fp32 columns of this thread's tensor-memory lane
__device__ __forceinline__ void lm_tmem_ld32(uint32_t taddr, uint32_t (&r)[32])
{
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x32.b32 "
                 "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
                 "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
                   "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]),
                   "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]),
                   "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]),
                   "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
                 : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// Shared-memory matrix descriptor of a K-major tile in the 128-byte swizzle
// layout the tensor loads write: rows of 64 bf16 (128 bytes), 8-row groups
// 1024 bytes apart (stride byte offset); the leading byte offset is unused
// for this layout (one MMA's K = 16 stays inside a swizzle row); descriptor
// version 1; the tile base is 1024-byte aligned (base offset 0).
__device__ __forceinline__ uint64_t lm_desc(uint32_t saddr)
{
    uint64_t d = 0;
    d |= static_cast<uint64_t>((saddr >> 4) & 0x3FFFu);
    d |= static_cast<uint64_t>(1u) << 16;           // leading byte offset 16 (unused)
    d |= static_cast<uint64_t>(1024u >> 4) << 32;   // stride byte offset
    d |= static_cast<uint64_t>(1u) << 46;           // descriptor version
    d |= static_cast<uint64_t>(2u) << 61;           // 128-byte swizzle
    return d;
}

// Instruction descriptor: D fp32, A and B bf16, both K-major, N = 256, M = 256 (the pair).
constexpr uint32_t kLmIdesc = (1u << 4) | (1u << 7) | (1u << 10) | ((static_cast<uint32_t>(kLmBN) >> 3) << 17) |
                              ((static_cast<uint32_t>(2 * kLmBM) >> 4) << 24);

__device__ __forceinline__ uint32_t bf16_rn_pair(float lo, float hi)
{
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

// ------------------------------------------------------------- the kernel

// The epilogue of one tile for one warp: its 32 rows (one per lane) of the
// accumulator at tensor-memory address `tl` (lane quarter and column base
// applied).  Pass 1 rounds to bf16, stores, and takes each row's maximum;
// pass 2 (with P.part) sums the softmax terms against that maximum.
__device__ __forceinline__ void lm_epilogue_tile(const LmParams &P, uint32_t tl, int row, int n0, int tile_n)
{
    const bool rok = row < P.M;
    const int ncols = P.N - n0 < kLmBN ? P.N - n0 : kLmBN;
    uint16_t *lrow = P.logits + static_cast<int64_t>(row) * P.N + n0;
    float mx = -INFINITY;
#pragma unroll 1
    for (int cb = 0; cb < kLmBN / 32; ++cb) {
        uint32_t v[32];
        lm_tmem_ld32(tl + cb * 32, v);
        uint32_t pk[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            pk[i] = bf16_rn_pair(__uint_as_float(v[2 * i]), __uint_as_float(v[2 * i + 1]));
            const int col = cb * 32 + 2 * i;
            if (col < ncols)
                mx = fmaxf(mx, __uint_as_float(pk[i] << 16));
            if (col + 1 < ncols)
                mx = fmaxf(mx, __uint_as_float(pk[i] & 0xFFFF0000u));
        }
        if (rok) {
            const int c0 = cb * 32;
            if (P.vec && c0 + 32 <= ncols) {
                uint4 *dst = reinterpret_cast<uint4 *>(lrow + c0);
#pragma unroll
                for (int q = 0; q < 4; ++q)
                    dst[q] = make_uint4(pk[4 * q], pk[4 * q + 1], pk[4 * q + 2], pk[4 * q + 3]);
            } else {
#pragma unroll
                for (int i = 0; i < 32; ++i)
                    if (c0 + i < ncols)
                        lrow[c0 + i] = static_cast<uint16_t>(i & 1 ? pk[i >> 1] >> 16 : pk[i >> 1] & 0xFFFFu);
            }
        }
    }
    if (!P.part)
        return;
    const float mc = mc_of(mx, P.c);
    float S = 0.0f;
#pragma unroll 1
    for (int cb = 0; cb < kLmBN / 32; ++cb) {
        uint32_t v[32];
        lm_tmem_ld32(tl + cb * 32, v);
#pragma unroll
        for (int i = 0; i < 32; i += 2) {
            const uint32_t pk = bf16_rn_pair(__uint_as_float(v[i]), __uint_as_float(v[i + 1]));
            const int col = cb * 32 + i;
            if (col < ncols)
                S += term(__uint_as_float(pk << 16), P.c, mc);
            if (col + 1 < ncols)
                S += term(__uint_as_float(pk & 0xFFFF0000u), P.c, mc);
        }
    }
    if (rok)
        P.part[static_cast<int64_t>(row) * P.NT + tile_n] = make_float2(mx, S);
}

// Launched in clusters of two CTAs, one CTA per SM; the grid is a whole
// number of pairs.  Pair p takes tiles p, p + pairs, ...; tile t covers rows
// 256 (t mod MT) and vocabulary ids 256 (t div MT).
__global__ void __launch_bounds__(kLmThreads, 1)
    lm_head_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB, const LmParams P)
{
    extern __shared__ uint8_t lm_smem_raw[];
    __shared__ __align__(8) unsigned long long full[kLmStages], empty[kLmStages], tfull[2], tempty[2], drain;
    __shared__ uint32_t tmem_base;
    __shared__ int stop;
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(lm_smem_raw) + 1023) & ~uintptr_t{1023});
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t rank = lm_cluster_rank();
    const bool leader = rank == 0;
    const int64_t pair = blockIdx.x >> 1, pairs = gridDim.x >> 1;
    const int nk = (P.Kd + kLmBK - 1) / kLmBK;
    const int64_t ntiles = static_cast<int64_t>(P.MT) * P.NT;
    const volatile int *vstop = &stop;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kLmStages; ++s) {
            lm_mbar_init(smem_addr(&full[s]), 1);  // the even CTA's arrival with both CTAs' bytes
            lm_mbar_init(smem_addr(&empty[s]), 1); // the pair's MMAs of the stage
        }
        for (int a = 0; a < 2; ++a) {
            lm_mbar_init(smem_addr(&tfull[a]), 1);
            lm_mbar_init(smem_addr(&tempty[a]), 2 * kLmEpiWarps); // every epilogue warp of the pair
        }
        lm_mbar_init(smem_addr(&drain), 1);
        stop = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 1)
        lm_tmem_alloc(smem_addr(&tmem_base), kLmTmemCols);
    lm_tc_before();
    __syncthreads();
    lm_cluster_sync(); // both CTAs' barriers exist before either CTA signals the other's
    lm_tc_after();
    const uint32_t tbase = tmem_base;
    auto fail = [&]() {
        if (!stop) {
            stop = 1;
            if (P.status)
                atomicOr(P.status, kTimeout);
        }
    };

    if (warp == 0 && lane == 0) {
        // stage s, its phase, and the even CTA's "full" barrier of stage 0
        // (the barriers are consecutive 8-byte words)
        int s = 0;
        uint32_t ph = 0;
        int64_t it = 0;
        const uint32_t fb0 = lm_mapa(smem_addr(&full[0]), 0);
        const uint32_t sbase = smem_addr(smem);
        for (int64_t t = pair; t < ntiles && !*vstop; t += pairs) {
            const int m0 = static_cast<int>(t % P.MT) * (2 * kLmBM) + static_cast<int>(rank) * kLmBM;
            const int n0 = static_cast<int>(t / P.MT) * kLmBN + static_cast<int>(rank) * (kLmBN / 2);
            int kb = 0;
            for (; kb < nk; ++kb, ++it) {
                if (it >= kLmStages && !lm_wait(smem_addr(&empty[s]), ph ^ 1u, vstop, P.wait_ns)) {
                    fail();
                    break;
                }
                const uint32_t sa = sbase + static_cast<uint32_t>(s * kLmStageBytes);
                const uint32_t fb = fb0 + static_cast<uint32_t>(s * 8);
                if (leader)
                    lm_mbar_expect(smem_addr(&full[s]), 2 * kLmStageBytes);
                lm_tma_2d(sa, &tmA, kb * kLmBK, m0, fb);
                lm_tma_2d(sa + kLmABytes, &tmB, kb * kLmBK, n0, fb);
                if (++s == kLmStages) {
                    s = 0;
                    ph ^= 1u;
                }
            }
            if (kb < nk)
                break;
        }
    } else if (warp == 1 && lane == 0 && leader) {
        // the descriptors of stage 0's A and B tiles; a stage or a K step
        // only moves the start address (16-byte units, the low field)
        const uint64_t ad0 = lm_desc(smem_addr(smem)), bd0 = lm_desc(smem_addr(smem + kLmABytes));
        int s = 0;
        uint32_t ph = 0;
        int i = 0;
        for (int64_t t = pair; t < ntiles && !*vstop; t += pairs, ++i) {
            const int acc = i & 1;
            if (i >= 2 &&
                !lm_wait(smem_addr(&tempty[acc]), static_cast<uint32_t>(((i >> 1) & 1) ^ 1), vstop, P.wait_ns)) {
                fail();
                break;
            }
            lm_tc_after();
            const uint32_t tacc = tbase + static_cast<uint32_t>(acc * kLmBN);
            int kb = 0;
            for (; kb < nk; ++kb) {
                if (!lm_wait(smem_addr(&full[s]), ph, vstop, P.wait_ns)) {
                    fail();
                    break;
                }
                lm_tc_after();
                const uint64_t so = static_cast<uint64_t>((s * kLmStageBytes) >> 4);
#pragma unroll
                for (int k = 0; k < kLmBK / 16; ++k)
                    lm_mma(tacc, ad0 + so + static_cast<uint64_t>(k * 2), bd0 + so + static_cast<uint64_t>(k * 2),
                           kLmIdesc, (kb | k) ? 1u : 0u);
                lm_commit_both(smem_addr(&empty[s])); // both CTAs' stage is free once these MMAs have read it
                if (++s == kLmStages) {
                    s = 0;
                    ph ^= 1u;
                }
            }
            if (kb < nk)
                break;
            lm_commit_both(smem_addr(&tfull[acc])); // the accumulator is complete in both CTAs
        }
    } else if (warp >= 2) {
        const int lq = warp & 3; // tensor-memory lane quarter this warp may read
        int i = 0;
        for (int64_t t = pair; t < ntiles; t += pairs, ++i) {
            const int acc = i & 1;
            // every lane waits (acquiring the barrier's phase itself); the
            // verdict is made warp-uniform, as tcgen05.ld is warp-collective
            const bool ok = __all_sync(0xFFFFFFFFu, lm_wait(smem_addr(&tfull[acc]),
                                                            static_cast<uint32_t>((i >> 1) & 1), vstop, P.wait_ns));
            if (!ok) {
                if (lane == 0)
                    fail();
                break;
            }
            lm_tc_after();
            const int row = static_cast<int>(t % P.MT) * (2 * kLmBM) + static_cast<int>(rank) * kLmBM + lq * 32 + lane;
            const int tn = static_cast<int>(t / P.MT);
            lm_epilogue_tile(P, tbase + (static_cast<uint32_t>(lq * 32) << 16) + static_cast<uint32_t>(acc * kLmBN),
                             row, tn * kLmBN, tn);
            lm_tc_before();
            __syncwarp();
            if (lane == 0) // this warp has read the accumulator: the MMAs may overwrite it
                lm_mbar_arrive_cluster(lm_mapa(smem_addr(&tempty[acc]), 0));
        }
    }
    // ---- teardown: copies and MMAs in flight complete before the memory goes
    lm_tc_before();
    __syncthreads();
    if (stop) {
        if (threadIdx.x == 0) { // copies issued before the stop land within microseconds
            const uint64_t t0 = lm_ns();
            while (lm_ns() - t0 < 50000ull) {
            }
        }
        if (warp == 1 && lane == 0 && leader) { // every MMA issued is done
            lm_commit_local(smem_addr(&drain));
            (void)lm_wait(smem_addr(&drain), 0u, nullptr, P.wait_ns);
        }
    }
    __syncthreads();
    lm_cluster_sync(); // neither CTA's memory goes while the pair's MMAs or signals may still use it
    if (warp == 1) {
        lm_tc_after();
        lm_tmem_dealloc(tbase, kLmTmemCols);
    }
}

// ------------------------------------------------------------- merge

// The row statistics and draft data for the draw stream, one warp per row:
// the row's per-tile (max, normaliser) pairs merged into one (slot 0 of the
// row's partials), and its draft token, z(x) (from the stored logits), q(x)
// and uniform.
template <bool DENSE>
__global__ void __launch_bounds__(256) lm_merge_kernel(const Params P, float2 *part, int32_t NT)
{
    const int lane = threadIdx.x & 31;
    const int64_t r = static_cast<int64_t>(blockIdx.x) * 8 + (threadIdx.x >> 5);
    const int64_t R = P.B * (static_cast<int64_t>(P.K) + 1);
    if (r < R) { // warp-uniform
        float M = -INFINITY, S = 0.0f;
        for (int32_t i = lane; i < NT; i += 32) {
            const float2 pr = part[r * NT + i];
            part[r * NT + i] = make_float2(0.0f, 0.0f); // the workspace goes back to zero once read
            merge_ms(M, S, pr.x, pr.y, P.c);
        }
        warp_merge_ms(M, S, P.c);
        if (lane == 0) {
            P.row_part[r * P.PM] = make_float2(M, S);
            const RowSide sd = fetch_side<uint16_t, DENSE>(P, r);
            P.row_side[r] = make_float4(__int_as_float(sd.x), sd.zx, sd.qx, sd.u);
        }
    }
    pdl_launch_dependents();
}

} // namespace sv
