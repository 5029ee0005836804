// sv_device.cuh -- device helpers shared by the two kernels of the
// verification step: launch parameters, element decoding, the exact
// fixed-point accumulation of probability masses, the exact product
// floor(u * Z), warp reductions, and the cluster / distributed-shared-memory
// primitives (inline PTX, sm_90+ cluster model, compiled for sm_103a).
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace sv {

constexpr int kRowThreads = 256;  // threads of a row-pass CTA
constexpr int kSurvThreads = 256; // threads of a survivor CTA
constexpr int kGroup = 8;         // contiguous elements per survivor thread
constexpr int kMaxTiles = 1024;   // tiles of one survivor CTA (V <= 2^24)
constexpr int kMaxCluster = 8;    // portable cluster size

// Device status bits (the same values the public header documents).
constexpr int32_t kBadU = 1, kBadToken = 2, kBadQ = 4, kBadRow = 8,
                  kDegenerate = 16;

struct Params {
    const void *logits;
    const float *q;        // nullptr: one-hot drafts
    const int32_t *tokens; // [B, K]
    const float *u;        // [B, K+1]
    float c;               // log2(e) / T
    int64_t B;
    int32_t K, V;
    int32_t *out_tokens;
    int32_t *num_emitted;
    int8_t *accept_flags;
    float *accept_prob;
    float *residual_mass;
    int32_t *status;
    // workspace views
    float2 *row_part;  // [R * S1]  (max of z, sum of exp2 relative to it)
    uint32_t *row_cnt; // [R]       arrival counters, left at zero
    float *row_m;      // [R]       max of z over the row
    float *seq_m;      // [B]       max of z over the row of the final draw
    uint8_t *acc;      // [B * K]   1 = accepted
    uint32_t *seq_cnt; // [B]       arrival counters, left at zero
    int32_t *seq_bad;  // [B]       status bits of the sequence, left at zero
    int32_t *seq_jstar;// [B]       row the final token is drawn from, -1 = bad
    // Every workspace word is returned to zero by its last reader, so a call
    // leaves the whole workspace zero-filled.
    int32_t S1;        // chunks per row in the row pass
    int32_t CL;        // cluster size of the survivor pass
    int32_t fix_bits;  // fractional bits of the fixed-point masses
};

// ------------------------------------------------------------ element loads

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

template <typename LT> __device__ __forceinline__ float load_elem(const LT *p);
template <> __device__ __forceinline__ float load_elem<uint16_t>(const uint16_t *p)
{
    return __uint_as_float(static_cast<uint32_t>(__ldg(p)) << 16);
}
template <> __device__ __forceinline__ float load_elem<float>(const float *p)
{
    return __ldg(p);
}

// 16-byte streaming load that does not allocate in L1.
__device__ __forceinline__ uint4 ld_stream_v4(const void *p)
{
    uint4 r;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "l"(p));
    return r;
}

// ------------------------------------------------------- softmax normaliser

// y-space offset of a running maximum M: fl(M * c), or 0 while nothing but
// -inf has been seen (then every finite-free term is exp2(-inf) = 0 and a
// NaN still propagates).
__device__ __forceinline__ float mc_of(float M, float c)
{
    return M == -INFINITY ? 0.0f : __fmul_rn(M, c);
}

// One softmax term relative to the offset mc: exp2(z*c - mc).
__device__ __forceinline__ float term(float z, float c, float mc)
{
    return exp2f(__fmaf_rn(z, c, -mc));
}

// Merge two partial (max, sum) pairs of the online softmax normaliser.
__device__ __forceinline__ void merge_ms(float &M, float &S, float M2, float S2, float c)
{
    float Mn = fmaxf(M, M2);
    float mn = mc_of(Mn, c);
    float f1 = (M == -INFINITY) ? 0.0f : exp2f(mc_of(M, c) - mn);
    float f2 = (M2 == -INFINITY) ? 0.0f : exp2f(mc_of(M2, c) - mn);
    S = __fadd_rn(__fmul_rn(S, f1), __fmul_rn(S2, f2));
    M = Mn;
}

// --------------------------------------------------- exact fixed-point mass

// A probability mass w in [0, 2] as an integer multiple of 2^-fix_bits.
// w * 2^fix_bits is exact in fp32 (a power-of-two scale); the conversion
// rounds to nearest.  Sums of these integers are exact and independent of
// the order of summation.
__device__ __forceinline__ long long to_fixed(float w, float scale)
{
    return __float2ll_rn(__fmul_rn(w, scale));
}

// floor(u * Z) exactly, for u in [0, 1) (fp32) and 0 <= Z < 2^63.
__device__ __forceinline__ unsigned long long floor_mul(float u, unsigned long long Z)
{
    uint32_t bits = __float_as_uint(u);
    uint32_t E = (bits >> 23) & 0xFFu;
    unsigned long long mant = (bits & 0x7FFFFFu) | (E ? 0x800000u : 0u);
    if (mant == 0ull || Z == 0ull)
        return 0ull;
    int shift = 150 - (E ? static_cast<int>(E) : 1); // u = mant * 2^-shift, shift >= 24
    unsigned long long lo = mant * Z;
    unsigned long long hi = __umul64hi(mant, Z);
    if (shift >= 128)
        return 0ull;
    if (shift >= 64)
        return hi >> (shift - 64);
    return (hi << (64 - shift)) | (lo >> shift);
}

// ------------------------------------------------------------ warp helpers

__device__ __forceinline__ long long warp_sum_ll(long long v)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
        v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
    return v;
}

// inclusive scan over the warp
__device__ __forceinline__ long long warp_incl_scan_ll(long long v, int lane)
{
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        long long n = __shfl_up_sync(0xFFFFFFFFu, v, o);
        if (lane >= o)
            v += n;
    }
    return v;
}

// ------------------------------------------------------- cluster primitives

__device__ __forceinline__ uint32_t cluster_ctarank()
{
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

__device__ __forceinline__ void cluster_sync_all()
{
    asm volatile("barrier.cluster.arrive.release.aligned;\n\t"
                 "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Read a 64-bit value from the shared memory of CTA `rank` of the cluster,
// at the address that `local` has in this CTA.
__device__ __forceinline__ long long ld_cluster_ll(const long long *local, uint32_t rank)
{
    uint32_t saddr = static_cast<uint32_t>(__cvta_generic_to_shared(local));
    uint32_t raddr;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(raddr) : "r"(saddr), "r"(rank));
    long long v;
    asm volatile("ld.shared::cluster.s64 %0, [%1];" : "=l"(v) : "r"(raddr) : "memory");
    return v;
}

} // namespace sv
