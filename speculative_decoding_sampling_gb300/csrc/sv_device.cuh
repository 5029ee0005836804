// sv_device.cuh -- device helpers of the verification kernel: launch
// parameters, element decoding, the base-2 online softmax normaliser, exact
// fixed-point masses, warp reductions and the acquire/release flag accesses.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace sv {

// Tuning knobs (defaults measured on GB300; each may be set with -D).
#ifndef SV_ROW_MIN_SPAN
#define SV_ROW_MIN_SPAN 1024 // row pass: fewest 16-byte vectors a CTA streams
#endif
#ifndef SV_ROW_WARPS
#define SV_ROW_WARPS 8    // row pass: streaming warps of a CTA
#endif
#ifndef SV_ROW_U
#define SV_ROW_U 4        // row pass: 16-byte vectors a thread loads per step
#endif
#ifndef SV_ROW_MIN_CTAS
#define SV_ROW_MIN_CTAS 4 // row pass: resident CTAs per SM the register budget is cut for
#endif
#ifndef SV_DRAW_STAGES
#define SV_DRAW_STAGES 3  // final draw: chunks in a warp's async-copy ring
#endif
#ifndef SV_DRAW_WARPS
#define SV_DRAW_WARPS 4   // final draw: warps of a CTA
#endif
#ifndef SV_MIN_CTAS
#define SV_MIN_CTAS 3     // final draw: resident CTAs per SM the register budget is cut for
#endif

constexpr int kThreads = 256;          // threads of a CTA
constexpr int kWarps = kThreads / 32;
constexpr int kRowMinSpan = SV_ROW_MIN_SPAN;
constexpr int kRowMaxCtas = 4096;      // row pass: most CTAs a call's span is cut for
constexpr int kGroup = 8;              // consecutive ids a lane owns in the final draw
constexpr int kChunkTiles = 4;        // warp tiles (32 groups each) of a final-draw chunk
constexpr int kChunkGroups = kChunkTiles * 32; // groups of a chunk (1024 ids)
constexpr int kDrawStages = SV_DRAW_STAGES; // chunks in a draw warp's async-copy ring
constexpr int kDrawWarps = SV_DRAW_WARPS;   // warps of a draw CTA
static_assert(kDrawStages >= 2 && kDrawWarps >= 1 && kDrawWarps <= 32, "draw ring shape");

// Device status bits (the values the public header documents).
constexpr int32_t kBadU = 1, kBadToken = 2, kBadQ = 4, kBadRow = 8, kDegenerate = 16, kTimeout = 32;

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
    unsigned long long *stats; // acceptance statistics (SV_STATS_WORDS(K) counters), or nullptr
    // workspace views; every word is returned to zero by its last reader, so
    // a completed call leaves the whole workspace zero-filled
    float2 *row_part;     // [R * PM]  (max of z, normaliser relative to it) per CTA a row falls in
    float4 *row_side;     // [R]       the row's draft token (int bits), z(x), q(x), u
    int4 *seq_info;       // [B]       the verdict for the final draw: j* (-1 = bad sequence), bits of the
                          //           surviving row's max m and normaliser s, the rejected draft x (one-hot) or -1
    long long *seq_E;     // [B]       exact sum of pt over the surviving row (dense), 2^-fix_bits units
    uint32_t *seq_cnt;    // [B]       draw-stream chunks of the sequence folded so far (inline final draws)
    long long *rec_a;     // [B * CPS] per chunk: mass A, 2^-fix_bits units
    float *rec_q;         // [B * CPS] per chunk: Qp
    int64_t total;        // R * V elements of the logits
    int64_t h;            // elements before the first 16-byte boundary (< 16 / element size)
    int64_t nvec;         // whole 16-byte vectors from there on
    int64_t NV;           // nvec + 2: the flat view's vectors, the two ragged ends included
    int64_t span;         // vectors per row-pass CTA
    int32_t PM;           // row_part slots per row
    int32_t CPS;          // final-draw chunks per sequence
    int64_t NC;           // final-draw chunks of the call, B * CPS
    int32_t ring_ok;      // rows of whole 16-byte aligned groups: the draw streams through its rings
    int32_t inline_final; // every sequence has its own draw warps, the last of which makes its final draw
    int32_t fix_bits;     // fractional bits of the fixed-point masses
    int32_t one_part;     // each row's statistics are one merged pair in slot 0 (the LM-head path)
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




// ------------------------------------------------------- async copies
//
// Each draw warp owns a ring of kDrawStages shared-memory stages.  A lane copies only
// the 16-byte pieces it will read itself, so completion is tracked with the
// lane's own copy groups (cp.async.wait_group) and no lane ever waits for
// another.

__device__ __forceinline__ uint32_t smem_addr(const void *p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void cp_async16(void *dst, const void *src)
{
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_addr(dst)), "l"(src) : "memory");
}

__device__ __forceinline__ void cp_async_commit()
{
    asm volatile("cp.async.commit_group;" ::: "memory");
}

// wait until at most N of this lane's copy groups are still in flight
template <int N> __device__ __forceinline__ void cp_async_wait()
{
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

__device__ __forceinline__ uint4 lds_v4(const void *p)
{
    uint4 r;
    asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "r"(smem_addr(p)));
    return r;
}

// ------------------------------------------------------- softmax normaliser

// 2^x on the special-function unit (flush-to-zero: results below 2^-126
// are far below every mass this library resolves).
__device__ __forceinline__ float ex2(float x)
{
    float y;
    asm volatile("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// y-space offset of a running maximum M: fl(M * c), or 0 while nothing but
// -inf has been seen (then every term is exp2(-inf) = 0 and a NaN still
// propagates).
__device__ __forceinline__ float mc_of(float M, float c)
{
    return M == -INFINITY ? 0.0f : __fmul_rn(M, c);
}

// One softmax term relative to the offset mc: exp2(z*c - mc).
__device__ __forceinline__ float term(float z, float c, float mc)
{
    return ex2(__fmaf_rn(z, c, -mc));
}

// Merge two partial (max, sum) pairs of the online softmax normaliser.
__device__ __forceinline__ void merge_ms(float &M, float &S, float M2, float S2, float c)
{
    const float Mn = fmaxf(M, M2);
    const float mn = mc_of(Mn, c);
    const float f1 = (M == -INFINITY) ? 0.0f : ex2(mc_of(M, c) - mn);
    const float f2 = (M2 == -INFINITY) ? 0.0f : ex2(mc_of(M2, c) - mn);
    S = __fadd_rn(__fmul_rn(S, f1), __fmul_rn(S2, f2));
    M = Mn;
}

// --------------------------------------------------- exact fixed-point mass

// A finite fp32 value w as the nearest integer multiple of 2^-fb (ties to
// even), for |w| * 2^fb < 2^55.  Sums of these integers are exact and
// independent of the order of summation.  x = |w| * 2^fb is exact (a power
// of two scale); it is split as x = hi * 2^32 + lo with hi = trunc(x / 2^32)
// (< 2^23, exact) and lo = x - hi * 2^32 (exact: x has 24 significant bits
// and lo keeps the ones below 2^32), and only lo is rounded, by a 32-bit
// conversion.  The float-to-64-bit-integer conversion instruction is
// avoided on purpose: it runs on the double-precision pipe, which is narrow
// on this GPU.
__device__ __forceinline__ long long to_fixed(float w, int fb)
{
    const float x = __fmul_rn(fabsf(w), __int_as_float((127 + fb) << 23));
    const float hi = truncf(__fmul_rn(x, 2.3283064365386963e-10f)); // x / 2^32
    const float lo = __fmaf_rn(hi, -4294967296.0f, x);
    const long long r = (static_cast<long long>(__float2uint_rz(hi)) << 32) + __float2uint_rn(lo);
    return w < 0.0f ? -r : r;
}

// floor(u * Z) for u in [0, 1) and 0 <= Z < 2^62, exactly: u = mu * 2^-k with
// a 24-bit mu and k >= 24, so u * Z = (mu * Z) / 2^k with a 96-bit product.
__device__ __forceinline__ long long mul_floor(float u, long long Z)
{
    const uint32_t b = __float_as_uint(u);
    const int e = static_cast<int>((b >> 23) & 0xFFu);
    if (e == 0 || Z <= 0)
        return 0; // u = 0 (or subnormal, below 2^-126: u * Z < 1)
    const unsigned long long mu = (b & 0x7FFFFFu) | 0x800000u;
    const int k = 150 - e; // u = mu * 2^-k, k >= 24 for u < 1
    const unsigned long long z = static_cast<unsigned long long>(Z);
    const unsigned long long lo = mu * z, hi = __umul64hi(mu, z);
    if (k >= 128)
        return 0;
    if (k >= 64)
        return static_cast<long long>(hi >> (k - 64));
    return static_cast<long long>((lo >> k) | (hi << (64 - k)));
}

// --------------------------------------------------- packed fp32 pairs
//
// Two fp32 lanes in one 64-bit register pair; each operation rounds both
// halves exactly as the scalar instruction would.

__device__ __forceinline__ unsigned long long pack2(float a, float b)
{
    unsigned long long r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
    return r;
}

__device__ __forceinline__ void unpack2(unsigned long long v, float &a, float &b)
{
    asm("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(v));
}

__device__ __forceinline__ unsigned long long fma2(unsigned long long a, unsigned long long b, unsigned long long c)
{
    unsigned long long r;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
    return r;
}

__device__ __forceinline__ unsigned long long add2(unsigned long long a, unsigned long long b)
{
    unsigned long long r;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}

__device__ __forceinline__ unsigned long long mul2(unsigned long long a, unsigned long long b)
{
    unsigned long long r;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}

// a / b and a % b for 0 <= a, 0 < b < 2^31, in 32-bit arithmetic when a fits
__device__ __forceinline__ int64_t divi(int64_t a, int64_t b)
{
    return a < 0x80000000ll ? static_cast<int64_t>(static_cast<uint32_t>(a) / static_cast<uint32_t>(b)) : a / b;
}

// ------------------------------------------------------ flat logits view
//
// The B*(K+1) rows of V ids are one array of R*V elements.  From the first
// 16-byte boundary on it is cut into whole 16-byte vectors 1..nvec; "vector"
// 0 stands for the h elements before that boundary and vector nvec+1 for the
// ragged end.  Row-pass CTA g owns the vectors [g*span, (g+1)*span).

// The vector holding element e (e - h + VW > 0 since h < VW).
template <typename LT>
__device__ __forceinline__ int64_t vec_of_elem(const Params &P, int64_t e)
{
    constexpr int VW = 16 / sizeof(LT);
    return (e - P.h + VW) / VW;
}

// The row-pass CTAs holding the first and last ids of row r: its partials
// are in slots 0 .. last - first of the row.
template <typename LT>
__device__ __forceinline__ void row_ctas(const Params &P, int64_t r, int64_t &first, int &n_parts)
{
    const int64_t V = P.V;
    first = divi(vec_of_elem<LT>(P, r * V), P.span);
    n_parts = static_cast<int>(divi(vec_of_elem<LT>(P, r * V + V - 1), P.span) - first + 1);
}

// ---------------------------------------------- release/acquire counters
//
// A completion counter bumped with acquire-release semantics: the bump
// releases this thread's earlier writes (partials, records) and, for the
// thread that sees the count complete, acquires everyone else's; no full
// fence is needed on either side.

__device__ __forceinline__ unsigned long long atom_add_acq_rel(unsigned long long *p, unsigned long long v)
{
    unsigned long long old;
    asm volatile("atom.acq_rel.gpu.global.add.u64 %0, [%1], %2;" : "=l"(old) : "l"(p), "l"(v) : "memory");
    return old;
}

__device__ __forceinline__ uint32_t atom_add_acq_rel(uint32_t *p, uint32_t v)
{
    uint32_t old;
    asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
    return old;
}

// ------------------------------------------------- programmatic launch

// Let the next kernel in the stream start launching its CTAs.
__device__ __forceinline__ void pdl_launch_dependents()
{
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Wait until the preceding kernel in the stream has completed and its
// memory is visible (a hardware dependency, not a polling loop).
__device__ __forceinline__ void pdl_wait_primary()
{
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

// ------------------------------------------------------- named barriers

// Arrive at named barrier `id` (expecting `count` threads) without waiting.
__device__ __forceinline__ void bar_arrive(uint32_t id, uint32_t count)
{
    asm volatile("bar.arrive %0, %1;" ::"r"(id), "r"(count) : "memory");
}

// Arrive at named barrier `id` and wait until `count` threads have arrived.
__device__ __forceinline__ void bar_sync(uint32_t id, uint32_t count)
{
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

// ------------------------------------------------------------ warp helpers

__device__ __forceinline__ long long warp_sum_ll(long long v)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
        v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
    return v;
}

// butterfly: every lane computes the same additions, so all lanes agree
__device__ __forceinline__ float warp_sum_f(float v)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
        v = __fadd_rn(v, __shfl_xor_sync(0xFFFFFFFFu, v, o));
    return v;
}

// Sum over the warp of values in [0, 2^58): three pieces (bits 0-20, 21-41,
// 42 on) summed as 32-bit lane values, each sum below 2^27: exact.
__device__ __forceinline__ unsigned long long warp_sum_u64(unsigned long long v)
{
    const uint32_t lo = static_cast<uint32_t>(v), hi = static_cast<uint32_t>(v >> 32);
    const uint32_t p0 = lo & 0x1FFFFFu;
    const uint32_t p1 = __funnelshift_r(lo, hi, 21) & 0x1FFFFFu;
    const uint32_t p2 = hi >> 10;
    const unsigned long long s0 = __reduce_add_sync(0xFFFFFFFFu, p0);
    const unsigned long long s1 = __reduce_add_sync(0xFFFFFFFFu, p1);
    const unsigned long long s2 = __reduce_add_sync(0xFFFFFFFFu, p2);
    return s0 + (s1 << 21) + (s2 << 42);
}

__device__ __forceinline__ long long warp_incl_scan_ll(long long v, int lane)
{
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const long long n = __shfl_up_sync(0xFFFFFFFFu, v, o);
        if (lane >= o)
            v += n;
    }
    return v;
}

} // namespace sv
