// spec_verify.cu -- C ABI of the verification library: argument checks,
// workspace layout, and the launches on the caller's stream -- the row
// pass, the draw stream and, when the draw stream does not fill the GPU,
// the final draws -- each chained to the one before by programmatic
// dependent launch; and the top-k / top-p filter.  The operations
// themselves are documented in spec_verify.h.
#include "spec_verify.h"

#include <cmath>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>
#include <mutex>

#include "sv_filter.cuh"
#include "sv_final.cuh"
#include "sv_lmhead.cuh"
#include "sv_tree.cuh"
#include "sv_rows.cuh"

namespace {

constexpr size_t kAlign = 256;

size_t align_up(size_t v) { return (v + kAlign - 1) / kAlign * kAlign; }

int ceil_log2_u64(uint64_t v)
{
    int n = 0;
    while ((uint64_t{1} << n) < v)
        ++n;
    return n;
}

int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

// How the work of one call is cut and where its scratch lives: a function of
// (B, K, V) only.
struct Plan {
    int64_t R;    // rows B*(K+1)
    int32_t PM;   // row_part slots per row
    int32_t CPS;  // final-draw chunks per sequence
    int32_t fix;  // fractional bits of the fixed-point masses
    size_t off_part, off_row_side, off_seq_info, off_seqE, off_cnt, off_rec_a, off_rec_q, bytes;
};

bool make_plan(int64_t B, int32_t K, int32_t V, Plan &p)
{
    if (B < 0 || K < 0 || V < 1 || V > SV_MAX_V)
        return false;
    if (B > 0 && static_cast<int64_t>(K) + 1 > INT64_MAX / B)
        return false;
    p.R = B * (static_cast<int64_t>(K) + 1);
    if (p.R > 0 && V > INT64_MAX / p.R)
        return false;
    // row_part slots per row: enough for any cut of the flat row array into
    // at most kRowMaxCtas spans (the launch widens spans to keep to it)
    p.PM = static_cast<int32_t>(p.R > 0 ? ceil_div(sv::kRowMaxCtas, p.R) + 3 : 4);
    p.CPS = static_cast<int32_t>(ceil_div(V, static_cast<int64_t>(sv::kChunkGroups) * sv::kGroup));
    const int fb = 62 - ceil_log2_u64(static_cast<uint64_t>(V) + 1);
    p.fix = fb < 40 ? fb : 40;
    const size_t Bz = static_cast<size_t>(B), R = static_cast<size_t>(p.R);
    size_t off = 0;
    p.off_part = off;     off = align_up(off + R * p.PM * sizeof(float2));
    p.off_row_side = off; off = align_up(off + R * sizeof(float4));
    p.off_seq_info = off; off = align_up(off + Bz * sizeof(int4));
    p.off_seqE = off;     off = align_up(off + Bz * sizeof(long long));
    p.off_cnt = off;      off = align_up(off + Bz * sizeof(uint32_t));
    p.off_rec_a = off;    off = align_up(off + Bz * p.CPS * sizeof(long long));
    p.off_rec_q = off;    off = align_up(off + Bz * p.CPS * sizeof(float));
    p.bytes = off;
    return true;
}

bool aligned(const void *p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

enum Stage { kRows = 1, kSurvivors = 2, kBoth = 3 };

constexpr uint64_t kWaitLimitNs = 1000000000ull; // every bounded wait of a kernel gives up after 1 s

constexpr int kMaxDevices = 64;

// The current context's process-unique id, or 0 when none can be had (no
// context current yet, or a driver without the query).  The driver calls
// are reached through the runtime's entry-point lookup, so the library does
// not link the driver library itself.
unsigned long long current_context_id()
{
    using GetCurrent = CUresult (*)(CUcontext *);
    using GetId = CUresult (*)(CUcontext, unsigned long long *);
    static GetCurrent get_current = nullptr;
    static GetId get_id = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 4000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_current = reinterpret_cast<GetCurrent>(f);
        f = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_id = reinterpret_cast<GetId>(f);
        (void)cudaGetLastError();
    });
    if (!get_current || !get_id)
        return 0;
    CUcontext ctx = nullptr;
    unsigned long long id = 0;
    if (get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr || get_id(ctx, &id) != CUDA_SUCCESS)
        return 0;
    return id;
}

// Per device and kernel instantiation: how many CTAs of each kernel fit on
// the device at once (the grids of the persistent kernels).  Cached per
// device for the context the figures were taken in: a context created anew
// (after cudaDeviceReset, or a caller's own context) has forgotten the draw
// kernel's shared-memory attribute, so the figures are taken again there.
struct Resident {
    int rows, draw;
    unsigned long long ctx; // context id the entry was made in (0: none)
};

template <typename LT, bool DENSE>
cudaError_t resident_ctas(Resident &out)
{
    static std::mutex mu;
    static Resident cache[kMaxDevices] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return e;
    if (dev < 0 || dev >= kMaxDevices)
        return cudaErrorInvalidDevice;
    const unsigned long long ctx = current_context_id();
    std::lock_guard<std::mutex> lock(mu);
    if (cache[dev].rows == 0 || cache[dev].ctx == 0 || cache[dev].ctx != ctx) {
        int sms = 0, rows = 0, draw = 0;
        e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess)
            return e;
        e = cudaFuncSetAttribute(sv::survivor_kernel<LT, DENSE>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 sv::DrawShape<LT, DENSE>::kCtaBytes);
        if (e != cudaSuccess)
            return e;
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&rows, sv::rows_kernel<LT, DENSE>, sv::kRowCtaThreads, 0);
        if (e != cudaSuccess)
            return e;
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&draw, sv::survivor_kernel<LT, DENSE>,
                                                          sv::kDrawWarps * 32, sv::DrawShape<LT, DENSE>::kCtaBytes);
        if (e != cudaSuccess)
            return e;
        sms = sms > 0 ? sms : 1;
        cache[dev].rows = (rows > 0 ? rows : 1) * sms;
        cache[dev].draw = (draw > 0 ? draw : 1) * sms;
        cache[dev].ctx = current_context_id(); // taken after the calls above made the context current
    }
    out = cache[dev];
    return cudaSuccess;
}

int64_t clamp_grid(int64_t want, int64_t cap) { return want < 1 ? 1 : (want > cap ? cap : want); }

// CTAs of the draw stream: at least one chunk per warp, at most one wave
int64_t draw_grid(int64_t NC, const Resident &res) { return clamp_grid(ceil_div(NC, sv::kDrawWarps), res.draw); }

// A stream that fills every SM, with at least as many draw warps as
// sequences: each sequence has its own warps, and the last of them makes its
// final draw (no final kernel, whose CTAs would only be placed once the
// stream's CTAs leave).  A smaller stream leaves SMs free, where the final
// kernel's CTAs wait for it and draw with block-wide scans, sooner than one
// warp can.
bool inline_final(int64_t grid, int64_t B, const Resident &res)
{
    return grid == res.draw && grid * sv::kDrawWarps >= B;
}

// Kernels one whole call launches on the current device: the row pass, the
// draw stream and, unless the stream makes the final draws, the final kernel.
template <typename LT, bool DENSE>
cudaError_t launches_per_call(int64_t B, const Plan &plan, int32_t &n)
{
    Resident res;
    const cudaError_t e = resident_ctas<LT, DENSE>(res);
    if (e != cudaSuccess)
        return e;
    const int64_t grid = draw_grid(B * static_cast<int64_t>(plan.CPS), res);
    n = inline_final(grid, B, res) ? 2 : 3;
    return cudaSuccess;
}

template <typename LT, bool DENSE>
cudaError_t launch(sv::Params &P, const Plan &plan, int stages, cudaStream_t stream)
{
    if (stages == 0)
        return cudaSuccess;
    Resident res;
    cudaError_t e = resident_ctas<LT, DENSE>(res);
    if (e != cudaSuccess)
        return e;
    // the flat view of the logits and its cut into one span per CTA
    constexpr int64_t VW = 16 / sizeof(LT);
    P.total = plan.R * P.V;
    P.h = static_cast<int64_t>((16 - reinterpret_cast<uintptr_t>(P.logits) % 16) % 16) / static_cast<int64_t>(sizeof(LT));
    if (P.h > P.total)
        P.h = P.total;
    P.nvec = (P.total - P.h) / VW;
    P.NV = P.nvec + 2;
    {
        int64_t want = clamp_grid(ceil_div(P.NV, sv::kRowMinSpan), res.rows < sv::kRowMaxCtas ? res.rows : sv::kRowMaxCtas);
        if (want < ceil_div(P.NV, sv::kRowMaxSpan))
            want = ceil_div(P.NV, sv::kRowMaxSpan); // offsets inside a span stay in int
        int64_t span = ceil_div(P.NV, want);
        // a row touches at most `touch` vectors; spans of at least
        // touch / (PM - 2) vectors put it in at most PM - 1 CTAs
        const int64_t touch = ceil_div(P.V, VW) + 2;
        const int64_t span_min = ceil_div(touch, plan.PM - 2);
        P.span = span > span_min ? span : span_min;
    }
    if (stages & kRows) {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(static_cast<unsigned>(ceil_div(P.NV, P.span)));
        cfg.blockDim = dim3(sv::kRowCtaThreads);
        cfg.stream = stream;
        e = cudaLaunchKernelEx(&cfg, sv::rows_kernel<LT, DENSE>, P);
        if (e != cudaSuccess)
            return e;
    }
    if (stages & kSurvivors) {
        const int64_t grid = draw_grid(P.NC, res);
        P.inline_final = inline_final(grid, P.B, res) ? 1 : 0;
        // programmatic dependent launch: the draw's CTAs may be scheduled
        // while the row pass drains; they wait in griddepcontrol.wait for
        // its completion before reading anything it wrote
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(static_cast<unsigned>(grid));
        cfg.blockDim = dim3(sv::kDrawWarps * 32);
        cfg.dynamicSmemBytes = sv::DrawShape<LT, DENSE>::kCtaBytes;
        cfg.stream = stream;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        e = cudaLaunchKernelEx(&cfg, sv::survivor_kernel<LT, DENSE>, P);
        if (e != cudaSuccess)
            return e;
        if (P.inline_final)
            return cudaSuccess;
        // the final draws: one CTA per sequence, chained the same way
        cudaLaunchConfig_t fcfg = {};
        fcfg.gridDim = dim3(static_cast<unsigned>(P.B < 0x7FFFFFFF ? P.B : 0x7FFFFFFF));
        fcfg.blockDim = dim3(sv::kFinalThreads);
        fcfg.dynamicSmemBytes = static_cast<size_t>(plan.CPS) * (sizeof(long long) + sizeof(float));
        fcfg.stream = stream;
        fcfg.attrs = attr;
        fcfg.numAttrs = 1;
        e = cudaLaunchKernelEx(&fcfg, sv::final_kernel<LT, DENSE>, P);
        if (e != cudaSuccess)
            return e;
    }
    return cudaSuccess;
}

sv_status_t run(int stages, const void *logits, sv_dtype_t dtype, const float *q, const int32_t *tokens,
                const float *u, float T, int64_t B, int32_t K, int32_t V, int32_t *out_tokens,
                int32_t *num_emitted, int8_t *accept_flags, float *accept_prob, float *residual_mass,
                int32_t *status_dev, void *workspace, size_t workspace_bytes, void *stream,
                unsigned long long *stats = nullptr, int one_part = 0)
{
    if (B < 0 || K < 0 || V < 1)
        return SV_EINVAL;
    if (V > SV_MAX_V)
        return SV_EUNSUPPORTED;
    if (dtype != SV_BF16 && dtype != SV_FP32)
        return SV_EINVAL;
    if (!std::isfinite(T) || !(T > 0.0f))
        return SV_EINVAL;
    const double c64 = 1.4426950408889634074 / static_cast<double>(T);
    const float c = static_cast<float>(c64);
    if (!std::isfinite(c) || !(c > 0.0f))
        return SV_EINVAL;
    if (!logits || !u || !out_tokens || !num_emitted || (K > 0 && !tokens) || !workspace)
        return SV_EINVAL;
    const size_t esize = dtype == SV_BF16 ? 2 : 4;
    if (!aligned(logits, esize) || (q && !aligned(q, 4)) || (tokens && !aligned(tokens, 4)) ||
        !aligned(u, 4) || !aligned(out_tokens, 4) || !aligned(num_emitted, 4) ||
        (accept_prob && !aligned(accept_prob, 4)) || (residual_mass && !aligned(residual_mass, 4)) ||
        (status_dev && !aligned(status_dev, 4)) || (stats && !aligned(stats, 8)) || !aligned(workspace, kAlign))
        return SV_EINVAL;
    Plan plan;
    if (!make_plan(B, K, V, plan))
        return SV_EUNSUPPORTED;
    if (workspace_bytes < plan.bytes)
        return SV_EINVAL;
    if (B == 0)
        return SV_OK;

    char *ws = static_cast<char *>(workspace);
    sv::Params P;
    P.logits = logits;
    P.q = K > 0 ? q : nullptr;
    P.tokens = tokens;
    P.u = u;
    P.c = c;
    P.B = B;
    P.K = K;
    P.V = V;
    P.out_tokens = out_tokens;
    P.num_emitted = num_emitted;
    P.accept_flags = accept_flags;
    P.accept_prob = accept_prob;
    P.residual_mass = residual_mass;
    P.status = status_dev;
    P.stats = stats;
    P.row_part = reinterpret_cast<float2 *>(ws + plan.off_part);
    P.row_side = reinterpret_cast<float4 *>(ws + plan.off_row_side);
    P.seq_info = reinterpret_cast<int4 *>(ws + plan.off_seq_info);
    P.seq_E = reinterpret_cast<long long *>(ws + plan.off_seqE);
    P.seq_cnt = reinterpret_cast<uint32_t *>(ws + plan.off_cnt);
    P.inline_final = 0;
    P.rec_a = reinterpret_cast<long long *>(ws + plan.off_rec_a);
    P.rec_q = reinterpret_cast<float *>(ws + plan.off_rec_q);
    P.PM = plan.PM;
    P.CPS = plan.CPS;
    P.NC = B * static_cast<int64_t>(plan.CPS);
    P.ring_ok = (V % sv::kGroup) == 0 && aligned(logits, 16) && (P.q == nullptr || aligned(P.q, 16)) ? 1 : 0;
    P.fix_bits = plan.fix;
    P.one_part = one_part;
    P.total = P.h = P.nvec = P.NV = P.span = 0;

    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e;
    const bool dense = P.q != nullptr;
    if (dtype == SV_BF16)
        e = dense ? launch<uint16_t, true>(P, plan, stages, s) : launch<uint16_t, false>(P, plan, stages, s);
    else
        e = dense ? launch<float, true>(P, plan, stages, s) : launch<float, false>(P, plan, stages, s);
    return e == cudaSuccess ? SV_OK : SV_ECUDA;
}

// ---------------------------------------------------------------- LM head

constexpr int64_t kLmMaxRows = int64_t{1} << 30;

int32_t lm_tiles(int32_t V) { return static_cast<int32_t>(ceil_div(V, sv::kLmBN)); }

size_t lm_part_bytes(int64_t M, int32_t V) { return align_up(static_cast<size_t>(M) * lm_tiles(V) * sizeof(float2)); }

// A 2-D tensor map of a row-major bf16 matrix [rows, cols] with boxes of
// box_rows x 64 elements in the 128-byte swizzle layout; out-of-range
// elements read as zero.  Reached through the runtime's entry-point lookup.
bool lm_tensor_map(CUtensorMap *map, const void *base, int64_t rows, int32_t cols, uint32_t box_rows)
{
    using Encode = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
    static Encode encode = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            encode = reinterpret_cast<Encode>(f);
        (void)cudaGetLastError();
    });
    if (!encode)
        return false;
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(cols) * 2};
    const cuuint32_t box[2] = {static_cast<cuuint32_t>(sv::kLmBK), box_rows};
    const cuuint32_t estr[2] = {1, 1};
    return encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

sv_status_t lm_check(const void *hidden, const void *lm_head, int64_t M, int32_t d, int32_t V, const void *logits)
{
    if (M < 0 || d < 8 || d % 8 != 0 || V < 1)
        return SV_EINVAL;
    if (V > SV_MAX_V || M > kLmMaxRows)
        return SV_EUNSUPPORTED;
    if (M > 0 && (!hidden || !lm_head || !logits || !aligned(hidden, 16) || !aligned(lm_head, 16) ||
                  !aligned(logits, 2)))
        return SV_EINVAL;
    return SV_OK;
}

// How many clusters of two LM-head CTAs fit on the current device at once
// (the persistent grid, in pairs); cached per device for the context it was
// taken in, like the verification kernels' figures.
cudaError_t lm_pairs(int &pairs)
{
    struct Entry {
        int pairs;
        unsigned long long ctx;
    };
    static std::mutex mu;
    static Entry cache[kMaxDevices] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return e;
    if (dev < 0 || dev >= kMaxDevices)
        return cudaErrorInvalidDevice;
    const unsigned long long ctx = current_context_id();
    std::lock_guard<std::mutex> lock(mu);
    if (cache[dev].pairs == 0 || cache[dev].ctx == 0 || cache[dev].ctx != ctx) {
        e = cudaFuncSetAttribute(sv::lm_head_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, sv::kLmSmem);
        if (e != cudaSuccess)
            return e;
        int sms = 0;
        e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess)
            return e;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = 2;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(static_cast<unsigned>(sms > 1 ? sms & ~1 : 2));
        cfg.blockDim = dim3(sv::kLmThreads);
        cfg.dynamicSmemBytes = sv::kLmSmem;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        int n = 0;
        e = cudaOccupancyMaxActiveClusters(&n, sv::lm_head_kernel, &cfg);
        if (e != cudaSuccess)
            return e;
        if (n < 1)
            return cudaErrorInvalidConfiguration;
        cache[dev].pairs = n;
        cache[dev].ctx = current_context_id();
    }
    pairs = cache[dev].pairs;
    return cudaSuccess;
}

// logits = h W^T (bf16 out) and, with `part`, the per-tile row statistics.
cudaError_t lm_launch(const void *hidden, const void *lm_head, int64_t M, int32_t d, int32_t V, void *logits,
                      float2 *part, float c, int32_t *status, cudaStream_t stream)
{
    CUtensorMap ta, tb;
    if (!lm_tensor_map(&ta, hidden, M, d, sv::kLmBM) || !lm_tensor_map(&tb, lm_head, V, d, sv::kLmBN / 2))
        return cudaErrorInvalidValue;
    int pairs = 0;
    cudaError_t e = lm_pairs(pairs);
    if (e != cudaSuccess)
        return e;
    sv::LmParams L;
    L.M = static_cast<int32_t>(M);
    L.N = V;
    L.Kd = d;
    L.MT = static_cast<int32_t>(ceil_div(M, 2 * sv::kLmBM));
    L.logits = static_cast<uint16_t *>(logits);
    L.part = part;
    L.NT = lm_tiles(V);
    L.c = c;
    L.vec = (V % 8 == 0 && aligned(logits, 16)) ? 1 : 0;
    L.status = status;
    L.wait_ns = kWaitLimitNs;
    // persistent: as many pairs of SMs as hold a cluster at once (the ring
    // takes most of the shared memory: one CTA per SM)
    const int64_t tiles = static_cast<int64_t>(L.MT) * L.NT;
    const int64_t np = tiles < pairs ? tiles : pairs;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(2 * np));
    cfg.blockDim = dim3(sv::kLmThreads);
    cfg.dynamicSmemBytes = sv::kLmSmem;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, sv::lm_head_kernel, ta, tb, L);
}

static_assert(sv::kTreeMaxNodes == SV_MAX_TREE_NODES, "tree size limit");
static_assert(sv::kBadTree == SV_BAD_TREE, "status bit");

} // namespace

extern "C" {

size_t sv_workspace_bytes(int64_t B, int32_t K, int32_t V)
{
    Plan p;
    if (!make_plan(B, K, V, p))
        return 0;
    return p.bytes;
}

sv_status_t spec_verify(const void *target_logits, sv_dtype_t logits_dtype, const float *draft_probs,
                        const int32_t *draft_tokens, const float *uniforms, float temperature, int64_t B,
                        int32_t K, int32_t V, int32_t *out_tokens, int32_t *num_emitted, int8_t *accept_flags,
                        float *accept_prob, float *residual_mass, int32_t *status_dev, void *workspace,
                        size_t workspace_bytes, void *stream)
{
    return run(kBoth, target_logits, logits_dtype, draft_probs, draft_tokens, uniforms, temperature, B, K, V,
               out_tokens, num_emitted, accept_flags, accept_prob, residual_mass, status_dev, workspace,
               workspace_bytes, stream);
}

sv_status_t spec_verify_stats(const void *target_logits, sv_dtype_t logits_dtype, const float *draft_probs,
                              const int32_t *draft_tokens, const float *uniforms, float temperature, int64_t B,
                              int32_t K, int32_t V, int32_t *out_tokens, int32_t *num_emitted, int8_t *accept_flags,
                              float *accept_prob, float *residual_mass, int32_t *status_dev, void *workspace,
                              size_t workspace_bytes, uint64_t *stats_dev, void *stream)
{
    if (!stats_dev)
        return SV_EINVAL;
    return run(kBoth, target_logits, logits_dtype, draft_probs, draft_tokens, uniforms, temperature, B, K, V,
               out_tokens, num_emitted, accept_flags, accept_prob, residual_mass, status_dev, workspace,
               workspace_bytes, stream, reinterpret_cast<unsigned long long *>(stats_dev));
}

sv_status_t sv_verify_rows(const void *target_logits, sv_dtype_t logits_dtype, const float *draft_probs,
                           const int32_t *draft_tokens, const float *uniforms, float temperature, int64_t B,
                           int32_t K, int32_t V, int32_t *out_tokens, int32_t *num_emitted, int8_t *accept_flags,
                           float *accept_prob, float *residual_mass, int32_t *status_dev, void *workspace,
                           size_t workspace_bytes, void *stream)
{
    return run(kRows, target_logits, logits_dtype, draft_probs, draft_tokens, uniforms, temperature, B, K, V,
               out_tokens, num_emitted, accept_flags, accept_prob, residual_mass, status_dev, workspace,
               workspace_bytes, stream);
}

sv_status_t sv_sample_survivors(const void *target_logits, sv_dtype_t logits_dtype, const float *draft_probs,
                                const int32_t *draft_tokens, const float *uniforms, float temperature, int64_t B,
                                int32_t K, int32_t V, int32_t *out_tokens, int32_t *num_emitted,
                                int8_t *accept_flags, float *accept_prob, float *residual_mass,
                                int32_t *status_dev, void *workspace, size_t workspace_bytes, void *stream)
{
    return run(kSurvivors, target_logits, logits_dtype, draft_probs, draft_tokens, uniforms, temperature, B, K,
               V, out_tokens, num_emitted, accept_flags, accept_prob, residual_mass, status_dev, workspace,
               workspace_bytes, stream);
}

sv_status_t sv_kernel_launches(sv_dtype_t logits_dtype, int32_t dense, int64_t B, int32_t K, int32_t V,
                               int32_t *launches)
{
    if (!launches || B < 0 || K < 0 || V < 1 || (logits_dtype != SV_BF16 && logits_dtype != SV_FP32))
        return SV_EINVAL;
    if (V > SV_MAX_V)
        return SV_EUNSUPPORTED;
    Plan plan;
    if (!make_plan(B, K, V, plan))
        return SV_EUNSUPPORTED;
    if (B == 0) {
        *launches = 0;
        return SV_OK;
    }
    const bool d = dense != 0 && K > 0; // K = 0 has no draft probabilities to read
    int32_t n = 0;
    cudaError_t e;
    if (logits_dtype == SV_BF16)
        e = d ? launches_per_call<uint16_t, true>(B, plan, n) : launches_per_call<uint16_t, false>(B, plan, n);
    else
        e = d ? launches_per_call<float, true>(B, plan, n) : launches_per_call<float, false>(B, plan, n);
    if (e != cudaSuccess)
        return SV_ECUDA;
    *launches = n;
    return SV_OK;
}

sv_status_t sv_filter_logits(const void *logits, sv_dtype_t logits_dtype, int64_t rows, int32_t V,
                             float temperature, int32_t top_k, float top_p, void *out_logits, int32_t *kept,
                             int32_t *status_dev, void *stream)
{
    if (rows < 0 || V < 1 || (logits_dtype != SV_BF16 && logits_dtype != SV_FP32))
        return SV_EINVAL;
    if (V > SV_MAX_V)
        return SV_EUNSUPPORTED;
    if (!std::isfinite(temperature) || !(temperature > 0.0f) || !(top_p > 0.0f))
        return SV_EINVAL;
    const float c = static_cast<float>(1.4426950408889634074 / static_cast<double>(temperature));
    if (!std::isfinite(c) || !(c > 0.0f))
        return SV_EINVAL;
    const size_t esize = logits_dtype == SV_BF16 ? 2 : 4;
    if (rows > 0 && (!logits || !out_logits))
        return SV_EINVAL;
    if (!aligned(logits, esize) || !aligned(out_logits, esize) || (kept && !aligned(kept, 4)) ||
        (status_dev && !aligned(status_dev, 4)))
        return SV_EINVAL;
    if (rows > 0 && static_cast<int64_t>(V) > INT64_MAX / rows)
        return SV_EUNSUPPORTED;
    if (rows == 0)
        return SV_OK;
    sv::FilterParams F;
    F.in = logits;
    F.out = out_logits;
    F.rows = rows;
    F.V = V;
    F.c = c;
    F.top_k = top_k;
    F.top_p = top_p;
    const int fb = 62 - ceil_log2_u64(static_cast<uint64_t>(V) + 1);
    F.fb = fb < 40 ? fb : 40;
    F.yscale = static_cast<float>(sv::kYBins) / static_cast<float>(F.fb + 2);
    F.vec = aligned(logits, 16) && aligned(out_logits, 16) && (static_cast<size_t>(V) * esize) % 16 == 0 ? 1 : 0;
    F.kept = kept;
    F.status = status_dev;
    int dev = 0, sms = 0, per_sm = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess)
        e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e == cudaSuccess)
        e = logits_dtype == SV_BF16
                ? cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, sv::filter_kernel<uint16_t>,
                                                                sv::kFilterThreads, 0)
                : cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, sv::filter_kernel<float>,
                                                                sv::kFilterThreads, 0);
    if (e != cudaSuccess)
        return SV_ECUDA;
    const int64_t resident = static_cast<int64_t>(sms > 0 ? sms : 1) * (per_sm > 0 ? per_sm : 1);
    const int64_t grid = rows < resident ? rows : resident;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (logits_dtype == SV_BF16)
        sv::filter_kernel<uint16_t><<<static_cast<unsigned>(grid), sv::kFilterThreads, 0, s>>>(F);
    else
        sv::filter_kernel<float><<<static_cast<unsigned>(grid), sv::kFilterThreads, 0, s>>>(F);
    return cudaGetLastError() == cudaSuccess ? SV_OK : SV_ECUDA;
}

size_t sv_lm_head_workspace_bytes(int64_t B, int32_t K, int32_t V)
{
    Plan p;
    if (!make_plan(B, K, V, p))
        return 0;
    return p.bytes + lm_part_bytes(B * (static_cast<int64_t>(K) + 1), V);
}

sv_status_t sv_lm_head_logits(const void *hidden, const void *lm_head, int64_t M, int32_t d, int32_t V,
                              void *logits, int32_t *status_dev, void *stream)
{
    const sv_status_t st = lm_check(hidden, lm_head, M, d, V, logits);
    if (st != SV_OK || M == 0)
        return st;
    if (status_dev && !aligned(status_dev, 4))
        return SV_EINVAL;
    return lm_launch(hidden, lm_head, M, d, V, logits, nullptr, 1.0f, status_dev, static_cast<cudaStream_t>(stream)) ==
                   cudaSuccess
               ? SV_OK
               : SV_ECUDA;
}

sv_status_t spec_verify_lm_head(const void *hidden, const void *lm_head, int32_t d, const float *draft_probs,
                                const int32_t *draft_tokens, const float *uniforms, float temperature, int64_t B,
                                int32_t K, int32_t V, void *logits_out, int32_t *out_tokens, int32_t *num_emitted,
                                int8_t *accept_flags, float *accept_prob, float *residual_mass, int32_t *status_dev,
                                void *workspace, size_t workspace_bytes, void *stream)
{
    if (B < 0 || K < 0)
        return SV_EINVAL;
    if (B > 0 && static_cast<int64_t>(K) + 1 > kLmMaxRows / B)
        return SV_EUNSUPPORTED;
    const int64_t M = B * (static_cast<int64_t>(K) + 1);
    sv_status_t st = lm_check(hidden, lm_head, M, d, V, logits_out);
    if (st != SV_OK)
        return st;
    Plan plan;
    if (!make_plan(B, K, V, plan))
        return SV_EUNSUPPORTED;
    if (!workspace || workspace_bytes < plan.bytes + lm_part_bytes(M, V))
        return SV_EINVAL;
    // host checks of the verification (nothing launched yet)
    st = run(0, logits_out, SV_BF16, draft_probs, draft_tokens, uniforms, temperature, B, K, V, out_tokens,
             num_emitted, accept_flags, accept_prob, residual_mass, status_dev, workspace, plan.bytes, stream);
    if (st != SV_OK || B == 0)
        return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    float2 *part = reinterpret_cast<float2 *>(static_cast<char *>(workspace) + plan.bytes);
    const float c = static_cast<float>(1.4426950408889634074 / static_cast<double>(temperature));
    if (lm_launch(hidden, lm_head, M, d, V, logits_out, part, c, status_dev, s) != cudaSuccess)
        return SV_ECUDA;
    // the row statistics and draft data, then the draw stream and final draws
    {
        sv::Params P = {};
        P.logits = logits_out;
        P.q = K > 0 ? draft_probs : nullptr;
        P.tokens = draft_tokens;
        P.u = uniforms;
        P.c = c;
        P.B = B;
        P.K = K;
        P.V = V;
        P.row_part = reinterpret_cast<float2 *>(static_cast<char *>(workspace) + plan.off_part);
        P.row_side = reinterpret_cast<float4 *>(static_cast<char *>(workspace) + plan.off_row_side);
        P.PM = plan.PM;
        const unsigned grid = static_cast<unsigned>(ceil_div(M, 8));
        if (P.q)
            sv::lm_merge_kernel<true><<<grid, 256, 0, s>>>(P, part, lm_tiles(V));
        else
            sv::lm_merge_kernel<false><<<grid, 256, 0, s>>>(P, part, lm_tiles(V));
        if (cudaGetLastError() != cudaSuccess)
            return SV_ECUDA;
    }
    return run(kSurvivors, logits_out, SV_BF16, draft_probs, draft_tokens, uniforms, temperature, B, K, V, out_tokens,
               num_emitted, accept_flags, accept_prob, residual_mass, status_dev, workspace, plan.bytes, stream,
               nullptr, 1);
}

size_t sv_tree_workspace_bytes(int64_t B, int32_t N, int32_t V)
{
    Plan p;
    if (N < 1 || N > SV_MAX_TREE_NODES || !make_plan(B, N - 1, V, p))
        return 0;
    return p.bytes;
}

sv_status_t spec_verify_tree(const void *logits, sv_dtype_t dtype, const float *draft_probs, const int32_t *parent,
                             const int32_t *tokens, const float *uniforms, float temperature, int64_t B, int32_t N,
                             int32_t V, int32_t *out_tokens, int32_t *out_nodes, int32_t *num_emitted,
                             float *accept_prob, int32_t *status_dev, void *workspace, size_t workspace_bytes,
                             void *stream)
{
    if (B < 0 || N < 1 || V < 1)
        return SV_EINVAL;
    if (N > SV_MAX_TREE_NODES || V > SV_MAX_V || B > 0x3FFFFFFFll)
        return SV_EUNSUPPORTED;
    if (dtype != SV_BF16 && dtype != SV_FP32)
        return SV_EINVAL;
    if (!std::isfinite(temperature) || !(temperature > 0.0f))
        return SV_EINVAL;
    const float c = static_cast<float>(1.4426950408889634074 / static_cast<double>(temperature));
    if (!std::isfinite(c) || !(c > 0.0f))
        return SV_EINVAL;
    if (!logits || !draft_probs || !parent || !tokens || !uniforms || !out_tokens || !num_emitted || !workspace)
        return SV_EINVAL;
    const size_t esize = dtype == SV_BF16 ? 2 : 4;
    if (!aligned(logits, esize) || !aligned(draft_probs, 4) || !aligned(parent, 4) || !aligned(tokens, 4) ||
        !aligned(uniforms, 4) || !aligned(out_tokens, 4) || !aligned(num_emitted, 4) ||
        (out_nodes && !aligned(out_nodes, 4)) || (accept_prob && !aligned(accept_prob, 4)) ||
        (status_dev && !aligned(status_dev, 4)) || !aligned(workspace, kAlign))
        return SV_EINVAL;
    Plan plan;
    if (!make_plan(B, N - 1, V, plan))
        return SV_EUNSUPPORTED;
    if (workspace_bytes < plan.bytes)
        return SV_EINVAL;
    if (B == 0)
        return SV_OK;
    char *ws = static_cast<char *>(workspace);
    sv::Params P = {};
    P.logits = logits;
    P.q = nullptr; // the row pass takes no draft data here; the tree kernel reads q
    P.tokens = tokens;
    P.u = uniforms;
    P.c = c;
    P.B = B;
    P.K = N - 1;
    P.V = V;
    P.row_part = reinterpret_cast<float2 *>(ws + plan.off_part);
    P.row_side = reinterpret_cast<float4 *>(ws + plan.off_row_side);
    P.PM = plan.PM;
    P.fix_bits = plan.fix;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    // the row pass over all B*N rows: every row's (max, normaliser) partials
    cudaError_t e = dtype == SV_BF16 ? launch<uint16_t, false>(P, plan, kRows, s)
                                     : launch<float, false>(P, plan, kRows, s);
    if (e != cudaSuccess)
        return SV_ECUDA;
    sv::TreeArgs A;
    A.parent = parent;
    A.tokens = tokens;
    A.q = draft_probs;
    A.u = uniforms;
    A.N = N;
    A.out_tokens = out_tokens;
    A.out_nodes = out_nodes;
    A.num_emitted = num_emitted;
    A.accept_prob = accept_prob;
    A.status = status_dev;
    // one cluster of two CTAs per sequence
    const size_t smem = static_cast<size_t>(ceil_div(V, sv::kTreeChunk)) * sizeof(long long);
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = sv::kTreeCtas;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    // programmatic dependent launch: the walk checks its inputs while the row
    // pass drains and waits in griddepcontrol.wait before reading its partials
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(B * sv::kTreeCtas));
    cfg.blockDim = dim3(sv::kTreeThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    if (dtype == SV_BF16) {
        if (smem > 48 * 1024 &&
            cudaFuncSetAttribute(sv::tree_kernel<uint16_t>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(smem)) != cudaSuccess)
            return SV_ECUDA;
        e = cudaLaunchKernelEx(&cfg, sv::tree_kernel<uint16_t>, P, A);
    } else {
        if (smem > 48 * 1024 &&
            cudaFuncSetAttribute(sv::tree_kernel<float>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(smem)) != cudaSuccess)
            return SV_ECUDA;
        e = cudaLaunchKernelEx(&cfg, sv::tree_kernel<float>, P, A);
    }
    return e == cudaSuccess ? SV_OK : SV_ECUDA;
}

const char *sv_status_string(sv_status_t status)
{
    switch (status) {
    case SV_OK:
        return "SV_OK: work enqueued";
    case SV_EINVAL:
        return "SV_EINVAL: invalid argument (null or misaligned pointer, bad size, temperature or workspace)";
    case SV_ECUDA:
        return "SV_ECUDA: a CUDA launch failed";
    case SV_EUNSUPPORTED:
        return "SV_EUNSUPPORTED: size beyond what one call supports";
    }
    return "unknown sv_status_t";
}

} // extern "C"

// ---------------------------------------------------------------------------
// Allocation-free entry point.  Some callers cannot hand the library a
// workspace: a server whose device memory is reserved up front by its own
// pool and that forbids cudaMalloc on the request path, or a plugin interface
// that passes a plugin its input and output buffers but no allocator.  For
// them, spec_verify_noalloc runs the same kernels with their scratch in a
// fixed-size array that lives in the library's device image.  The array is
// shared by every call on a device and keeps the last call's contents, so
// each call clears the bytes it needs before launching; calls that overlap on
// the GPU (two streams, two host threads) race on it.
#include <mutex>

namespace {
constexpr size_t kNoallocScratchBytes = SV_NOALLOC_SCRATCH_BYTES;
} // namespace

// Every GPU that loads this library holds this array until the process exits.
static __device__ __align__(256) unsigned char g_sv_noalloc_scratch[kNoallocScratchBytes];

namespace {
// The device address of the scratch array in the current context.  In host
// code the array's name is only a stand-in, so the address is looked up
// with the device current, on every call: the lookup is host-side and
// cheap, and a kept address would go stale when the context is destroyed
// and made again (cudaDeviceReset), which places the module anew.
sv_status_t noalloc_scratch(void **out)
{
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_sv_noalloc_scratch) != cudaSuccess || p == nullptr) {
        (void)cudaGetLastError();
        return SV_ECUDA;
    }
    *out = p;
    return SV_OK;
}
} // namespace

extern "C" sv_status_t spec_verify_noalloc(const void *target_logits, sv_dtype_t logits_dtype,
                                           const float *draft_probs, const int32_t *draft_tokens,
                                           const float *uniforms, float temperature, int64_t B, int32_t K,
                                           int32_t V, int32_t *out_tokens, int32_t *num_emitted,
                                           int8_t *accept_flags, float *accept_prob, float *residual_mass,
                                           int32_t *status_dev, void *stream)
{
    Plan plan;
    if (make_plan(B, K, V, plan) && plan.bytes > kNoallocScratchBytes)
        return SV_EUNSUPPORTED; // this batch needs more scratch than the array holds
    void *scratch = nullptr;
    sv_status_t st = noalloc_scratch(&scratch);
    if (st != SV_OK)
        return st;
    // host checks only (stage mask 0 launches nothing)
    st = run(0, target_logits, logits_dtype, draft_probs, draft_tokens, uniforms, temperature, B, K, V,
             out_tokens, num_emitted, accept_flags, accept_prob, residual_mass, status_dev, scratch,
             kNoallocScratchBytes, stream);
    if (st != SV_OK || B == 0)
        return st;
    // the kernels expect zeroed scratch; a previous call may not have finished cleanly
    if (cudaMemsetAsync(scratch, 0, plan.bytes, static_cast<cudaStream_t>(stream)) != cudaSuccess)
        return SV_ECUDA;
    return run(kBoth, target_logits, logits_dtype, draft_probs, draft_tokens, uniforms, temperature, B, K, V,
               out_tokens, num_emitted, accept_flags, accept_prob, residual_mass, status_dev, scratch,
               kNoallocScratchBytes, stream);
}
