// sv_rows.cuh -- the row pass of the verification step.
//
// Every one of the B*(K+1) target rows is streamed once from HBM with 16-byte
// loads.  A row is cut into S1 chunks, one CTA per chunk; each thread keeps an
// online (max, normaliser) pair of softmax(z / T) in the base-2 form
// sum_i exp2(z_i * c - fl(M * c)), c = log2(e) / T (one exp2 per element).
// The CTA that finishes a row last merges the chunk partials and runs the
// accept test of the draft that row verifies: a = min(1, p(x) / q(x)),
// accept iff u < a ("推测解码：草稿、验证与实际加速", section
// 接受与拒绝怎样保住分布, equation for a(x); the replay in section
// 算完三个 token 的全部概率 accepts when the draw is strictly below the
// threshold).  The row finisher that completes a sequence last finds the
// first rejection j* and writes the accepted prefix; later drafts are void
// (same page, section 候选已知，验证才能并行).  No thread ever waits for
// another CTA: completion is detected with arrival counters, and each
// counter is returned to zero by the CTA that saw it complete.
#pragma once

#include "sv_device.cuh"

namespace sv {

__device__ __forceinline__ uint8_t ld_cg_u8(const uint8_t *p)
{
    uint16_t v;
    asm volatile("ld.global.cg.u8 %0, [%1];" : "=h"(v) : "l"(p) : "memory");
    return static_cast<uint8_t>(v);
}

// Fold a group of N elements into the running (M, S) of one thread.
template <int N>
__device__ __forceinline__ void online_group(const float (&z)[N], float &M, float &S, float c)
{
    float gm = z[0];
#pragma unroll
    for (int i = 1; i < N; ++i)
        gm = fmaxf(gm, z[i]);
    if (gm > M) {
        // rescale what was summed against the old maximum
        S = (M == -INFINITY) ? __fmul_rn(S, 0.0f)
                             : __fmul_rn(S, exp2f(mc_of(M, c) - mc_of(gm, c)));
        M = gm;
    }
    const float mc = mc_of(M, c);
#pragma unroll
    for (int i = 0; i < N; ++i)
        S = __fadd_rn(S, term(z[i], c, mc));
}

__device__ __forceinline__ void warp_merge_ms(float &M, float &S, float c)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        float M2 = __shfl_xor_sync(0xFFFFFFFFu, M, o);
        float S2 = __shfl_xor_sync(0xFFFFFFFFu, S, o);
        merge_ms(M, S, M2, S2, c);
    }
}

template <typename LT>
__device__ __forceinline__ void decode16(const uint4 w, float *z)
{
    if constexpr (sizeof(LT) == 2) {
        z[0] = bf16_lo(w.x); z[1] = bf16_hi(w.x);
        z[2] = bf16_lo(w.y); z[3] = bf16_hi(w.y);
        z[4] = bf16_lo(w.z); z[5] = bf16_hi(w.z);
        z[6] = bf16_lo(w.w); z[7] = bf16_hi(w.w);
    } else {
        z[0] = __uint_as_float(w.x); z[1] = __uint_as_float(w.y);
        z[2] = __uint_as_float(w.z); z[3] = __uint_as_float(w.w);
    }
}

// Per sequence: first rejection, accepted prefix, flags.  One warp.
template <bool DENSE>
__device__ void finish_sequence(const Params &P, int64_t b, int lane)
{
    const int32_t K = P.K;
    __threadfence();
    const int32_t bad = __ldcg(&P.seq_bad[b]);
    int32_t jstar = K;
    for (int32_t k0 = 0; k0 < K; k0 += 32) {
        const int32_t k = k0 + lane;
        const bool rej = (k < K) && ld_cg_u8(&P.acc[b * K + k]) == 0;
        const unsigned m = __ballot_sync(0xFFFFFFFFu, rej);
        if (m) {
            jstar = k0 + __ffs(m) - 1;
            break;
        }
    }
    // hand the surviving row's maximum to the draw, clear the per-row state
    const float m_sel = __ldcg(&P.row_m[b * (K + 1) + (jstar < K ? jstar : K)]);
    __syncwarp();
    for (int32_t j = lane; j <= K; j += 32)
        P.row_m[b * (K + 1) + j] = 0.0f;
    for (int32_t k = lane; k < K; k += 32)
        P.acc[b * K + k] = 0;
    int32_t *out = P.out_tokens + b * (K + 1);
    if (bad) {
        for (int32_t k = lane; k <= K; k += 32)
            out[k] = -1;
        for (int32_t k = lane; k < K; k += 32) {
            if (P.accept_flags) P.accept_flags[b * K + k] = -1;
            if (P.accept_prob) P.accept_prob[b * K + k] = 0.0f;
        }
        if (lane == 0) {
            P.num_emitted[b] = 0;
            if (P.residual_mass) P.residual_mass[b] = 0.0f;
            P.seq_jstar[b] = -1;
            if (P.status) atomicOr(P.status, bad);
        }
    } else {
        for (int32_t k = lane; k <= K; k += 32)
            out[k] = k < jstar ? P.tokens[b * K + k] : -1;
        if (P.accept_flags)
            for (int32_t k = lane; k < K; k += 32)
                P.accept_flags[b * K + k] = k < jstar ? 1 : (k == jstar ? 0 : -1);
        if (lane == 0) {
            P.num_emitted[b] = jstar + 1;
            P.seq_jstar[b] = jstar;
            P.seq_m[b] = m_sel;
        }
    }
    if (lane == 0) {
        P.seq_cnt[b] = 0u;
        P.seq_bad[b] = 0;
    }
}

// The last CTA of row r merges the chunk partials and tests the draft.
// One warp.
template <typename LT, bool DENSE>
__device__ void finish_row(const Params &P, int64_t r, int lane)
{
    __threadfence();
    const float c = P.c;
    const int32_t K = P.K, V = P.V;
    float M = -INFINITY, S = 0.0f;
    for (int32_t i = lane; i < P.S1; i += 32) {
        const float2 pr = __ldcg(&P.row_part[r * P.S1 + i]);
        P.row_part[r * P.S1 + i] = make_float2(0.0f, 0.0f);
        merge_ms(M, S, pr.x, pr.y, c);
    }
    warp_merge_ms(M, S, c);

    const int64_t b = r / (K + 1);
    const int32_t j = static_cast<int32_t>(r - b * (K + 1));
    int last_seq = 0;
    if (lane == 0) {
        int32_t bad = 0;
        const bool row_ok = isfinite(M) && isfinite(S);
        if (!row_ok)
            bad |= kBadRow;
        const float uj = P.u[b * (K + 1) + j];
        if (!(uj >= 0.0f && uj < 1.0f))
            bad |= kBadU;
        P.row_m[r] = M;
        P.row_cnt[r] = 0u;
        if (j < K) {
            const int32_t x = P.tokens[b * K + j];
            float a = 0.0f;
            uint8_t acc = 0;
            if (x < 0 || x >= V) {
                bad |= kBadToken;
            } else {
                const float qx = DENSE ? __ldg(&P.q[(b * K + j) * static_cast<int64_t>(V) + x]) : 1.0f;
                if (DENSE && !(qx > 0.0f && isfinite(qx)))
                    bad |= kBadQ;
                else if (row_ok) {
                    const LT *row = static_cast<const LT *>(P.logits) + r * static_cast<int64_t>(V);
                    const float px = __fdiv_rn(term(load_elem<LT>(row + x), c, mc_of(M, c)), S);
                    a = fminf(1.0f, __fdiv_rn(px, qx));
                    acc = uj < a ? 1 : 0;
                }
            }
            P.acc[b * K + j] = acc;
            if (P.accept_prob)
                P.accept_prob[b * K + j] = a;
        }
        if (bad)
            atomicOr(&P.seq_bad[b], bad);
        __threadfence();
        last_seq = atomicAdd(&P.seq_cnt[b], 1u) == static_cast<unsigned>(K);
    }
    last_seq = __shfl_sync(0xFFFFFFFFu, last_seq, 0);
    if (last_seq)
        finish_sequence<DENSE>(P, b, lane);
}

template <typename LT, bool DENSE>
__global__ void __launch_bounds__(kRowThreads) rows_kernel(const Params P)
{
    constexpr int VW = 16 / sizeof(LT); // elements per 16-byte vector
    constexpr int U = 4;                // vectors in flight per thread
    constexpr int NW = kRowThreads / 32;
    __shared__ float sM[NW], sS[NW];
    __shared__ int s_last;

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int64_t item = blockIdx.x;
    const int64_t r = item / P.S1;
    const int32_t ch = static_cast<int32_t>(item - r * P.S1);
    const int32_t V = P.V;
    const float c = P.c;
    const LT *row = static_cast<const LT *>(P.logits) + r * static_cast<int64_t>(V);

    // split the row into a scalar head (until 16-byte aligned), whole
    // vectors (shared out over the S1 chunks) and a scalar tail
    const uintptr_t addr = reinterpret_cast<uintptr_t>(row);
    int32_t head = static_cast<int32_t>(((16u - (addr & 15u)) & 15u) / sizeof(LT));
    if (head > V)
        head = V;
    const int32_t nvec = (V - head) / VW;
    const int32_t tail0 = head + nvec * VW;
    const int32_t v0 = static_cast<int32_t>(static_cast<int64_t>(nvec) * ch / P.S1);
    const int32_t v1 = static_cast<int32_t>(static_cast<int64_t>(nvec) * (ch + 1) / P.S1);
    const LT *vbase = row + head;

    float M = -INFINITY, S = 0.0f;
    const uint4 neg_inf = sizeof(LT) == 2 ? make_uint4(0xFF80FF80u, 0xFF80FF80u, 0xFF80FF80u, 0xFF80FF80u)
                                          : make_uint4(0xFF800000u, 0xFF800000u, 0xFF800000u, 0xFF800000u);
    for (int32_t v = v0 + tid; v < v1; v += U * kRowThreads) {
        uint4 w[U];
#pragma unroll
        for (int k = 0; k < U; ++k) {
            const int32_t vv = v + k * kRowThreads;
            w[k] = vv < v1 ? ld_stream_v4(vbase + static_cast<int64_t>(vv) * VW) : neg_inf;
        }
        float z[U * VW];
#pragma unroll
        for (int k = 0; k < U; ++k)
            decode16<LT>(w[k], z + k * VW);
        online_group<U * VW>(z, M, S, c);
    }
    if (ch == 0)
        for (int32_t i = tid; i < head; i += kRowThreads) {
            const float z[1] = {load_elem<LT>(row + i)};
            online_group<1>(z, M, S, c);
        }
    if (ch == P.S1 - 1)
        for (int32_t i = tail0 + tid; i < V; i += kRowThreads) {
            const float z[1] = {load_elem<LT>(row + i)};
            online_group<1>(z, M, S, c);
        }

    warp_merge_ms(M, S, c);
    if (lane == 0) {
        sM[warp] = M;
        sS[warp] = S;
    }
    __syncthreads();
    if (warp == 0) {
        M = lane < NW ? sM[lane] : -INFINITY;
        S = lane < NW ? sS[lane] : 0.0f;
        warp_merge_ms(M, S, c);
        if (lane == 0) {
            P.row_part[item] = make_float2(M, S);
            __threadfence();
            s_last = atomicAdd(&P.row_cnt[r], 1u) == static_cast<unsigned>(P.S1 - 1);
        }
    }
    __syncthreads();
    if (s_last && warp == 0)
        finish_row<LT, DENSE>(P, r, lane);
}

} // namespace sv
