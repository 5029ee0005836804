// sv_verdict.cuh -- the per-sequence verdict of the verification step.
//
// From the row pass's partials: each row's (max, normaliser) is the merge of
// its CTAs' pairs, p(x) = exp2(z(x) * c - fl(M * c)) / S; the draft of row j
// is accepted iff u_j < a_j = min(1, p(x) / q(x)) ("推测解码：草稿、验证与实际加速",
// section 接受与拒绝怎样保住分布, equation for a(x); the replay in section
// 算完三个 token 的全部概率 accepts when the draw is strictly below the
// threshold); the first rejected position j* ends the accepted prefix and
// the drafts after it are void (same page, section 候选已知，验证才能并行).  If
// every draft passes, j* = K and the final token comes from row K.
#pragma once

#include "sv_device.cuh"

namespace sv {

struct Verdict {
    int32_t jstar; // row the final token is drawn from (first rejection, or K); -1: bad sequence
    float m, s;    // that row's max of z and fp32 normaliser (relative to fl(m*c))
    int32_t x;     // the rejected draft token (one-hot residual), else -1
};

// The verdict of sequence b.  One warp; lane j takes row j (32 rows at a
// time).  Deterministic: every warp that computes it gets the same answer.
// With `write`, the warp also writes the sequence's accepted prefix, flags,
// accept probabilities, count, status bits, and the surviving row's
// statistics for the final draw (exactly one warp per sequence does).
template <typename LT, bool DENSE>
__device__ Verdict seq_verdict(const Params &P, int64_t b, int lane, bool write)
{
    const int32_t K = P.K;
    const int64_t V = P.V;
    const float c = P.c;
    int32_t jstar = K, bad = 0, xsel = -1;
    bool found = false;
    float m_sel = 0.0f, s_sel = 0.0f;
    for (int32_t j0 = 0; j0 <= K; j0 += 32) {
        const int32_t j = j0 + lane;
        float M = -INFINITY, S = 0.0f, a = 0.0f;
        int32_t x = -1;
        bool rej = false;
        int32_t rbad = 0;
        if (j <= K) {
            const int64_t r = b * (K + 1) + j;
            int64_t first;
            int n;
            if (P.one_part)
                n = 1;
            else
                row_ctas<LT>(P, r, first, n);
            const float2 *part = P.row_part + r * P.PM;
#pragma unroll 4
            for (int i = 0; i < n; ++i) {
                const float2 pr = __ldcg(&part[i]);
                merge_ms(M, S, pr.x, pr.y, c);
            }
            const float4 sd = __ldcg(&P.row_side[r]);
            x = __float_as_int(sd.x);
            const float zx = sd.y, qx = sd.z, u = sd.w;
            const bool row_ok = isfinite(M) && isfinite(S);
            if (!row_ok)
                rbad |= kBadRow;
            if (!(u >= 0.0f && u < 1.0f))
                rbad |= kBadU;
            if (j < K) {
                rej = true;
                if (x < 0 || x >= V) {
                    rbad |= kBadToken;
                } else if (DENSE && !(qx > 0.0f && isfinite(qx))) {
                    rbad |= kBadQ;
                } else if (row_ok) {
                    const float px = __fdiv_rn(term(zx, c, mc_of(M, c)), S);
                    a = fminf(1.0f, __fdiv_rn(px, qx));
                    rej = !(u < a);
                }
            }
        }
        bad |= static_cast<int32_t>(__reduce_or_sync(0xFFFFFFFFu, static_cast<unsigned>(rbad)));
        if (write && P.accept_prob && j < K)
            P.accept_prob[b * K + j] = a;
        if (!found) {
            const unsigned msk = __ballot_sync(0xFFFFFFFFu, j < K && rej);
            int32_t src = -1;
            if (msk) {
                src = __ffs(msk) - 1;
                jstar = j0 + src;
                found = true;
            } else if (K - j0 < 32) {
                src = K - j0; // every draft passed: the bonus row K
            }
            if (src >= 0) {
                m_sel = __shfl_sync(0xFFFFFFFFu, M, src);
                s_sel = __shfl_sync(0xFFFFFFFFu, S, src);
                xsel = __shfl_sync(0xFFFFFFFFu, x, src);
            }
        }
    }
    if (write) {
        int32_t *out = P.out_tokens + b * (K + 1);
        if (bad) {
            for (int32_t k = lane; k <= K; k += 32)
                out[k] = -1;
            for (int32_t k = lane; k < K; k += 32) {
                if (P.accept_flags) P.accept_flags[b * K + k] = -1;
                if (P.accept_prob) P.accept_prob[b * K + k] = 0.0f;
            }
        } else {
            for (int32_t k = lane; k <= K; k += 32)
                out[k] = k < jstar ? P.tokens[b * K + k] : -1;
            if (P.accept_flags)
                for (int32_t k = lane; k < K; k += 32)
                    P.accept_flags[b * K + k] = k < jstar ? 1 : (k == jstar ? 0 : -1);
        }
        if (lane == 0) {
            if (bad) {
                P.num_emitted[b] = 0;
                if (P.residual_mass) P.residual_mass[b] = 0.0f;
                if (P.status) atomicOr(P.status, bad);
            } else {
                P.num_emitted[b] = jstar + 1;
                if (P.stats) { // the call's acceptance statistics (sequences with bad data count in none)
                    unsigned long long *st = P.stats;
                    atomicAdd(&st[0], 1ull);
                    atomicAdd(&st[1], static_cast<unsigned long long>(K));
                    atomicAdd(&st[2], static_cast<unsigned long long>(jstar));
                    atomicAdd(&st[3], static_cast<unsigned long long>(jstar + 1));
                    atomicAdd(&st[4 + jstar], 1ull);
                }
            }
            P.seq_info[b] = make_int4(bad ? -1 : jstar, __float_as_int(m_sel), __float_as_int(s_sel),
                                      (!DENSE && !bad && jstar < K) ? xsel : -1);
        }
    }
    Verdict v;
    v.jstar = bad ? -1 : jstar;
    v.m = m_sel;
    v.s = s_sel;
    v.x = (!DENSE && !bad && jstar < K) ? xsel : -1;
    return v;
}

} // namespace sv
