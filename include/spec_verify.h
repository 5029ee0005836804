/*
 * spec_verify.h -- C ABI of the GB300 speculative-sampling verification
 * library (libspecverify.so, sm_103a).
 *
 * The operation (one call verifies a whole batch of B sequences):
 *
 *   for every sequence b and target row j = 0..K:
 *       p_j = softmax(z_{b,j} / T)
 *     ("推测解码采样验证优化策略 —— 深度调研报告", part 1 section 4, verify():
 *      the softmax of target logits / temperature; "推测解码：草稿、验证与实际加速",
 *      section 接受与拒绝怎样保住分布: p already carries the temperature and q is
 *      passed exactly as the draft used it)
 *   row j verifies draft x_{j+1} (0-based: row k verifies draft k); row K only
 *   serves the extra token ("推测解码：草稿、验证与实际加速", section
 *   候选已知，验证才能并行, the equation listing p_1 .. p_4);
 *   drafts are tested left to right, draft k accepted iff
 *       u[b,k] < a_k,  a_k = min(1, p_k(x_k) / q_k(x_k))
 *     (same page, section 接受与拒绝怎样保住分布, equation for a(x));
 *   at the first rejection j*, one token is drawn from
 *       r = max(0, p_{j*} - q_{j*}) / sum(max(0, p_{j*} - q_{j*}))
 *     and later drafts are discarded; if all K drafts pass, one extra token is
 *     drawn from p_K (same page, equation for r(x); "投机采样", section
 *     机制：起草-验证-接受: each round emits n in [1, K+1] tokens);
 *   the draw uses the final uniform u[b,K]: the token is the smallest id i
 *     with u[b,K] * sum(w) < w_0 + ... + w_i ("推测解码：草稿、验证与实际加速",
 *     section 算完三个 token 的全部概率, the replay's sampler and final draw).
 *   A deterministic draft (n-gram, prompt lookup) is q = one-hot on x: pass
 *   draft_probs = NULL; then a_k = min(1, p_k(x_k)) and r is p without x.
 *   A target that samples with top-k / top-p runs its raw logits through
 *   sv_filter_logits first (same temperature); p is then the filtered,
 *   renormalised distribution.
 *
 * Entry points: spec_verify (the whole step), spec_verify_stats (plus
 * acceptance counters), sv_verify_rows / sv_sample_survivors (its two
 * stages), spec_verify_noalloc (no workspace argument), sv_filter_logits
 * (top-k / top-p), spec_verify_lm_head / sv_lm_head_logits (the target's LM
 * head on the tensor cores, fused with the row statistics), spec_verify_tree
 * (a candidate tree: several drafts per position), sv_workspace_bytes,
 * sv_lm_head_workspace_bytes, sv_tree_workspace_bytes, sv_kernel_launches,
 * sv_status_string.
 *
 * Conventions for every entry point below:
 *   - All tensor pointers are DEVICE pointers (inputs may also be mapped
 *     page-locked host memory, see spec_verify), row-major and contiguous,
 *     owned by the caller.  The library allocates nothing; its only state is
 *     per-device cached occupancy figures and, for spec_verify_noalloc, one
 *     static scratch array.  Calls on distinct workspaces are independent.
 *   - Calls are asynchronous on `stream` (a cudaStream_t; NULL = the legacy
 *     default stream).  A return of SV_OK means the work was enqueued.
 *   - Host-side checks run before anything is launched and return SV_EINVAL
 *     (null pointer, K < 0, B < 0, V < 1, temperature not finite or <= 0,
 *     misaligned pointer, workspace too small) or SV_EUNSUPPORTED (V above
 *     SV_MAX_V, or a batch too large for one launch).  B == 0 is a no-op.
 *     Launch failures return SV_ECUDA.  Nothing traps on the device.
 *   - Bad DATA is reported on the device: the sequence's outputs are set to
 *     "nothing emitted" (num_emitted 0, tokens and flags -1, probabilities 0)
 *     and SV_BAD_* bits are OR-ed into *status_dev (when not NULL).
 */
#ifndef SPEC_VERIFY_H
#define SPEC_VERIFY_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    SV_OK = 0,
    SV_EINVAL = 1,
    SV_ECUDA = 2,
    SV_EUNSUPPORTED = 3
} sv_status_t;

typedef enum { SV_BF16 = 0, SV_FP32 = 1 } sv_dtype_t;

/* Device status bits OR-ed into *status_dev. */
#define SV_BAD_U 1               /* a uniform outside [0, 1) or NaN          */
#define SV_BAD_TOKEN 2           /* a draft token outside [0, V)             */
#define SV_BAD_Q 4               /* q_k(x_k) <= 0 or not finite (dense q)    */
#define SV_BAD_ROW 8             /* a logit row with NaN / +inf / no finite  */
#define SV_DEGENERATE_RESIDUAL 16 /* residual mass 0 after a rejection: the  */
                                  /* token was drawn from p instead          */
#define SV_INTERNAL_TIMEOUT 32   /* a kernel's bounded wait ran out (the LM */
                                  /* head's pipeline); outputs undefined     */
#define SV_BAD_TREE 64           /* spec_verify_tree: parent[i] outside [0, i) */

/* Largest vocabulary supported. */
#define SV_MAX_V (1 << 21)
#define SV_MAX_TREE_NODES 256  /* nodes of one candidate tree (spec_verify_tree) */

/* Bytes of workspace spec_verify needs for (B, K, V).  The workspace must be
 * zero-filled before its first use.  A completed spec_verify (or the two
 * stages below, in order) returns every byte it used to zero, so the same
 * workspace can serve later calls of any shape that fits in it without being
 * cleared.  Two calls that may run at the same time need distinct
 * workspaces. */
size_t sv_workspace_bytes(int64_t B, int32_t K, int32_t V);

/* Verify a batch.
 *   target_logits  [B, K+1, V] bf16 or fp32 (logits_dtype); row j of sequence
 *                  b at offset (b*(K+1) + j) * V.  -inf entries are allowed
 *                  (masked tokens).  2-byte (bf16) / 4-byte (fp32) aligned.
 *   draft_probs    [B, K, V] fp32, the draft's processed distribution q, or
 *                  NULL for one-hot drafts.  4-byte aligned.
 *   draft_tokens   [B, K] int32 (may be NULL when K == 0).
 *   uniforms       [B, K+1] fp32 in [0, 1); u[b,k] tests draft k, u[b,K] is
 *                  the final draw used for the correction or extra token.
 *   temperature    T > 0, applied to the target logits only.
 * Input pointers may be device memory or page-locked host memory mapped into
 * the device's address space (cudaHostAlloc / cudaHostRegister); host inputs
 * are read in place by the kernels, so only the bytes the step touches cross
 * the host link: every logit once, the surviving rows' logits again, the
 * draft probabilities of the rejected rows and the drafted entries of q.
 * Outputs:
 *   out_tokens     [B, K+1] int32: accepted drafts, then the drawn token, then
 *                  -1 padding.
 *   num_emitted    [B] int32 in [1, K+1] (0 for a sequence with bad data).
 *   accept_flags   [B, K] int8: 1 accepted, 0 the first rejection, -1 not
 *                  reached.  May be NULL.
 *   accept_prob    [B, K] fp32: a_k for every draft (also those not reached).
 *                  May be NULL.
 *   residual_mass  [B] fp32: sum(max(0, p_{j*} - q_{j*})) at the rejection,
 *                  0 when the extra token was drawn.  May be NULL.
 *   status_dev     one device int32; SV_BAD_* bits are OR-ed in.  May be NULL.
 *   workspace      device scratch of at least sv_workspace_bytes(B, K, V)
 *                  bytes, 256-byte aligned (see sv_workspace_bytes).
 */
sv_status_t spec_verify(const void *target_logits, sv_dtype_t logits_dtype,
                        const float *draft_probs, const int32_t *draft_tokens,
                        const float *uniforms, float temperature, int64_t B,
                        int32_t K, int32_t V, int32_t *out_tokens,
                        int32_t *num_emitted, int8_t *accept_flags,
                        float *accept_prob, float *residual_mass,
                        int32_t *status_dev, void *workspace,
                        size_t workspace_bytes, void *stream);

/* spec_verify, plus the call's acceptance statistics, counted by the verdict
 * of every sequence (atomic adds into stats_dev; no extra launch).  What the
 * pages ask a deployment to record per round -- candidates, accepted
 * drafts, tokens committed ("推测解码：草稿、验证与实际加速", section
 * 在相同负载和质量下比较, the table of what to record) -- and what their
 * engine's acceptance-rate monitor feeds its adaptive draft length ("推测解码
 * 采样验证优化策略 —— 深度调研报告", part 1 §2, the engine's monitor step and
 * _adjust_K).  stats_dev: SV_STATS_WORDS(K) uint64 counters in device memory,
 * 8-byte aligned, added to (zero them to start a window):
 *   [0] sequences verified          [1] drafts proposed (K per sequence)
 *   [2] drafts accepted             [3] tokens emitted (accepted + 1)
 *   [4 + n] sequences that accepted exactly n drafts, n = 0..K
 * Sequences with bad data (num_emitted = 0) count in none of them.
 * Returns SV_EINVAL when stats_dev is NULL or misaligned. */
#define SV_STATS_WORDS(K) (4 + (K) + 1)
sv_status_t spec_verify_stats(const void *target_logits, sv_dtype_t logits_dtype,
                              const float *draft_probs, const int32_t *draft_tokens,
                              const float *uniforms, float temperature, int64_t B,
                              int32_t K, int32_t V, int32_t *out_tokens,
                              int32_t *num_emitted, int8_t *accept_flags,
                              float *accept_prob, float *residual_mass,
                              int32_t *status_dev, void *workspace,
                              size_t workspace_bytes, uint64_t *stats_dev,
                              void *stream);

/* The two stages of spec_verify, for callers that time or schedule them
 * separately.  Same arguments and meaning as spec_verify.
 *
 * sv_verify_rows: the row pass over all B*(K+1) rows: the max and softmax
 * normaliser of every row, in pieces, and the draft data of every row
 * (x, z(x), q(x), u), left in the workspace.  Writes no output.
 *
 * sv_sample_survivors: per sequence, the accept tests and the first
 * rejection (accept_flags, accept_prob, num_emitted, the accepted prefix of
 * out_tokens and its -1 padding, status bits), then the draw of the final
 * token from the residual (after a rejection) or from p_K (all accepted):
 * out_tokens[b, num_emitted-1] and residual_mass.  Must follow
 * sv_verify_rows on the same stream with the same workspace and inputs; it
 * returns the workspace to zero. */
sv_status_t sv_verify_rows(const void *target_logits, sv_dtype_t logits_dtype,
                           const float *draft_probs,
                           const int32_t *draft_tokens, const float *uniforms,
                           float temperature, int64_t B, int32_t K, int32_t V,
                           int32_t *out_tokens, int32_t *num_emitted,
                           int8_t *accept_flags, float *accept_prob,
                           float *residual_mass, int32_t *status_dev,
                           void *workspace, size_t workspace_bytes,
                           void *stream);

sv_status_t sv_sample_survivors(
    const void *target_logits, sv_dtype_t logits_dtype,
    const float *draft_probs, const int32_t *draft_tokens,
    const float *uniforms, float temperature, int64_t B, int32_t K, int32_t V,
    int32_t *out_tokens, int32_t *num_emitted, int8_t *accept_flags,
    float *accept_prob, float *residual_mass, int32_t *status_dev,
    void *workspace, size_t workspace_bytes, void *stream);

/* Allocation-free variant of spec_verify.  The pages have no counterpart:
 * this entry point exists for callers that cannot allocate device memory,
 * for example a server whose device memory is reserved up front by its own
 * pool and that forbids cudaMalloc on the request path, or a plugin interface
 * that hands a plugin its input and output buffers but no allocator.
 *
 * Same arguments and results as spec_verify, without the workspace: the
 * scratch is a fixed array of SV_NOALLOC_SCRATCH_BYTES in the library's
 * device image, present on every GPU that loads the library until the
 * process exits.  The caller still passes all inputs and outputs.
 *   - Returns SV_EUNSUPPORTED when sv_workspace_bytes(B, K, V) exceeds
 *     SV_NOALLOC_SCRATCH_BYTES (4 MiB holds, e.g., B = 256, K = 8 at V = 151936).
 *   - Calls no cudaMalloc / cudaFree and no allocating library routine.
 *   - Every call looks up the array's device address in the current
 *     context (cudaGetSymbolAddress, host-side and cheap), so the address
 *     stays right after a context is destroyed and made again.  The first
 *     call on a device may also load the library's device code into the
 *     context; make that first call before any stream capture.
 *   - Every call on a device shares the one array: each call clears the
 *     bytes it uses (an asynchronous memset on `stream`) and then launches.
 *     Calls whose work may overlap on the GPU (different streams or host
 *     threads without ordering between them) race on the array and give
 *     undefined results; order them on one stream. */
#define SV_NOALLOC_SCRATCH_BYTES (4u << 20)
sv_status_t spec_verify_noalloc(const void *target_logits,
                                sv_dtype_t logits_dtype,
                                const float *draft_probs,
                                const int32_t *draft_tokens,
                                const float *uniforms, float temperature,
                                int64_t B, int32_t K, int32_t V,
                                int32_t *out_tokens, int32_t *num_emitted,
                                int8_t *accept_flags, float *accept_prob,
                                float *residual_mass, int32_t *status_dev,
                                void *stream);

/* Top-k / top-p filtering of target logit rows, for targets that sample
 * with those filters: the accept test and the final draw must see the
 * target's processed distribution -- temperature, top-k, top-p -- and q must
 * be what the draft actually used ("推测解码：草稿、验证与实际加速", section
 * 接受与拒绝怎样保住分布).  The pages name the filters without defining them;
 * this library's reading: the ids of a row are ordered by
 * p = softmax(z / T) descending, equal p by ascending id; top-k keeps the
 * first min(top_k, #finite) ids (top_k <= 0: no top-k); top-p keeps the
 * shortest prefix of that set whose mass reaches top_p times the set's mass,
 * the crossing id included (top_p >= 1: no top-p).  Kept logits are copied
 * unchanged and every other entry becomes -inf, so passing out_logits to
 * spec_verify with the same temperature verifies against the filtered p.
 *   logits      [rows, V] bf16 or fp32 (logits_dtype), device.
 *   out_logits  [rows, V], same dtype; may be the same pointer as logits (in
 *               place); other overlaps are not allowed.
 *   kept        [rows] int32: ids kept per row (0 for a bad row).  May be NULL.
 *   status_dev  SV_BAD_ROW is OR-ed in for a row with NaN, +inf or no finite
 *               logit; such a row is copied unchanged.  May be NULL.
 * Masses are formed as the verification forms them (exp2 on the
 * special-function unit, summed exactly in fixed point), so a row whose
 * cumulative mass crosses top_p within ~1e-6 of an id's boundary may keep
 * one id more or less than an fp64 computation would.
 * Returns SV_EINVAL (NULL or misaligned pointer, rows < 0, V < 1, T not
 * finite or <= 0, top_p <= 0 or NaN, unknown dtype), SV_EUNSUPPORTED
 * (V > SV_MAX_V) or SV_ECUDA.  rows == 0 is a no-op.  One launch on
 * `stream`; allocates nothing. */
sv_status_t sv_filter_logits(const void *logits, sv_dtype_t logits_dtype,
                             int64_t rows, int32_t V, float temperature,
                             int32_t top_k, float top_p, void *out_logits,
                             int32_t *kept, int32_t *status_dev, void *stream);

/* The target's LM head fused with the verification ("推测解码采样验证优化策略 ——
 * 深度调研报告", part 1 section 6, 扩展性与安全性: operator fusion of the
 * verification into the target's last layer).
 *
 * sv_lm_head_logits: logits = hidden * lm_head^T on the tensor cores (fp32
 * accumulation, result rounded to bf16 round-to-nearest-even).
 *   hidden   [M, d] bf16, 16-byte aligned, row-major;
 *   lm_head  [V, d] bf16 (the output embedding), 16-byte aligned;
 *   logits   [M, V] bf16 out (2-byte aligned; 16-byte aligned with V % 8 == 0
 *            for the fast stores).
 *   status_dev: optional device int32; SV_INTERNAL_TIMEOUT is OR-ed into it
 *   if one of the kernel's bounded waits ran out (the logits are then
 *   incomplete); the caller zeroes it.
 *   d must be a multiple of 8 (the rows' 16-byte stride) and at least 8;
 *   M <= 2^30, V <= SV_MAX_V.  Returns SV_EINVAL / SV_EUNSUPPORTED on bad
 *   sizes or pointers, SV_ECUDA when a launch (or the tensor-map set-up)
 *   fails.  One launch on `stream`; allocates nothing.
 *
 * spec_verify_lm_head: spec_verify on logits the LM head computes in the same
 * step: hidden [B, K+1, d] bf16 (the target's last hidden states of the K+1
 * verified positions), lm_head [V, d] bf16; the logits are written to
 * logits_out [B, K+1, V] bf16 (the surviving rows are read again by the
 * draws) and each row's softmax statistics are formed by the GEMM's
 * epilogue from those bf16 values, so no separate pass over the logits is
 * made.  Every other argument as spec_verify; the workspace must hold
 * sv_lm_head_workspace_bytes(B, K, V) bytes, zero-filled before first use;
 * every completed call returns all of it to zero (the GEMM's per-tile
 * statistics included), so one workspace serves every entry point. */
size_t sv_lm_head_workspace_bytes(int64_t B, int32_t K, int32_t V);
sv_status_t sv_lm_head_logits(const void *hidden, const void *lm_head,
                              int64_t M, int32_t d, int32_t V, void *logits,
                              int32_t *status_dev, void *stream);
sv_status_t spec_verify_lm_head(const void *hidden, const void *lm_head,
                                int32_t d, const float *draft_probs,
                                const int32_t *draft_tokens,
                                const float *uniforms, float temperature,
                                int64_t B, int32_t K, int32_t V,
                                void *logits_out, int32_t *out_tokens,
                                int32_t *num_emitted, int8_t *accept_flags,
                                float *accept_prob, float *residual_mass,
                                int32_t *status_dev, void *workspace,
                                size_t workspace_bytes, void *stream);

/* Verification of a candidate tree: several drafts per position, one path
 * committed.  The pages require that a tree commits one contiguous path and
 * keeps the target distribution ("推测解码：草稿、验证与实际加速", section
 * 链、树与自推测) but give no rule; the rule implemented is multi-step
 * speculative sampling (SpecInfer, Miao et al., ASPLOS 2024).
 *
 * Per sequence, N nodes (1 <= N <= SV_MAX_TREE_NODES): node 0 is the
 * committed prefix; node i >= 1 holds draft token tokens[i] and has parent
 * parent[i] in [0, i).  The children of a node are its nodes in increasing
 * index order and must have been drafted i.i.d. (with replacement) from
 * that node's draft distribution.
 *   logits      [B, N, V] bf16 or fp32: row i is the target's next-token
 *               logits after node i's path (one tree-attention forward);
 *   draft_probs [B, N, V] fp32: row i is the draft distribution node i's
 *               children were drawn from (rows of leaves are not read);
 *   parent, tokens [B, N] int32 (entry 0 of each is not read);
 *   uniforms    [B, N] fp32 in [0, 1): uniforms[i] (i >= 1) is the
 *               acceptance test of node i, uniforms[0] the final draw.
 * From node 0: the children of the current node v are tested in order
 * against a running target r (first r = p_v = softmax(z_v / T)); child c
 * with token x is accepted iff u[c] < min(1, r(x) / q_v(x)), and then the
 * walk continues at c; after a rejection r = max(0, r - q_v) normalised.
 * When every child of v is rejected the final token is drawn from r, and
 * at a leaf from p_v, by inverse CDF with u[0].
 * Outputs: out_tokens [B, N] (the accepted path's tokens, then the final
 * token, then -1), out_nodes [B, N] (optional: the accepted path's node
 * ids, then -1), num_emitted [B] (path length + 1), accept_prob [B, N]
 * (optional: min(1, r(x)/q(x)) of every tested node, -1 for the others).
 * A sequence with an invalid input emits nothing (num_emitted 0, -1 tokens)
 * and SV_BAD_U / SV_BAD_TREE / SV_BAD_TOKEN / SV_BAD_Q / SV_BAD_ROW is OR-ed
 * into *status_dev (optional); SV_DEGENERATE_RESIDUAL as for spec_verify.
 * The workspace (sv_tree_workspace_bytes(B, N, V) bytes, 256-byte aligned)
 * follows spec_verify's rule: zero-filled before its first use, returned to
 * zero by every completed call, so one workspace serves both.  Two launches
 * on `stream` (the row pass over all B*N rows, then a cluster of two CTAs per
 * sequence for the walk); allocates nothing.  B <= 2^30.
 * Returns SV_EINVAL / SV_EUNSUPPORTED on bad arguments (nothing launched)
 * and SV_ECUDA when a launch fails. */
size_t sv_tree_workspace_bytes(int64_t B, int32_t N, int32_t V);
sv_status_t spec_verify_tree(const void *logits, sv_dtype_t dtype,
                             const float *draft_probs, const int32_t *parent,
                             const int32_t *tokens, const float *uniforms,
                             float temperature, int64_t B, int32_t N, int32_t V,
                             int32_t *out_tokens, int32_t *out_nodes,
                             int32_t *num_emitted, float *accept_prob,
                             int32_t *status_dev, void *workspace,
                             size_t workspace_bytes, void *stream);

/* Number of kernels one spec_verify (or spec_verify_stats) call with these
 * arguments launches on the CURRENT device: 2 (the row pass and the draw
 * stream, which then also makes the final draws) or 3 (plus the final
 * kernel).  The choice depends on B, K, V, the logits dtype, whether draft
 * probabilities are passed (dense != 0; ignored when K == 0) and how many
 * CTAs of each kernel the device holds at once.  *launches is 0 for B == 0.
 * Returns SV_EINVAL (NULL launches, B < 0, K < 0, V < 1, unknown dtype),
 * SV_EUNSUPPORTED (sizes spec_verify would reject as unsupported) or
 * SV_ECUDA (the device could not be queried).  Launches nothing.  The pages
 * have no counterpart: it serves callers that account for launches. */
sv_status_t sv_kernel_launches(sv_dtype_t logits_dtype, int32_t dense,
                               int64_t B, int32_t K, int32_t V,
                               int32_t *launches);

/* Static, NUL-terminated description of a status code. */
const char *sv_status_string(sv_status_t status);

#ifdef __cplusplus
}
#endif

#endif /* SPEC_VERIFY_H */
