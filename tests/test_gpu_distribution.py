"""Statistical checks of the GPU path itself (10^6 sequences in one call).

Unbiasedness ("投机采样", section 深入推导; "推测解码：草稿、验证与实际加速", section
接受与拒绝怎样保住分布): the token emitted at position j, among the sequences
that reach j, is distributed as p_j = softmax(z_j).  Chi-square at
alpha = 0.001 per position, dense and one-hot drafts.

Expected length ("推测解码：草稿、验证与实际加速", section 好草稿也要算得便宜;
"投机采样", section 参考答案): with i.i.d. acceptance rate alpha the mean
number of tokens per sequence is (1 - alpha^(gamma+1)) / (1 - alpha)
(3.3616 and 4.0951 for gamma = 4, alpha = .8 / .9; 2.95 for gamma = 3,
alpha = .8), within 5 standard errors."""
import numpy as np
import pytest
import torch

import speculative_decoding_sampling_gb300 as sv

pytestmark = pytest.mark.gpu

N = 1_000_000


def _draws(rng, dist, n):
    """n ids from each row of `dist` (test-local inverse-CDF sampler), [n, rows]."""
    c = np.cumsum(dist, axis=-1)
    c[..., -1] = 1.0
    return np.stack([np.searchsorted(c[j], rng.random(n), side="right")
                     for j in range(dist.shape[0])], axis=1).astype(np.int32)


def _run(p, q, rng):
    """N sequences: target logits ln p (T = 1), drafts ~ q (or uniform ids for
    one-hot drafts), seeded uniforms.  Returns (out_tokens, num_emitted)."""
    K1, V = p.shape
    K = K1 - 1
    with np.errstate(divide="ignore"):
        z = np.log(p).astype(np.float32)                       # p = 0 -> -inf
    logits = torch.from_numpy(np.ascontiguousarray(np.broadcast_to(z, (N, K1, V)))).cuda()
    if q is None:
        tok = rng.integers(0, V, size=(N, K), dtype=np.int32)
        dq = None
    else:
        tok = _draws(rng, q, N)
        dq = torch.from_numpy(np.ascontiguousarray(np.broadcast_to(q.astype(np.float32), (N, K, V)))).cuda()
    u = rng.random((N, K1), dtype=np.float32)
    status = torch.zeros(1, dtype=torch.int32, device="cuda:0")
    res = sv.spec_verify(logits, dq, torch.from_numpy(tok).cuda(), torch.from_numpy(u).cuda(), 1.0,
                         status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    return res.out_tokens.cpu().numpy(), res.num_emitted.cpu().numpy()


def _softmax64(z32):
    z = z32.astype(np.float64)
    e = np.exp(z - z.max(axis=-1, keepdims=True))
    return e / e.sum(axis=-1, keepdims=True)


@pytest.mark.parametrize("V,K,onehot", [(3, 3, False), (8, 4, False), (8, 3, True)],
                         ids=["V3_K3_dense", "V8_K4_dense", "V8_K3_onehot"])
def test_emitted_token_distribution(V, K, onehot):
    from scipy.stats import chisquare
    rng = np.random.default_rng(1000 * V + K)
    p = rng.dirichlet(np.ones(V) * 0.8, size=K + 1)
    q = None if onehot else rng.dirichlet(np.ones(V) * 0.8, size=K)
    out, n = _run(p, q, rng)
    assert (n >= 1).all() and (n <= K + 1).all()
    with np.errstate(divide="ignore"):
        target = _softmax64(np.log(p).astype(np.float32))     # what the logits define
    for j in range(K + 1):
        reached = n > j
        counts = np.bincount(out[reached, j], minlength=V)
        exp = target[j] * reached.sum()
        stat, pval = chisquare(counts, exp)
        assert pval > 1e-3, (V, K, onehot, j, pval)


@pytest.mark.parametrize("alpha,gamma", [(0.8, 4), (0.9, 4), (0.8, 3)])
def test_mean_tokens_per_sequence(alpha, gamma):
    rng = np.random.default_rng(int(alpha * 100) + gamma)
    V = 8
    base = rng.dirichlet(np.ones(V - 1))
    p1 = np.append(base, 0.0)                 # p = 0 on the last id
    q1 = alpha * p1
    q1[-1] = 1 - alpha                         # sum_x min(p, q) = alpha
    p = np.tile(p1, (gamma + 1, 1))
    q = np.tile(q1, (gamma, 1))
    _, n = _run(p, q, rng)
    mean = n.mean()
    se = n.std() / np.sqrt(N)
    want = (1 - alpha ** (gamma + 1)) / (1 - alpha)
    assert abs(mean - want) < 5 * se, (alpha, gamma, mean, want, se)
