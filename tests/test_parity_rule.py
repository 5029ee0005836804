"""The verification comparison rule itself (CPU).

Candidates are built from the oracle's own outputs: exact copies must pass,
planted mistakes must fail, and a decision flipped by an amount inside the
1e-5 window around its boundary must be counted as excused, not failed."""
import numpy as np
import pytest

from oracle import parity

B, K, V, T = 6, 3, 50, 1.0


def _inputs(seed=5):
    rng = np.random.default_rng(seed)
    z = (2.0 * rng.standard_normal((B, K + 1, V))).astype(np.float32)
    qz = z[:, :K] + rng.standard_normal((B, K, V)).astype(np.float32)
    q = np.exp(qz - qz.max(-1, keepdims=True))
    q = (q / q.sum(-1, keepdims=True)).astype(np.float32)
    def draw(row):
        pk = row.astype(np.float64)
        return rng.choice(V, p=pk / pk.sum())
    tok = np.array([[draw(q[b, k]) for k in range(K)] for b in range(B)], dtype=np.int32)
    u = rng.random((B, K + 1), dtype=np.float32)
    return z, q, tok, u


def _cand(res):
    return {"out_tokens": res.out_tokens.copy(), "num_emitted": res.num_emitted.copy(),
            "accept_flags": res.accept_flags.copy(), "accept_prob": res.accept_prob.astype(np.float32),
            "residual_mass": res.residual_mass.astype(np.float32)}


def test_exact_candidate_passes(orc):
    z, q, tok, u = _inputs()
    rep = parity.compare(orc, z, q, tok, u, T, _cand(orc.verify(z, q, tok, u, T)))
    assert rep.ok() and rep.excused == 0 and rep.sequences == B


@pytest.mark.parametrize("mistake", ["token", "count", "flag", "prob", "mass"])
def test_planted_mistakes_fail(orc, mistake):
    z, q, tok, u = _inputs()
    res = orc.verify(z, q, tok, u, T)
    c = _cand(res)
    b = 0
    n = int(c["num_emitted"][b])
    if mistake == "token":
        c["out_tokens"][b, n - 1] = (c["out_tokens"][b, n - 1] + 1) % V
    elif mistake == "count":
        c["num_emitted"][b] = n % (K + 1) + 1
    elif mistake == "flag":
        c["accept_flags"][b, 0] = 1 - c["accept_flags"][b, 0] if c["accept_flags"][b, 0] >= 0 else 1
    elif mistake == "prob":
        c["accept_prob"][b, 0] += 1e-4
    else:
        c["residual_mass"][b] += 1e-4
    rep = parity.compare(orc, z, q, tok, u, T, c)
    assert not rep.ok() and rep.failures and rep.failures[0][0] == b


def test_small_probability_error_passes(orc):
    z, q, tok, u = _inputs()
    c = _cand(orc.verify(z, q, tok, u, T))
    c["accept_prob"] += np.float32(2e-6)
    assert parity.compare(orc, z, q, tok, u, T, c).ok()


def _first_test(orc, z, q, tok, u):
    """(b, a) of a sequence whose first accept test has a threshold in
    (0.05, 0.95)."""
    res = orc.verify(z, q, tok, u, T)
    for b in range(B):
        a = float(res.accept_prob[b, 0])
        if 0.05 < a < 0.95:
            return b, a
    pytest.skip("no suitable threshold in this batch")


@pytest.mark.parametrize("rel,excused", [(3e-6, True), (3e-3, False)])
def test_accept_flip_near_threshold(orc, rel, excused):
    z, q, tok, u = _inputs()
    b, a = _first_test(orc, z, q, tok, u)
    u_ref = u.copy()
    u_ref[b, 0] = np.float32(a * (1 + rel))     # the oracle rejects the first draft
    u_cand = u.copy()
    u_cand[b, 0] = np.float32(a * (1 - rel))    # the candidate accepted it
    cand = _cand(orc.verify(z, q, tok, u_cand, T))
    rep = parity.compare(orc, z, q, tok, u_ref, T, cand)
    if excused:
        assert not rep.failures and rep.excused == 1, rep.summary()
    else:
        assert rep.failures, rep.summary()


@pytest.mark.parametrize("rel,excused", [(2e-6, True), (2e-3, False)])
def test_final_draw_across_a_boundary(orc, rel, excused):
    z, q, tok, u = _inputs()
    res = orc.verify(z, q, tok, u, T)
    b = 0
    n = int(res.num_emitted[b])
    j = n - 1
    _, w, cdf, Z = orc.row_dists(z, q, tok, T, b, j, j < K)
    # an interior boundary with mass on both sides
    i = int(np.argmax((w[:-1] > 1e-3) & (w[1:] > 1e-3)))
    c_i = cdf[i] / cdf[-1]                      # the boundary as a fraction of the total
    u_ref = u.copy()
    u_ref[b, K] = np.float32(c_i * (1 + rel))   # the oracle draws id i + 1
    u_cand = u.copy()
    u_cand[b, K] = np.float32(c_i * (1 - rel))  # the candidate drew id i
    ref = orc.verify(z, q, tok, u_ref, T)
    cand = _cand(orc.verify(z, q, tok, u_cand, T))
    assert cand["out_tokens"][b, j] != ref.out_tokens[b, j]
    rep = parity.compare(orc, z, q, tok, u_ref, T, cand)
    if excused:
        assert not rep.failures and rep.excused == 1, rep.summary()
    else:
        assert rep.failures, rep.summary()
