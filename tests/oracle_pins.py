"""Pins that tie the fp64 oracle to what the pages and the mathematics fix.

Each ``pin_*`` takes an oracle handle and raises AssertionError when the
oracle disagrees with a value printed on the pages, a closed form, an
invariant, a textbook special case, or exact brute force.  The same pins run
against the real oracle (tests/test_oracle_pins.py) and against deliberately
broken copies of it (tests/test_oracle_mutants.py), which must each fail at
least one pin.

Sources:
  [NOTE]  "推测解码：草稿、验证与实际加速" -- sections 候选已知，验证才能并行,
          接受与拒绝怎样保住分布, 算完三个 token 的全部概率 (worked example),
          好草稿也要算得便宜 (E[N] and its printed values).
  [KB]    "投机采样" -- sections 机制：起草-验证-接受, 收益账,
          深入推导 (pointwise identity), 参考答案 (E[n] for alpha=0.8, gamma=3).
  [SURVEY-REPORT] "推测解码采样验证优化策略 —— 深度调研报告", part 1 section 4
          (softmax of logits / temperature before verification); part 1
          section 6 (fusing the verification into the target's last layer:
          the LM head's logits = h W^T).
"""
from __future__ import annotations

import os
from fractions import Fraction as F

import numpy as np

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


# ----------------------------------------------------------------- helpers

def read_golden(name: str) -> dict[str, list[str]]:
    out = {}
    with open(os.path.join(GOLDEN, name), encoding="utf-8") as fh:
        for line in fh:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, val = line.split("=", 1)
            out[key.strip()] = val.split()
    return out


def probs_call(orc, p_rows, q_rows, tokens, u, B=1):
    """Single-sequence call of the probabilities entry (p rows K+1, q rows K)."""
    p = np.asarray(p_rows, np.float64)[None].repeat(B, 0)
    q = None if q_rows is None else np.asarray(q_rows, np.float64)[None].repeat(B, 0)
    t = np.asarray(tokens, np.int32)[None].repeat(B, 0)
    uu = np.asarray(u, np.float64)[None].repeat(B, 0)
    return orc.verify_probs(p, q, t, uu)


def _softmax64(z):
    z = np.asarray(z, np.float64)
    m = z[np.isfinite(z)].max()
    e = np.exp(z - m)
    return e / e.sum()


def _categorical_by_library(w, u):
    """Textbook inverse-CDF draw: smallest i with u*sum(w) < cumsum(w)[i]."""
    c = np.cumsum(np.asarray(w, np.float64))
    return int(np.searchsorted(c, u * c[-1], side="right"))


# -------------------------------------------------- the pages' worked example

def pin_worked_example(orc):
    """[NOTE] 算完三个 token 的全部概率: p=(.5,.3,.2), q=(.6,.1,.3), drafts A,C,B,
    draws .7,.9,.2 and final draw .2 emit [A, B]; A passes at 0.833, C fails
    at 0.667, the rest is discarded."""
    g = read_golden("worked_example.txt")
    ids = {name: i for i, name in enumerate(g["tokens"])}
    p = [float(F(x)) for x in g["p"]]
    q = [float(F(x)) for x in g["q"]]
    draft = [ids[x] for x in g["draft"]]
    u = [float(F(x)) for x in g["draws"]] + [float(F(g["final_draw"][0]))]
    K = len(draft)
    r = probs_call(orc, [p] * (K + 1), [q] * K, draft, u)
    emit = [ids[x] for x in g["emit"]]
    assert r.status[0] == 0
    assert r.num_emitted[0] == len(emit), r.num_emitted
    assert list(r.out_tokens[0, :len(emit)]) == emit, r.out_tokens
    assert (r.out_tokens[0, len(emit):] == -1).all()
    # A accepted, C rejected, B never reached (discarded)
    assert list(r.accept_flags[0]) == [1, 0, -1], r.accept_flags
    assert abs(r.accept_prob[0, 0] - float(g["threshold_A"][0])) < 5e-4
    assert abs(r.accept_prob[0, 1] - float(g["threshold_C"][0])) < 5e-4
    # residual mass at the rejection = 1 - acceptance
    assert abs(r.residual_mass[0] - (1 - float(F(g["acceptance"][0])))) < 1e-12


def pin_worked_example_probabilities(orc):
    """[NOTE] 算完三个 token 的全部概率: per-token acceptance (5/6, 1, 2/3),
    accepted mass (.5,.1,.2), total acceptance .8."""
    g = read_golden("worked_example.txt")
    p = [float(F(x)) for x in g["p"]]
    q = [float(F(x)) for x in g["q"]]
    V = len(p)
    r = probs_call(orc, [p] * (V + 1), [q] * V, list(range(V)), [0.0] * (V + 1))
    want = [float(F(x)) for x in g["accept_prob_per_token"]]
    assert np.allclose(r.accept_prob[0], want, atol=1e-15, rtol=0), r.accept_prob
    mass = r.accept_prob[0] * np.asarray(q)
    assert np.allclose(mass, [float(F(x)) for x in g["accepted_mass_per_token"]],
                       atol=1e-15, rtol=0)
    assert abs(mass.sum() - float(F(g["acceptance"][0]))) < 1e-15


def pin_worked_example_residual(orc):
    """[NOTE] 算完三个 token 的全部概率: the residual is (0, 1, 0) and
    accepted mass + (1-acceptance)*residual rebuilds p.  Checked through the
    logits path: logits = ln p at T = 1."""
    g = read_golden("worked_example.txt")
    p = np.array([float(F(x)) for x in g["p"]])
    q = np.array([float(F(x)) for x in g["q"]], np.float32)
    V = 3
    logits = np.log(p).astype(np.float32)[None, None].repeat(V + 1, 1)
    qq = q[None, None].repeat(V, 1)
    tok = np.arange(V, dtype=np.int32)[None]
    pr, w, cdf, Z = orc.row_dists(logits, qq, tok, 1.0, 0, 0, True)
    assert np.allclose(w, [float(F(x)) for x in g["residual"]], atol=1e-6)
    assert abs(Z - (1 - float(F(g["acceptance"][0])))) < 1e-6
    res = orc.verify(logits, qq, tok, np.zeros((1, V + 1), np.float32), 1.0)
    rebuilt = res.accept_prob[0] * q + Z * w
    assert np.allclose(rebuilt, [float(F(x)) for x in g["reconstructed"]],
                       atol=1e-6)


# ------------------------------------------------------------- special cases

def pin_p_equals_q(orc):
    """[NOTE] 接受与拒绝怎样保住分布: if p = q every draft is accepted and the
    correction branch is never entered; the extra token comes from p_{K+1}."""
    rng = np.random.default_rng(11)
    V, K, B = 9, 5, 200
    p = rng.dirichlet(np.ones(V), size=(B, K + 1))
    q = p[:, :K].copy()
    tok = np.stack([[rng.choice(V, p=q[b, k]) for k in range(K)] for b in range(B)])
    u = rng.random((B, K + 1))
    r = orc.verify_probs(p, q, tok, u)
    assert (r.num_emitted == K + 1).all()
    assert (r.accept_flags == 1).all()
    assert (r.accept_prob == 1.0).all()
    assert (r.residual_mass == 0.0).all()
    assert (r.out_tokens[:, :K] == tok).all()
    for b in range(B):
        assert r.out_tokens[b, K] == _categorical_by_library(p[b, K], u[b, K])


def pin_k0_is_categorical(orc):
    """K = 0 leaves only the extra token: a textbook inverse-CDF draw from
    softmax(z / T) ([SURVEY-REPORT] part 1 section 4 for the softmax)."""
    rng = np.random.default_rng(12)
    from scipy.special import softmax
    for T in (0.5, 1.0, 1.7):
        z = rng.normal(0, 2, size=(300, 1, 37)).astype(np.float32)
        u = rng.random((300, 1)).astype(np.float32)
        r = orc.verify(z, None, np.zeros((300, 0), np.int32), u, T)
        assert (r.num_emitted == 1).all()
        for b in range(300):
            pb = softmax(z[b, 0].astype(np.float64) / T)
            assert r.out_tokens[b, 0] == _categorical_by_library(pb, float(u[b, 0]))


def pin_temperature_direction(orc):
    """softmax(z / T): z = (0, ln 3) at T = 1/2 gives p = (1/10, 9/10)."""
    z = np.array([[[0.0, np.log(3.0)], [0.0, np.log(3.0)]]], np.float32)
    tok = np.array([[1]], np.int32)
    r = orc.verify(z, None, tok, np.array([[0.0, 0.0]], np.float32), 0.5)
    # one-hot draft on token 1: acceptance probability is p(1)
    assert abs(r.accept_prob[0, 0] - 0.9) < 1e-6, r.accept_prob


def pin_bf16_decoding(orc):
    """bf16 bit patterns decode as the top half of an fp32: 0x3F80 = 1,
    0x0000 = 0, 0xFF80 = -inf, 0xC000 = -2."""
    bits = np.array([0x3F80, 0x0000, 0xFF80, 0xC000], np.uint16)
    logits = bits[None, None].repeat(2, 1)
    pr, w, cdf, Z = orc.row_dists(logits, None, np.array([[0]], np.int32), 1.0,
                                  0, 1, False)
    e = np.array([np.e, 1.0, 0.0, np.exp(-2.0)])
    assert np.allclose(pr, e / e.sum(), rtol=1e-14, atol=0)


def pin_onehot_draft(orc):
    """q = delta_x: a(x) = p(x); the residual is p with x removed and
    renormalised (deterministic drafts, [KB] 变体谱系 N-gram row)."""
    rng = np.random.default_rng(13)
    V, K = 11, 3
    z = rng.normal(0, 1.5, size=(1, K + 1, V)).astype(np.float32)
    tok = rng.integers(0, V, size=(1, K), dtype=np.int32)
    from scipy.special import softmax
    u = np.zeros((1, K + 1), np.float32)
    r = orc.verify(z, None, tok, u, 1.0)
    for k in range(K):
        pk = softmax(z[0, k].astype(np.float64))
        assert abs(r.accept_prob[0, k] - pk[tok[0, k]]) < 1e-14
        _, w, _, Z = orc.row_dists(z, None, tok, 1.0, 0, k, True)
        want = pk.copy()
        want[tok[0, k]] = 0.0
        assert abs(Z - (1 - pk[tok[0, k]])) < 1e-12
        assert np.allclose(w, want / want.sum(), rtol=1e-12, atol=1e-15)


def pin_vocab_of_one(orc):
    """V = 1: p = q = 1, every draft accepted, K+1 tokens, all id 0."""
    B, K = 5, 4
    z = np.zeros((B, K + 1, 1), np.float32)
    q = np.ones((B, K, 1), np.float32)
    u = np.random.default_rng(14).random((B, K + 1)).astype(np.float32)
    r = orc.verify(z, q, np.zeros((B, K), np.int32), u, 1.0)
    assert (r.num_emitted == K + 1).all() and (r.out_tokens == 0).all()


def pin_strict_accept(orc):
    """Reading of [NOTE] 算完三个 token 的全部概率 (the replay accepts iff the
    draw is strictly below the threshold): u = a rejects, u just below accepts."""
    p = [0.25, 0.75]
    q = [0.5, 0.5]
    r = probs_call(orc, [p, p], [q], [0], [0.5, 0.3])
    assert r.accept_flags[0, 0] == 0 and r.num_emitted[0] == 1
    r = probs_call(orc, [p, p], [q], [0], [np.nextafter(0.5, 0), 0.3])
    assert r.accept_flags[0, 0] == 1 and r.num_emitted[0] == 2


def pin_zero_mass_never_drawn(orc):
    """A token of zero mass is never drawn, even by u = 0 (strict t < C(i))."""
    p = [0.0, 0.0, 1.0, 0.0]
    r = probs_call(orc, [p], None, [], [0.0])
    assert r.out_tokens[0, 0] == 2
    # residual of zero mass on ids 0, 1: draw at u = 0 lands on id 2
    p = [0.3, 0.2, 0.5]
    q = [0.4, 0.5, 0.1]
    r = probs_call(orc, [p, p], [q], [1], [0.99, 0.0])
    assert r.accept_flags[0, 0] == 0 and r.out_tokens[0, 0] == 2


def pin_final_draw_for_correction(orc):
    """Reading of [NOTE] 算完三个 token 的全部概率: the correction is drawn with
    the final draw u[K], not with the draw that rejected."""
    p = [0.5, 0.5, 0.0]
    q = [0.0, 0.0, 1.0]
    # draft 2 has p = 0: rejected; residual = (0.5, 0.5, 0)
    r = probs_call(orc, [p, p, p], [q, q], [2, 2], [0.9, 0.9, 0.2])
    assert r.out_tokens[0, 0] == 0
    r = probs_call(orc, [p, p, p], [q, q], [2, 2], [0.2, 0.2, 0.9])
    assert r.out_tokens[0, 0] == 1


def pin_first_rejection_discards_rest(orc):
    """[NOTE] 候选已知，验证才能并行: after the first rejection the later drafts
    and their verdicts are void, even ones that would pass."""
    p = [0.1, 0.6, 0.3]
    q = [0.6, 0.1, 0.3]
    # draft 0 fails (a = 1/6 < .5), drafts 1 and 2 would pass (a = 1)
    r = probs_call(orc, [p] * 4, [q] * 3, [0, 1, 2], [0.5, 0.0, 0.0, 0.5])
    assert r.num_emitted[0] == 1
    assert list(r.accept_flags[0]) == [0, -1, -1]
    assert list(r.out_tokens[0, 1:]) == [-1, -1, -1]
    assert np.allclose(r.accept_prob[0], [1 / 6, 1, 1])


def pin_bonus_uses_last_row(orc):
    """[NOTE] 候选已知，验证才能并行: with every draft accepted the extra token
    comes from p_{K+1}, the row after the last draft."""
    K = 2
    rows = [[1 / 3, 1 / 3, 1 / 3]] * K + [[0.0, 0.0, 1.0]]
    r = probs_call(orc, rows, [[1 / 3] * 3] * K, [0, 1], [0.1, 0.1, 0.5])
    assert r.num_emitted[0] == K + 1 and r.out_tokens[0, K] == 2


def pin_batch_consistency(orc):
    """Sequences are independent: a batch gives what each sequence gives alone."""
    rng = np.random.default_rng(15)
    B, K, V = 7, 3, 13
    z = rng.normal(0, 2, size=(B, K + 1, V)).astype(np.float32)
    q = rng.dirichlet(np.ones(V), size=(B, K)).astype(np.float32)
    tok = rng.integers(0, V, size=(B, K), dtype=np.int32)
    u = rng.random((B, K + 1)).astype(np.float32)
    whole = orc.verify(z, q, tok, u, 0.9, nthreads=3)
    for b in range(B):
        one = orc.verify(z[b:b + 1], q[b:b + 1], tok[b:b + 1], u[b:b + 1], 0.9)
        assert (one.out_tokens[0] == whole.out_tokens[b]).all()
        assert one.num_emitted[0] == whole.num_emitted[b]
        assert (one.accept_prob[0] == whole.accept_prob[b]).all()


def pin_invalid_inputs(orc):
    """Preconditions of [NOTE] 算完三个 token 的全部概率 (q(x) > 0, 0 <= u < 1)
    and of a well-formed softmax row; a violating sequence emits nothing."""
    V, K = 4, 2
    z = np.zeros((1, K + 1, V), np.float32)
    q = np.full((1, K, V), 0.25, np.float32)
    tok = np.array([[1, 2]], np.int32)
    u = np.full((1, K + 1), 0.5, np.float32)
    import oracle as O

    def run(z=z, q=q, tok=tok, u=u):
        return orc.verify(z, q, tok, u, 1.0)

    cases = []
    u1 = u.copy(); u1[0, 2] = 1.0; cases.append((run(u=u1), O.ORC_BAD_U))
    u2 = u.copy(); u2[0, 0] = np.nan; cases.append((run(u=u2), O.ORC_BAD_U))
    t1 = tok.copy(); t1[0, 1] = V; cases.append((run(tok=t1), O.ORC_BAD_TOKEN))
    t2 = tok.copy(); t2[0, 0] = -1; cases.append((run(tok=t2), O.ORC_BAD_TOKEN))
    q1 = q.copy(); q1[0, 0, 1] = 0.0; cases.append((run(q=q1), O.ORC_BAD_Q))
    z1 = z.copy(); z1[0, 1, :] = -np.inf; cases.append((run(z=z1), O.ORC_BAD_ROW))
    z2 = z.copy(); z2[0, 2, 3] = np.nan; cases.append((run(z=z2), O.ORC_BAD_ROW))
    z3 = z.copy(); z3[0, 0, 0] = np.inf; cases.append((run(z=z3), O.ORC_BAD_ROW))
    for r, bit in cases:
        assert r.status[0] & bit, (r.status, bit)
        assert r.num_emitted[0] == 0
        assert (r.out_tokens == -1).all() and (r.accept_flags == -1).all()
    ok = run(u=np.full((1, K + 1), -0.0, np.float32))
    assert ok.status[0] == 0 and ok.num_emitted[0] >= 1


# ------------------------------------------------------------- invariants

def pin_pointwise_identity(orc):
    """[KB] 深入推导: q*min(1,p/q) + (1 - sum_y q(y)min(1,p(y)/q(y))) * r = p,
    pointwise, on the oracle's own fp64 vectors."""
    rng = np.random.default_rng(16)
    for V in (3, 8, 50):
        for trial in range(5):
            z = rng.normal(0, 2, size=V)
            zq = z + rng.normal(0, 1.0, size=V)
            q = np.exp(zq - zq.max())
            q = (q / q.sum()).astype(np.float32)
            q = np.maximum(q, np.float32(1e-30))
            logits = z.astype(np.float32)[None, None].repeat(V + 1, 1)
            qq = q[None, None].repeat(V, 1)
            tok = np.arange(V, dtype=np.int32)[None]
            res = orc.verify(logits, qq, tok, np.zeros((1, V + 1), np.float32), 1.0)
            a = res.accept_prob[0]
            p, r, _, Z = orc.row_dists(logits, qq, tok, 1.0, 0, 0, True)
            q64 = q.astype(np.float64)
            beta = float(np.sum(q64 * a))
            assert abs(Z - (1 - beta)) < 1e-12
            assert np.max(np.abs(q64 * a + (1 - beta) * r - p)) < 1e-12


def _sample_rows(rng, dist, n):
    """Draw n ids from each of the rows of `dist` (test-local sampler)."""
    c = np.cumsum(dist, axis=-1)
    c[..., -1] = 1.0
    return np.stack([np.searchsorted(c[j], rng.random(n), side="right")
                     for j in range(dist.shape[0])], axis=1).astype(np.int32)


def emitted_position_counts(orc, p, q, n_rounds, seed, chunk=200_000):
    """Run n_rounds i.i.d. rounds (drafts ~ q, or one-hot fixed drafts when q
    is None) and count, at every position j, the token emitted there among
    rounds that reach j."""
    rng = np.random.default_rng(seed)
    K1, V = p.shape
    K = K1 - 1
    counts = np.zeros((K1, V), np.int64)
    total_emitted = 0
    sq_emitted = 0
    done = 0
    while done < n_rounds:
        n = min(chunk, n_rounds - done)
        if q is None:
            tok = np.tile(rng.integers(0, V, size=K, dtype=np.int32), (n, 1))
        else:
            tok = _sample_rows(rng, q, n)
        u = rng.random((n, K1))
        r = orc.verify_probs(np.broadcast_to(p, (n, K1, V)),
                             None if q is None else np.broadcast_to(q, (n, K, V)),
                             tok, u)
        assert (r.status == 0).all()
        for j in range(K1):
            reached = r.num_emitted > j
            counts[j] += np.bincount(r.out_tokens[reached, j], minlength=V)
        total_emitted += int(r.num_emitted.sum())
        sq_emitted += int((r.num_emitted.astype(np.int64) ** 2).sum())
        done += n
    return counts, total_emitted, sq_emitted


def pin_output_distribution(orc):
    """[KB] 深入推导 / [NOTE] 接受与拒绝怎样保住分布: the token emitted at each
    position, given that the round reaches it, is distributed as p_j.
    10^6 seeded rounds, V = 3 and V = 8, chi-square at alpha = 0.001."""
    from scipy.stats import chisquare
    rng = np.random.default_rng(17)
    for V, K, onehot in ((3, 3, False), (8, 4, False), (8, 3, True)):
        p = rng.dirichlet(np.ones(V) * 0.8, size=K + 1)
        q = None if onehot else rng.dirichlet(np.ones(V) * 0.8, size=K)
        counts, _, _ = emitted_position_counts(orc, p, q, 1_000_000,
                                               seed=V * 100 + K)
        for j in range(K + 1):
            n = counts[j].sum()
            exp = p[j] * n
            keep = exp > 0
            assert counts[j][~keep].sum() == 0
            stat, pval = chisquare(counts[j][keep], exp[keep])
            assert pval > 1e-3, (V, K, onehot, j, pval)


def expected_tokens_closed_form(alpha: float, gamma: int) -> float:
    """E[N] = 1 + alpha + ... + alpha^gamma = (1 - alpha^(gamma+1)) / (1 - alpha)."""
    return (1 - alpha ** (gamma + 1)) / (1 - alpha)


def pin_expected_tokens(orc):
    """[NOTE] 好草稿也要算得便宜 prints 3.3616 (alpha .8) and 4.0951 (alpha .9)
    for gamma = 4; [KB] 参考答案 gives about 2.95 for alpha .8, gamma 3.
    The oracle's mean tokens per round over 10^6 rounds with i.i.d.
    acceptance alpha (sum_x min(p, q) = alpha at every position) must match
    within 5 standard errors."""
    assert round(expected_tokens_closed_form(0.8, 4), 4) == 3.3616
    assert round(expected_tokens_closed_form(0.9, 4), 4) == 4.0951
    assert round(expected_tokens_closed_form(0.8, 3), 2) == 2.95
    rng = np.random.default_rng(18)
    for alpha, gamma in ((0.8, 4), (0.9, 4), (0.8, 3)):
        V = 8
        base = rng.dirichlet(np.ones(V - 1))
        p1 = np.append(base, 0.0)                # p(y) = 0 on the last id
        q1 = alpha * p1
        q1[-1] = 1 - alpha                        # sum min(p, q) = alpha
        p = np.tile(p1, (gamma + 1, 1))
        q = np.tile(q1, (gamma, 1))
        n = 1_000_000
        _, tot, sq = emitted_position_counts(orc, p, q, n, seed=int(alpha * 10) + gamma)
        mean = tot / n
        var = sq / n - mean ** 2
        se = np.sqrt(var / n)
        want = expected_tokens_closed_form(alpha, gamma)
        assert abs(mean - want) < 5 * se, (alpha, gamma, mean, want, se)


# ----------------------------------------------------------- brute force

def _exact_round(p_rows, q_rows, draft, u):
    """The round's outcome in exact rational arithmetic, stepping through the
    rule of [NOTE] 接受与拒绝怎样保住分布 one draft at a time."""
    K = len(draft)
    out = []
    for k in range(K):
        x = draft[k]
        a = min(F(1), p_rows[k][x] / q_rows[k][x])
        if u[k] < a:
            out.append(x)
            continue
        w = [max(F(0), pi - qi) for pi, qi in zip(p_rows[k], q_rows[k])]
        break
    else:
        w = list(p_rows[K])
    t = u[K] * sum(w)
    acc = F(0)
    for i, wi in enumerate(w):
        acc += wi
        if t < acc:
            out.append(i)
            return out
    raise AssertionError("no token drawn")


def pin_bruteforce_tiny(orc):
    """V = 3, K <= 3, rational p and q: on a grid of draws (odd multiples of
    1/128, never equal to a threshold) the oracle's outcome equals the exact
    rational outcome at every grid point."""
    rng = np.random.default_rng(19)
    grid = [F(2 * i + 1, 128) for i in range(0, 64, 5)]
    for K in (0, 1, 2, 3):
        for trial in range(3):
            def rand_dist():
                c = rng.integers(1, 7, size=3)
                c[rng.integers(0, 3)] = 0 if rng.random() < 0.3 else c[0]
                c = [int(x) for x in c]
                if sum(c) == 0:
                    c = [1, 1, 1]
                return [F(x, sum(c)) for x in c]
            p_rows = [rand_dist() for _ in range(K + 1)]
            q_rows = []
            draft = []
            for _ in range(K):
                qd = rand_dist()
                q_rows.append(qd)
                draft.append(int(rng.choice([i for i in range(3) if qd[i] > 0])))
            pts = list(np.ndindex(*([len(grid)] * (K + 1))))
            if len(pts) > 3000:
                pts = [pts[i] for i in rng.choice(len(pts), 3000, replace=False)]
            us = [[grid[i] for i in pt] for pt in pts]
            n = len(us)
            P = np.array([[float(v) for v in row] for row in p_rows])
            Q = None if K == 0 else np.array([[float(v) for v in row] for row in q_rows])
            r = orc.verify_probs(np.broadcast_to(P, (n, K + 1, 3)),
                                 None if Q is None else np.broadcast_to(Q, (n, K, 3)),
                                 np.tile(np.array(draft, np.int32), (n, 1)).reshape(n, K),
                                 np.array([[float(x) for x in uu] for uu in us]))
            for b in range(n):
                want = _exact_round(p_rows, q_rows, draft, us[b])
                got = list(r.out_tokens[b, :r.num_emitted[b]])
                assert got == want, (K, p_rows, q_rows, draft, us[b], got, want)



# ------------------------------------------------ top-k / top-p filtering
# The target's p carries its own temperature, top-k and top-p ("推测解码：
# 草稿、验证与实际加速", section 接受与拒绝怎样保住分布); the pages do not define
# the two filters, so these pins fix the reading taken (ids ordered by p
# descending, ties by lower id; top-k keeps the first k; top-p keeps the
# shortest prefix of the top-k set reaching top_p of its mass).

def _filter_kept(orc, z, T=1.0, top_k=0, top_p=1.0):
    z = np.asarray(z, np.float32)[None, :]
    r = orc.filter_logits(z, T, top_k, top_p)
    kept = [int(i) for i in np.nonzero(np.isfinite(r.logits[0]))[0]]
    assert int(r.kept[0]) == len(kept) and int(r.status[0]) == 0
    # kept logits are copied bit for bit
    assert np.array_equal(r.logits[0][kept].view(np.uint32), z[0][kept].view(np.uint32))
    return kept


def pin_filter_closed_forms(orc):
    z = np.log([0.4, 0.3, 0.2, 0.1])
    assert _filter_kept(orc, z, top_p=0.35) == [0]
    assert _filter_kept(orc, z, top_p=0.5) == [0, 1]
    assert _filter_kept(orc, z, top_p=0.75) == [0, 1, 2]
    assert _filter_kept(orc, z, top_p=0.95) == [0, 1, 2, 3]
    assert _filter_kept(orc, z, top_k=2) == [0, 1]
    assert _filter_kept(orc, z, top_k=1) == [0]
    assert _filter_kept(orc, z, top_k=9) == [0, 1, 2, 3]
    # top-p measured against the top-k set's mass: 0.4 / 0.7 >= 0.5
    assert _filter_kept(orc, z, top_k=2, top_p=0.5) == [0]
    assert _filter_kept(orc, z, top_k=2, top_p=0.6) == [0, 1]
    # top-3 mass 0.9: 0.77 of it is 0.693, reached by 0.4 + 0.3
    assert _filter_kept(orc, z, top_k=3, top_p=0.77) == [0, 1]
    assert _filter_kept(orc, z, top_p=0.77) == [0, 1, 2]
    # order of the ids in the row does not matter
    assert _filter_kept(orc, z[::-1].copy(), top_p=0.5) == [2, 3]


def pin_filter_ties_by_id(orc):
    z = [1.0, 2.0, 2.0, 0.0, 2.0]
    assert _filter_kept(orc, z, top_k=1) == [1]
    assert _filter_kept(orc, z, top_k=2) == [1, 2]
    assert _filter_kept(orc, z, top_k=3) == [1, 2, 4]
    assert _filter_kept(orc, z, top_p=1e-9) == [1]
    # equal logits have exact unit masses: 0.5 of four is reached exactly by
    # the second id, which is kept (reaching the mass is enough)
    assert _filter_kept(orc, [0.0, 0.0, 0.0, 0.0], top_p=0.5) == [0, 1]
    assert _filter_kept(orc, [0.0, 0.0, 0.0, 0.0], top_p=0.75) == [0, 1, 2]


def pin_filter_temperature(orc):
    z = np.log([0.6, 0.4])
    # T = 1: p = (0.6, 0.4)
    assert _filter_kept(orc, z, T=1.0, top_p=0.55) == [0]
    assert _filter_kept(orc, z, T=1.0, top_p=0.8) == [0, 1]
    # T = 4: p0 = 0.6^(1/4) / (0.6^(1/4) + 0.4^(1/4)) = 0.5253
    assert _filter_kept(orc, z, T=4.0, top_p=0.55) == [0, 1]
    assert _filter_kept(orc, z, T=4.0, top_p=0.52) == [0]
    # T = 1/4: p0 = 0.6^4 / (0.6^4 + 0.4^4) = 0.8351
    assert _filter_kept(orc, z, T=0.25, top_p=0.8) == [0]


def pin_filter_masked_and_bad_rows(orc):
    ninf = -np.inf
    # -inf ids have p = 0: never kept, not counted
    assert _filter_kept(orc, [ninf, 1.0, ninf, 0.5], top_k=3) == [1, 3]
    assert _filter_kept(orc, [ninf, 1.0, ninf, 0.5], top_p=0.999999) == [1, 3]
    bad = np.array([[0.0, np.nan, 1.0], [0.0, np.inf, 1.0], [ninf, ninf, ninf], [0.0, 1.0, 2.0]],
                   np.float32)
    r = orc.filter_logits(bad, 1.0, 1, 0.5)
    assert list(r.status) == [8, 8, 8, 0] and list(r.kept) == [0, 0, 0, 1]
    assert np.array_equal(r.logits[:3].view(np.uint32), bad[:3].view(np.uint32))
    # bf16 rows: the masked ids become the bf16 -inf pattern
    zb = np.array([[0x3F80, 0x4000, 0xBF80]], np.uint16)   # 1.0, 2.0, -1.0
    rb = orc.filter_logits(zb, 1.0, 1, 1.0)
    assert list(rb.logits[0]) == [0xFF80, 0x4000, 0xFF80] and int(rb.kept[0]) == 1


def _bruteforce_kept(z, T, top_k, top_p):
    """The smallest order-closed set of finite ids (no id outside it ranks
    before an id inside it) within the top-k set whose mass reaches top_p
    of the top-k set's, by enumerating all subsets."""
    V = len(z)
    fin = [i for i in range(V) if np.isfinite(z[i])]
    m = max(z[i] / T for i in fin)
    e = {i: float(np.exp(z[i] / T - m)) for i in fin}

    def before(j, i):   # j ranks before i
        return z[j] > z[i] or (z[j] == z[i] and j < i)

    closed = []
    for mask in range(1, 1 << V):
        S = [i for i in range(V) if mask >> i & 1]
        if any(not np.isfinite(z[i]) for i in S):
            continue
        if all(j in S for i in S for j in fin if before(j, i)):
            closed.append(S)
    nk = len(fin) if top_k < 1 else min(top_k, len(fin))
    topk = [S for S in closed if len(S) == nk][0]
    if top_p >= 1.0:
        return sorted(topk), False
    tau = top_p * sum(e[i] for i in topk)
    ok = [S for S in closed if len(S) <= nk and sum(e[i] for i in S) >= tau]
    best = min(ok, key=len)
    near = any(abs(sum(e[i] for i in S) - tau) < 1e-12 for S in closed)
    return sorted(best), near


def pin_filter_bruteforce_tiny(orc):
    rng = np.random.default_rng(7)
    checked = 0
    for trial in range(60):
        V = int(rng.integers(1, 7))
        z = rng.choice([-2.0, -1.0, -0.5, 0.0, 0.5, 1.0, 2.0, -np.inf], size=V).astype(np.float32)
        if not np.isfinite(z).any():
            z[0] = 0.0
        for top_k in (0, 1, 2, 3, 6):
            for top_p in (0.3, 0.5, 0.8, 0.95, 1.0):
                for T in (0.5, 1.0, 2.0):
                    want, near = _bruteforce_kept(z.astype(np.float64), T, top_k, top_p)
                    if near:
                        continue
                    assert _filter_kept(orc, z, T=T, top_k=top_k, top_p=top_p) == want, \
                        (z, top_k, top_p, T)
                    checked += 1
    assert checked > 2000


def pin_filter_topk_matches_library_sort(orc):
    """Top-k on rows of 5000 ids with many ties (values on a coarse grid):
    the kept ids are the first k of numpy's stable sort by value descending
    (equal values keep ascending id order)."""
    rng = np.random.default_rng(23)
    z = (np.round(rng.standard_normal((6, 5000)) * 4.0) / 2.0).astype(np.float32)
    z[2, rng.random(5000) < 0.4] = -np.inf
    for k in (1, 7, 100, 2999):
        r = orc.filter_logits(z, 0.9, k, 1.0)
        for row in range(z.shape[0]):
            order = np.argsort(-z[row].astype(np.float64), kind="stable")
            finite = order[np.isfinite(z[row][order])]
            want = np.sort(finite[:k])
            got = np.nonzero(np.isfinite(r.logits[row]))[0]
            assert np.array_equal(got, want), (k, row)


def pin_filter_matches_generator_nucleus(orc):
    """The input generator marks the top-p nucleus of the 64-sequence workload
    with its own sort (synth.c); the oracle's filter must mask the same ids."""
    import synth
    w = synth.WORKLOADS["b64_k5_v128256_bf16_topp"].with_(B=2, V=6000)
    masked = synth.generate(w).logits
    raw = synth.generate(w.with_(top_p=0.0)).logits
    kept = masked != 0xFF80
    assert np.array_equal(masked[kept], raw[kept])
    r = orc.filter_logits(raw, w.T, 0, w.top_p)
    assert np.array_equal(r.logits, masked)
    assert (r.status == 0).all() and int(r.kept.min()) >= 1


# ------------------------------------------- the LM head (logits = h W^T)

def _bf16_bits(x):
    """fp32 values that are bf16 numbers -> their bf16 bit patterns."""
    u = np.ascontiguousarray(x, np.float32).view(np.uint32)
    assert not (u & 0xFFFF).any()
    return (u >> 16).astype(np.uint16)


def _rand_bf16(rng, shape):
    """Random bf16 bit patterns (the top halves of N(0, 1) fp32 draws)."""
    return (rng.standard_normal(shape).astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)


def _bf16_value(bits):
    return (np.asarray(bits, np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def pin_bf16_round_textbook(orc):
    """Round to nearest, ties to the even significand, 8 significant bits:
    1 + 2^-8 is halfway between 1 and 1 + 2^-7 and goes to 1 (even); 1 + 3 2^-8
    is halfway between 1 + 2^-7 and 1 + 2^-6 and goes to 1 + 2^-6; anything
    above a halfway point goes up; pi -> 3.140625; -2.5 and 0 are exact."""
    x = np.array([1.0, 1 + 2.0**-8, 1 + 3 * 2.0**-8, 1 + 2.0**-8 + 2.0**-20, -2.5, 0.0, np.pi,
                  -(1 + 2.0**-8), 255.5, 2.0**-100 * 1.00390625], np.float64)
    want = [0x3F80, 0x3F80, 0x3F82, 0x3F81, 0xC020, 0x0000, 0x4049, 0xBF80, 0x4380, 0x0D80]
    got = orc.bf16_round(x)
    assert [int(v) for v in got] == want, [hex(v) for v in got]


def pin_bf16_round_matches_bit_rounding(orc):
    """On fp32 inputs the fp64 rounding equals the integer form of
    round-to-nearest-even on the fp32 bit pattern (add 0x7FFF plus the kept
    low bit, drop 16 bits) -- a different algorithm for the same function."""
    rng = np.random.default_rng(7)
    x32 = (rng.standard_normal(4096) * np.exp2(rng.integers(-30, 30, 4096))).astype(np.float32)
    x32[:64] = (np.float32(1) + np.arange(64, dtype=np.float32) * np.float32(2.0**-9))  # halfway cases
    u = x32.view(np.uint32)
    want = ((u + 0x7FFF + ((u >> 16) & 1)) >> 16).astype(np.uint16)
    got = orc.bf16_round(x32.astype(np.float64))
    assert np.array_equal(got, want)


def pin_lm_head_identity_and_permutation(orc):
    """W = a permutation matrix (V = d): logits[:, v] = h[:, pi(v)] exactly;
    W = I: logits = h.  A transposed or shifted operand index breaks both."""
    rng = np.random.default_rng(11)
    M, d = 5, 24
    h = _rand_bf16(rng, (M, d))
    for perm in (np.arange(d), rng.permutation(d)):
        W = np.zeros((d, d), np.float32)
        W[np.arange(d), perm] = 1.0
        out = orc.lm_head(h, _bf16_bits(W))
        assert np.array_equal(out, _bf16_value(h)[:, perm])


def pin_lm_head_rectangular_closed_forms(orc):
    """V != d: W row v = c_v e_{k(v)} gives logits[:, v] = c_v h[:, k(v)];
    h = all ones gives logits = the row sums of W (exact here: every entry
    is a small dyadic number)."""
    rng = np.random.default_rng(12)
    M, d, V = 3, 16, 40
    k = rng.integers(0, d, V)
    cv = rng.choice([-2.0, -0.5, 0.25, 1.0, 3.0], V)
    W = np.zeros((V, d), np.float32)
    W[np.arange(V), k] = cv
    h = _bf16_bits(rng.choice([-1.5, 0.5, 2.0, 0.0], (M, d)).astype(np.float32))
    out = orc.lm_head(h, _bf16_bits(W))
    assert np.array_equal(out, _bf16_value(h)[:, k] * cv[None, :])
    W2 = _bf16_bits(rng.choice([-0.75, 0.0, 0.125, 1.0], (V, d)).astype(np.float32))
    ones = _bf16_bits(np.ones((M, d), np.float32))
    out2 = orc.lm_head(ones, W2)
    assert np.array_equal(out2, np.repeat(_bf16_value(W2).sum(1)[None], M, 0))


def pin_lm_head_matches_library_matmul(orc):
    """Random bf16 operands: the fp64 dot products equal numpy's fp64 matmul
    of the decoded values up to fp64 summation order, and single entries
    equal the full product's."""
    rng = np.random.default_rng(13)
    M, d, V = 7, 40, 33
    h = _rand_bf16(rng, (M, d))
    W = _rand_bf16(rng, (V, d))
    want = _bf16_value(h) @ _bf16_value(W).T
    out = orc.lm_head(h, W)
    assert np.allclose(out, want, rtol=1e-13, atol=1e-13)
    rows, cols = np.array([0, 6, 3]), np.array([32, 0, 17])
    assert np.array_equal(orc.lm_head_entries(h, W, rows, cols), out[rows, cols])


# ------------------------------------------------ tree (multi-candidate)
# The rule: SpecInfer's multi-step speculative sampling (Miao et al., ASPLOS
# 2024) -- the pages require that a tree commits one path and keeps the
# target distribution ("推测解码：草稿、验证与实际加速", section 链、树与自推测)
# but give no rule of their own.

def _tree_probs(orc, p_rows, q_rows, parent, tokens, u):
    return orc.tree_verify_probs(np.asarray(p_rows, np.float64)[None], np.asarray(q_rows, np.float64)[None],
                                 np.asarray(parent, np.int32)[None], np.asarray(tokens, np.int32)[None],
                                 np.asarray(u, np.float64)[None])


def pin_tree_hand_example(orc):
    """Three siblings at the root, worked by hand: p = (.5, .3, .2),
    q = (.2, .2, .6), children C, C, B.  C: a = .2/.6 = 1/3; after its
    rejection r = (.3, .1, 0)/.4 = (3/4, 1/4, 0); the second C: a = 0 (and
    u = 0 still rejects: the test is strict); then r = (.55, .05, 0)/.6 =
    (11/12, 1/12, 0); B: a = (1/12)/.2 = 5/12; if B is rejected too,
    r = (11/12 - .2, 0, 0) -> the final token is A whatever u[0]."""
    P = [[.5, .3, .2], [1, 0, 0], [1, 0, 0], [0, 0, 1]]
    Q = [[.2, .2, .6], [1 / 3] * 3, [1 / 3] * 3, [1 / 3] * 3]
    par, tok = [-1, 0, 0, 0], [0, 2, 2, 1]
    r = _tree_probs(orc, P, Q, par, tok, [0.99, 0.5, 0.0, 0.5])   # all three rejected
    assert np.allclose(r.accept_prob[0, 1:], [1 / 3, 0, 5 / 12], rtol=1e-14, atol=1e-15), r.accept_prob
    assert r.num_emitted[0] == 1 and r.out_tokens[0, 0] == 0 and r.status[0] == 0
    r = _tree_probs(orc, P, Q, par, tok, [0.5, 0.5, 0.0, 0.4])    # B accepted (0.4 < 5/12): leaf, bonus from its row
    assert list(r.out_nodes[0, :1]) == [3] and list(r.out_tokens[0, :2]) == [1, 2] and r.num_emitted[0] == 2
    r = _tree_probs(orc, P, Q, par, tok, [0.5, 0.3, 0.0, 0.4])    # the first C accepted (0.3 < 1/3)
    assert list(r.out_tokens[0, :2]) == [2, 0] and r.out_nodes[0, 0] == 1
    assert r.accept_prob[0, 2] == -1 and r.accept_prob[0, 3] == -1  # never tested
    # the pages' worked distributions: after A is rejected the residual is
    # (0, 1, 0), so a second child C is rejected and B is drawn
    r = _tree_probs(orc, [[.5, .3, .2], [1, 0, 0], [1, 0, 0]], [[.6, .1, .3], [1 / 3] * 3, [1 / 3] * 3],
                    [-1, 0, 0], [0, 0, 2], [0.2, 0.9, 0.5])
    assert r.out_tokens[0, 0] == 1 and r.num_emitted[0] == 1
    assert np.allclose(r.accept_prob[0, 1:], [5 / 6, 0], rtol=1e-14)


def pin_tree_chain_reduces_to_chain(orc):
    """A tree that is a chain (parent[i] = i - 1) is verified exactly as the
    chain rule verifies it: same tokens, counts and acceptance probabilities
    (tree u[i] = chain u[i-1], tree u[0] = chain u[K])."""
    rng = np.random.default_rng(21)
    B, K, V = 400, 5, 7
    p = rng.dirichlet(np.ones(V) * 0.7, (B, K + 1))
    q = rng.dirichlet(np.ones(V) * 0.7, (B, K))
    tok = np.array([[rng.choice(V, p=q[b, k]) for k in range(K)] for b in range(B)], np.int32)
    u = rng.random((B, K + 1))
    chain = orc.verify_probs(p, q, tok, u)
    qt = np.concatenate([q, np.full((B, 1, V), 1.0 / V)], 1)
    par = np.tile(np.arange(-1, K, dtype=np.int32), (B, 1))
    tt = np.concatenate([np.zeros((B, 1), np.int32), tok], 1)
    ut = np.concatenate([u[:, K:], u[:, :K]], 1)
    tr = orc.tree_verify_probs(p, qt, par, tt, ut)
    assert np.array_equal(tr.num_emitted, chain.num_emitted)
    assert np.array_equal(tr.out_tokens, chain.out_tokens)
    for b in range(B):
        n = int(chain.num_emitted[b])
        tested = min(n, K)  # drafts 1..tested were tested
        assert np.allclose(tr.accept_prob[b, 1:1 + tested], chain.accept_prob[b, :tested], rtol=1e-14)
        assert (tr.accept_prob[b, 1 + tested:] == -1).all()


def pin_tree_p_equals_q(orc):
    """p_v = q_v at every node: the first child is always accepted (a = 1),
    so the path follows first children down to a leaf."""
    rng = np.random.default_rng(22)
    V = 6
    par = [-1, 0, 0, 1, 1, 2, 3]
    tok = [0, 1, 2, 3, 4, 5, 0]
    P = rng.dirichlet(np.ones(V), 7)
    for _ in range(50):
        r = _tree_probs(orc, P, P, par, tok, rng.random(7))
        assert list(r.out_nodes[0, :3]) == [1, 3, 6] and r.num_emitted[0] == 4


def pin_tree_invalid_inputs(orc):
    """Parent not before the node, token outside [0, V), q(x) = 0 for a
    drafted token, u outside [0, 1): the sequence emits nothing."""
    P = [[.5, .5]] * 3
    Q = [[.5, .5], [.5, .5], [.5, .5]]
    bad = [([-1, 0, 2], [0, 1, 1], [.1] * 3, Q, 64), ([-1, 0, 0], [0, 1, 2], [.1] * 3, Q, 2),
           ([-1, 0, 0], [0, 1, 0], [.1] * 3, [[1, 0], [.5, .5], [.5, .5]], 4),
           ([-1, 0, 1], [0, 1, 1], [.1, .1, 1.0], Q, 1)]
    for par, tok, u, q, bit in bad:
        r = _tree_probs(orc, P, q, par, tok, u)
        assert r.status[0] & bit and r.num_emitted[0] == 0 and (r.out_tokens[0] == -1).all(), (par, tok, bit)


def pin_tree_keeps_target_distribution(orc):
    """Monte Carlo, 4e5 rounds: siblings drafted i.i.d. from their parent's q
    (with replacement), fresh uniforms.  The first emitted token follows p_0,
    and after an accepted child with token y the next emitted token follows
    that child's row -- chi-square at alpha = 0.001 (the property the pages
    require of a tree; SpecInfer's theorem for this rule)."""
    from scipy import stats
    rng = np.random.default_rng(23)
    V = 4
    # topology: root with 3 children; its first child has 2 children
    par = np.array([-1, 0, 0, 0, 1, 1], np.int32)
    N = len(par)
    p0 = np.array([.4, .3, .2, .1])
    P2 = rng.dirichlet(np.ones(V) * 2, V)      # target after token y: P2[y]
    q0 = np.array([.1, .2, .3, .4])
    Q2 = rng.dirichlet(np.ones(V) * 2, V)      # draft after token y
    P3 = rng.dirichlet(np.ones(V) * 2, V)      # target after the second token (grand-children rows)
    n = 400_000
    tok = np.zeros((n, N), np.int32)
    tok[:, 1:4] = rng.choice(V, (n, 3), p=q0)
    y1 = tok[:, 1]
    cdf = np.cumsum(Q2[y1], -1)
    for c in (4, 5):
        tok[:, c] = np.minimum((rng.random((n, 1)) * cdf[:, -1:] >= cdf).sum(-1), V - 1)
    p = np.empty((n, N, V))
    q = np.empty((n, N, V))
    p[:, 0], q[:, 0] = p0, q0
    for c in (1, 2, 3):
        p[:, c], q[:, c] = P2[tok[:, c]], Q2[tok[:, c]]
    for c in (4, 5):
        p[:, c], q[:, c] = P3[tok[:, c]], 1.0 / V
    r = orc.tree_verify_probs(p, q, np.tile(par, (n, 1)), tok, rng.random((n, N)))
    assert (r.status == 0).all()
    first = np.bincount(r.out_tokens[:, 0], minlength=V)
    assert stats.chisquare(first, p0 * n).pvalue > 1e-3, first / n
    cont = r.num_emitted >= 2
    for y in range(V):
        sel = cont & (r.out_tokens[:, 0] == y)
        if sel.sum() < 1000:
            continue
        h = np.bincount(r.out_tokens[sel, 1], minlength=V)
        assert stats.chisquare(h, P2[y] * sel.sum()).pvalue > 1e-3, (y, h / sel.sum(), P2[y])


ALL_PINS = [
    # cheap first: mutants should fail fast
    pin_worked_example,
    pin_worked_example_probabilities,
    pin_worked_example_residual,
    pin_strict_accept,
    pin_zero_mass_never_drawn,
    pin_final_draw_for_correction,
    pin_first_rejection_discards_rest,
    pin_bonus_uses_last_row,
    pin_temperature_direction,
    pin_bf16_decoding,
    pin_vocab_of_one,
    pin_onehot_draft,
    pin_invalid_inputs,
    pin_p_equals_q,
    pin_k0_is_categorical,
    pin_batch_consistency,
    pin_pointwise_identity,
    pin_bruteforce_tiny,
    pin_filter_closed_forms,
    pin_filter_ties_by_id,
    pin_filter_temperature,
    pin_filter_masked_and_bad_rows,
    pin_filter_bruteforce_tiny,
    pin_filter_topk_matches_library_sort,
    pin_filter_matches_generator_nucleus,
    pin_bf16_round_textbook,
    pin_bf16_round_matches_bit_rounding,
    pin_lm_head_identity_and_permutation,
    pin_lm_head_rectangular_closed_forms,
    pin_lm_head_matches_library_matmul,
    pin_tree_hand_example,
    pin_tree_chain_reduces_to_chain,
    pin_tree_p_equals_q,
    pin_tree_invalid_inputs,
    pin_output_distribution,
    pin_expected_tokens,
    pin_tree_keeps_target_distribution,
]
