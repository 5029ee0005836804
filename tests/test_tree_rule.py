"""The tree comparison rule itself (CPU).

Candidates are built from the oracle's own tree outputs: exact copies must
pass, planted mistakes must fail, and a decision flipped by an amount inside
the 1e-5 window around its boundary must be counted as excused."""
import numpy as np
import pytest

import synth
from oracle import parity

SHAPE = synth.TREE_SHAPES["tree16"]


def _inputs(seed=3, B=24, V=400):
    w = synth.WORKLOADS["b8_k4_v32000_bf16"].with_(B=B, V=V, dtype="fp32")
    return synth.tree_inputs(w, SHAPE, seed=seed)


def _cand(r):
    return {"out_tokens": r.out_tokens.copy(), "out_nodes": r.out_nodes.copy(),
            "num_emitted": r.num_emitted.copy(), "accept_prob": r.accept_prob.astype(np.float32)}


def test_exact_candidate_passes(orc):
    lg, q, par, tok, u, T = _inputs()
    rep = parity.compare_tree(orc, lg, q, par, tok, u, T, _cand(orc.tree_verify(lg, q, par, tok, u, T)))
    assert rep.ok() and rep.excused == 0 and rep.sequences == lg.shape[0]


@pytest.mark.parametrize("mistake", ["final", "path_node", "count", "prob", "untested_prob", "padding"])
def test_planted_mistakes_fail(orc, mistake):
    lg, q, par, tok, u, T = _inputs()
    res = orc.tree_verify(lg, q, par, tok, u, T)
    c = _cand(res)
    # a sequence whose path has at least one accepted node
    b = int(np.nonzero(res.num_emitted >= 2)[0][0])
    n = int(c["num_emitted"][b])
    V = lg.shape[2]
    if mistake == "final":
        c["out_tokens"][b, n - 1] = (c["out_tokens"][b, n - 1] + 1) % V
    elif mistake == "path_node":
        c["out_nodes"][b, 0] = (c["out_nodes"][b, 0] % (len(SHAPE) - 1)) + 1 if c["out_nodes"][b, 0] != 1 else 2
    elif mistake == "count":
        c["num_emitted"][b] = n - 1
    elif mistake == "prob":
        tested = np.nonzero(res.accept_prob[b] >= 0)[0]
        c["accept_prob"][b, tested[0]] += 1e-4
    elif mistake == "untested_prob":
        untested = np.nonzero(res.accept_prob[b] < 0)[0]
        c["accept_prob"][b, untested[-1]] = 0.5
    else:
        c["out_tokens"][b, len(SHAPE) - 1] = 7 if n < len(SHAPE) else c["out_tokens"][b, -1]
    rep = parity.compare_tree(orc, lg, q, par, tok, u, T, c)
    assert not rep.ok(), (mistake, rep.summary())


def test_decision_inside_the_window_is_excused(orc):
    """Move a tested node's uniform to 3e-6 (relative) across its threshold:
    the oracle flips that decision; the unmoved candidate is excused.  The
    same move 3e-3 away is a failure."""
    lg, q, par, tok, u, T = _inputs()
    res = orc.tree_verify(lg, q, par, tok, u, T)
    cand = _cand(res)
    # the first tested node with a threshold well inside (0, 1)
    hits = [(b, c) for b in range(lg.shape[0]) for c in range(1, len(SHAPE))
            if 0.05 < res.accept_prob[b, c] < 0.95]
    b, c = hits[0]
    a = float(res.accept_prob[b, c])
    for rel, ok in ((3e-6, True), (3e-3, False)):
        u2 = u.copy()
        accepted = u[b, c] < a
        # put u just on the other side of a: the oracle re-run decides the other way
        u2[b, c] = np.float32(a * (1 + rel)) if accepted else np.float32(a * (1 - rel))
        rep = parity.compare_tree(orc, lg, q, par, tok, u2, T, cand, seqs=[b])
        if ok:  # excused, not failed (one excused draw of five is over the 1e-4 share on its own)
            assert not rep.failures and rep.excused >= 1, rep.summary()
        else:
            assert rep.failures, rep.summary()


def test_invalid_sequence_must_emit_nothing(orc):
    lg, q, par, tok, u, T = _inputs()
    par = par.copy()
    par[0, 5] = 9  # a parent after its node
    res = orc.tree_verify(lg, q, par, tok, u, T)
    assert res.status[0] & 64 and res.num_emitted[0] == 0
    c = _cand(res)
    c["num_emitted"][0] = 1
    c["out_tokens"][0, 0] = 3
    rep = parity.compare_tree(orc, lg, q, par, tok, u, T, c)
    assert not rep.ok()
