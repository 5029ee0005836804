"""Compare a candidate's verification outputs with the fp64 oracle.

TEST INFRASTRUCTURE ONLY (tests, smoke check, bench).

Rule (tokens and counts are index work decided by floating point):
  * accept_prob and residual_mass: within 1e-5 absolute of the oracle.
  * emitted tokens, num_emitted, flags: bit-exact, except a draw whose
    decision the fp64 oracle places within 1e-5 relative of a boundary:
      - an accept test whose uniform u satisfies |u - a| <= 1e-5 * a, or
      - a final draw where every oracle CDF boundary between the oracle's
        token and the candidate's token lies within 1e-5 relative of u.
    Such draws are counted as "excused"; their number must stay below 1e-4
    of all draws.  After an excused accept-test disagreement the rest of the
    sequence is checked against the oracle re-run with that one decision
    forced the candidate's way, so the continuation is still checked exactly.
  * a sequence with invalid input must emit nothing, exactly as the oracle.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

from . import ORC_DEGENERATE_RESIDUAL as _DEGENERATE

TOL_PROB = 1e-5
WINDOW = 1e-5
MAX_EXCUSED_FRACTION = 1e-4


@dataclass
class ParityReport:
    sequences: int = 0
    draws: int = 0
    excused: int = 0
    failures: list = field(default_factory=list)
    max_prob_err: float = 0.0
    max_mass_err: float = 0.0

    @property
    def excused_fraction(self) -> float:
        return self.excused / max(self.draws, 1)

    def ok(self) -> bool:
        return not self.failures and self.excused <= MAX_EXCUSED_FRACTION * self.draws

    def summary(self) -> str:
        s = (f"{self.sequences} sequences, {self.draws} draws, {self.excused} excused "
             f"({self.excused_fraction:.2e}), max |dprob| {self.max_prob_err:.2e}, "
             f"max |dmass| {self.max_mass_err:.2e}, {len(self.failures)} failures")
        if self.failures:
            s += "; first: " + str(self.failures[0])
        return s


def _draws_of(n_emitted: int, K: int) -> int:
    """Uniforms a valid round consumes: the accept tests made plus the final draw."""
    j = n_emitted - 1
    return (j + 1 if j < K else K) + 1


def _forced_u(a: float, accept: bool) -> np.float32 | None:
    """A float32 uniform that makes the oracle take `accept` at threshold a."""
    if accept:
        return np.float32(0.0) if a > 0 else None
    v = np.float32(a)
    if float(v) < a:
        v = np.nextafter(v, np.float32(1))
    return v if float(v) < 1.0 else None


def compare(orc, inp_logits, inp_q, inp_tokens, inp_u, T, cand, oracle_res=None,
            seqs=None, report: ParityReport | None = None) -> ParityReport:
    """cand: dict of numpy arrays out_tokens, num_emitted, accept_flags,
    accept_prob (or None), residual_mass (or None), for the same batch.
    seqs: indices of the sequences to check (default: all).  The oracle is
    run on those sequences only."""
    rep = report or ParityReport()
    B, K1, V = inp_logits.shape
    K = K1 - 1
    idx = np.arange(B) if seqs is None else np.asarray(seqs)
    if oracle_res is None:
        oracle_res = orc.verify(inp_logits[idx], None if inp_q is None else inp_q[idx],
                                inp_tokens[idx], inp_u[idx], T, nthreads=8)
        local = True
    else:
        local = False
    for n, b in enumerate(idx):
        o_i = n if local else b
        _check_sequence(orc, inp_logits, inp_q, inp_tokens, inp_u, T, cand, int(b),
                        oracle_res, o_i, rep, depth=0)
        rep.sequences += 1
    return rep


def _single(orc, logits, q, tokens, u_row, T, b):
    return orc.verify(logits[b:b + 1], None if q is None else q[b:b + 1],
                      tokens[b:b + 1], u_row[None], T)


def _check_sequence(orc, logits, q, tokens, u, T, cand, b, ores, oi, rep, depth,
                    u_row=None, k_start=0):
    K = logits.shape[1] - 1
    u_row = u[b].copy() if u_row is None else u_row
    o_tok = ores.out_tokens[oi]
    o_n = int(ores.num_emitted[oi])
    o_flags = ores.accept_flags[oi]
    c_tok = cand["out_tokens"][b]
    c_n = int(cand["num_emitted"][b])
    c_flags = cand["accept_flags"][b] if cand.get("accept_flags") is not None else None
    c_prob = cand.get("accept_prob")
    c_mass = cand.get("residual_mass")

    # bad data (every bit but the degenerate-residual report, which still
    # emits its tokens): the sequence emits nothing
    if int(ores.status[oi]) & ~_DEGENERATE:
        if not (c_n == 0 and (c_tok == -1).all() and
                (c_flags is None or (c_flags == -1).all())):
            rep.failures.append((b, "invalid sequence emitted tokens", int(ores.status[oi])))
        return
    if depth == 0:
        rep.draws += _draws_of(o_n, K)
        if c_prob is not None and K > 0:
            err = float(np.max(np.abs(c_prob[b].astype(np.float64) - ores.accept_prob[oi])))
            rep.max_prob_err = max(rep.max_prob_err, err)
            if not err <= TOL_PROB:
                rep.failures.append((b, "accept_prob", err))

    # accept decisions, left to right
    c_jstar = c_n - 1
    o_jstar = o_n - 1
    for k in range(k_start, K):
        o_acc = k < o_jstar
        c_acc = k < c_jstar
        if o_acc == c_acc:
            if not o_acc:
                break
            continue
        a = float(ores.accept_prob[oi, k])
        if abs(float(u_row[k]) - a) <= WINDOW * a:
            rep.excused += 1
            forced = _forced_u(a, c_acc)
            if forced is None or depth > 4:
                return
            u2 = u_row.copy()
            u2[k] = forced
            r2 = _single(orc, logits, q, tokens, u2, T, b)
            _check_sequence(orc, logits, q, tokens, u, T, cand, b, r2, 0, rep,
                            depth + 1, u_row=u2, k_start=k + 1)
            return
        rep.failures.append((b, f"accept decision at draft {k}", float(u_row[k]), a))
        return

    if c_n != o_n:
        rep.failures.append((b, "num_emitted", c_n, o_n))
        return
    if not np.array_equal(c_tok[:o_jstar], o_tok[:o_jstar]) or not (c_tok[o_n:] == -1).all():
        rep.failures.append((b, "accepted prefix / padding"))
        return
    if c_flags is not None and not np.array_equal(c_flags, o_flags):
        rep.failures.append((b, "accept_flags", c_flags.tolist(), o_flags.tolist()))
        return
    rejected = o_jstar < K
    if c_mass is not None:
        err = abs(float(c_mass[b]) - float(ores.residual_mass[oi]))
        rep.max_mass_err = max(rep.max_mass_err, err)
        if not err <= TOL_PROB:
            rep.failures.append((b, "residual_mass", err))
    g, o = int(c_tok[o_jstar]), int(o_tok[o_jstar])
    if g == o:
        return
    V = logits.shape[2]
    if not 0 <= g < V:
        rep.failures.append((b, "final token out of range", g))
        return
    _, _, cdf, _ = orc.row_dists(logits, q, tokens, T, b, o_jstar, rejected)
    uk = float(u_row[K])
    if g > o:
        worst = cdf[g - 1]
        excusable = worst <= uk * (1 + WINDOW)
    else:
        worst = cdf[g]
        excusable = worst >= uk * (1 - WINDOW)
    if excusable:
        rep.excused += 1
    else:
        rep.failures.append((b, "final token", g, o, uk, float(worst)))


# ------------------------------------------------ top-k / top-p filtering

FILTER_WINDOW = 1e-5


@dataclass
class FilterReport:
    rows: int = 0
    excused: list = field(default_factory=list)    # (row, oracle kept, candidate kept)
    failures: list = field(default_factory=list)   # (row, reason)

    def ok(self, max_excused_fraction: float = 1e-3) -> bool:
        return not self.failures and len(self.excused) <= max(1, max_excused_fraction * self.rows)

    def summary(self) -> str:
        return (f"{self.rows} rows, {len(self.excused)} excused, {len(self.failures)} failures"
                + (f"; first failure {self.failures[0]}" if self.failures else ""))


def compare_filter(orc, logits, T, top_k, top_p, cand_out, cand_kept) -> FilterReport:
    """Filtered rows of a candidate against the oracle's.  A row must match
    the oracle bit for bit, except when the two keep different numbers of
    ids and every cumulative mass between the two cuts lies within
    FILTER_WINDOW (relative) of the top-p target: then the candidate's row
    must still be exactly the oracle's order cut at the candidate's count,
    and the row is counted as excused.  Top-k counts are never excused."""
    logits = np.ascontiguousarray(logits)
    V = logits.shape[-1]
    flat_in = logits.reshape(-1, V)
    ref = orc.filter_logits(flat_in, T, top_k, top_p)
    flat_c = np.ascontiguousarray(cand_out).reshape(-1, V)
    kept_c = np.asarray(cand_kept).reshape(-1)
    rep = FilterReport(rows=flat_in.shape[0])
    neg = np.uint16(0xFF80) if flat_in.dtype == np.uint16 else np.float32(-np.inf)
    for r in range(flat_in.shape[0]):
        a = ref.logits[r].view(np.uint16 if flat_in.dtype == np.uint16 else np.uint32)
        b = flat_c[r].view(a.dtype)
        if np.array_equal(a, b) and int(kept_c[r]) == int(ref.kept[r]):
            continue
        order = orc.filter_order(flat_in, r, T, top_k, top_p)
        if order is None or ref.status[r] != 0:
            rep.failures.append((r, "bad row not copied unchanged"))
            continue
        ng, no = int(kept_c[r]), int(ref.kept[r])
        if not (1 <= ng <= order.n_topk):
            rep.failures.append((r, f"kept {ng} outside [1, {order.n_topk}]"))
            continue
        want = flat_in[r].copy()
        drop = order.ids[ng:]
        want[drop] = neg
        if not np.array_equal(want.view(a.dtype), b):
            rep.failures.append((r, f"row is not the order cut at {ng}"))
            continue
        lo, hi = min(ng, no), max(ng, no)
        tau = order.tau
        if all(abs(order.cum[n - 1] - tau) <= FILTER_WINDOW * tau for n in range(lo, hi)):
            rep.excused.append((r, no, ng))
        else:
            rep.failures.append((r, f"kept {ng} vs oracle {no} outside the window"))
    return rep


# ------------------------------------------------ tree verification

@dataclass
class TreeReport:
    sequences: int = 0
    draws: int = 0
    excused: int = 0
    failures: list = field(default_factory=list)
    max_prob_err: float = 0.0

    def ok(self) -> bool:
        return not self.failures and self.excused <= MAX_EXCUSED_FRACTION * self.draws

    def summary(self) -> str:
        s = (f"{self.sequences} sequences, {self.draws} draws, {self.excused} excused, "
             f"max |dprob| {self.max_prob_err:.2e}, {len(self.failures)} failures")
        if self.failures:
            s += "; first: " + str(self.failures[0])
        return s


def compare_tree(orc, logits, q, parent, tokens, u, T, cand, seqs=None) -> TreeReport:
    """Tree outputs of a candidate (dict of numpy arrays out_tokens,
    out_nodes, num_emitted, accept_prob or None) against the oracle's, by
    the same rule as the chain: the path, tokens and count exactly, except a
    decision whose uniform the fp64 oracle places within 1e-5 relative of
    its threshold (an accept test with |u - a| <= 1e-5 a, or a final draw
    whose token moves to the candidate's when u[0] moves by at most 1e-5
    relative); such draws are excused (at most 1e-4 of all draws) and after
    an excused accept test the rest is checked against the oracle re-run
    with that decision forced the candidate's way.  accept_prob of the tested
    nodes within 1e-5 absolute; a sequence with invalid input emits nothing."""
    rep = TreeReport()
    B = logits.shape[0]
    idx = np.arange(B) if seqs is None else np.asarray(seqs)
    ores = orc.tree_verify(logits[idx], q[idx], parent[idx], tokens[idx], u[idx], T)
    for n, b in enumerate(idx):
        _check_tree(orc, logits, q, parent, tokens, u[b].copy(), T, cand, int(b), ores, n, rep, 0)
        rep.sequences += 1
    return rep


def _tree_single(orc, logits, q, parent, tokens, u_row, T, b):
    return orc.tree_verify(logits[b:b + 1], q[b:b + 1], parent[b:b + 1], tokens[b:b + 1], u_row[None], T)


def _check_tree(orc, logits, q, parent, tokens, u_row, T, cand, b, ores, oi, rep, depth):
    N = logits.shape[1]
    o_tok, o_nodes, o_n = ores.out_tokens[oi], ores.out_nodes[oi], int(ores.num_emitted[oi])
    o_prob = ores.accept_prob[oi]
    c_tok, c_n = cand["out_tokens"][b], int(cand["num_emitted"][b])
    c_nodes = cand["out_nodes"][b] if cand.get("out_nodes") is not None else None
    c_prob = cand.get("accept_prob")
    if int(ores.status[oi]) & ~_DEGENERATE:
        if not (c_n == 0 and (c_tok == -1).all()):
            rep.failures.append((b, "invalid sequence emitted tokens", int(ores.status[oi])))
        return
    if depth == 0:
        rep.draws += int((o_prob >= 0).sum()) + 1
    if c_nodes is None:
        rep.failures.append((b, "out_nodes missing"))
        return
    L = o_n - 1
    cL = c_n - 1
    # the first node where the two walks decide differently
    d = 0
    while d < min(L, cL) and o_nodes[d] == c_nodes[d]:
        d += 1
    if d < L or d < cL:
        cands = [int(x) for x in ((o_nodes[d] if d < L else None), (c_nodes[d] if d < cL else None)) if x is not None]
        s = min(cands)  # the earlier sibling: one side accepted it, the other rejected it
        c_acc = d < cL and c_nodes[d] == s
        a = float(o_prob[s]) if 0 <= s < N else -1.0
        if a >= 0 and abs(float(u_row[s]) - a) <= WINDOW * a:
            rep.excused += 1
            forced = _forced_u(a, c_acc)
            if forced is None or depth > 4:
                return
            u2 = u_row.copy()
            u2[s] = forced
            r2 = _tree_single(orc, logits, q, parent, tokens, u2, T, b)
            _check_tree(orc, logits, q, parent, tokens, u2, T, cand, b, r2, 0, rep, depth + 1)
            return
        rep.failures.append((b, f"accept decision at node {s}", float(u_row[s]) if s < N else None, a))
        return
    if not (c_tok[c_n:] == -1).all() or not (c_nodes[L:] == -1).all():
        rep.failures.append((b, "padding"))
        return
    if not np.array_equal(c_tok[:L], o_tok[:L]):
        rep.failures.append((b, "path tokens"))
        return
    if c_prob is not None and depth == 0:
        tested = o_prob >= 0
        err = float(np.max(np.abs(c_prob[b][tested].astype(np.float64) - o_prob[tested]))) if tested.any() else 0.0
        rep.max_prob_err = max(rep.max_prob_err, err)
        if not err <= TOL_PROB:
            rep.failures.append((b, "accept_prob", err))
        if not (c_prob[b][~tested] == -1).all():
            rep.failures.append((b, "accept_prob of untested nodes"))
    g, o = int(c_tok[L]), int(o_tok[L])
    if g == o:
        return
    # the final draw: excused if moving u[0] by 1e-5 relative reaches g
    lo, hi = u_row.copy(), u_row.copy()
    lo[0] = np.float32(float(u_row[0]) * (1 - WINDOW))
    hi[0] = min(np.float32(float(u_row[0]) * (1 + WINDOW)), np.nextafter(np.float32(1), np.float32(0)))
    y_lo = int(_tree_single(orc, logits, q, parent, tokens, lo, T, b).out_tokens[0, L])
    y_hi = int(_tree_single(orc, logits, q, parent, tokens, hi, T, b).out_tokens[0, L])
    if min(y_lo, y_hi) <= g <= max(y_lo, y_hi):
        rep.excused += 1
    else:
        rep.failures.append((b, "final token", g, o, float(u_row[0])))
