"""fp64 CPU oracle for the speculative-sampling verification step.

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the
bench's CPU-baseline leg are the only callers.  The product library never
imports this package, and this package never imports the product.

The arithmetic lives in ``sv_oracle.c`` (plain C, fp64, sequential sums in
token-id order); this module only compiles it with gcc and marshals numpy
arrays through ctypes.  See the header of ``sv_oracle.c`` for the pages and
sections each step follows.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from dataclasses import dataclass

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "sv_oracle.c")
_LIB_DIR = os.path.join(_HERE, "_build")
_LIB = os.path.join(_LIB_DIR, "libsvoracle.so")

# per-sequence status bits, as the oracle reports them
ORC_BAD_U = 1
ORC_BAD_TOKEN = 2
ORC_BAD_Q = 4
ORC_BAD_ROW = 8
ORC_DEGENERATE_RESIDUAL = 16
ORC_BAD_TREE = 64

_c_i32p = ctypes.POINTER(ctypes.c_int32)
_c_i8p = ctypes.POINTER(ctypes.c_int8)
_c_f64p = ctypes.POINTER(ctypes.c_double)


def compile_oracle(src: str = _SRC, out: str = _LIB) -> str:
    """Compile an oracle source file into a shared library (gcc, -O2).

    ``-ffp-contract=off`` keeps gcc from fusing multiply-adds, so x86 and
    aarch64 builds round identically.
    """
    os.makedirs(os.path.dirname(out), exist_ok=True)
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off",
           "-pthread", "-o", out, src, "-lm"]
    subprocess.run(cmd, check=True)
    return out


def build() -> str:
    """Compile ``sv_oracle.c`` if the library is missing or stale."""
    if (not os.path.exists(_LIB)
            or os.path.getmtime(_LIB) < os.path.getmtime(_SRC)):
        compile_oracle()
    return _LIB


def _bind(lib: ctypes.CDLL) -> ctypes.CDLL:
    lib.sv_oracle_verify.restype = ctypes.c_int
    lib.sv_oracle_verify.argtypes = [
        ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p,
        ctypes.c_void_p, ctypes.c_double, ctypes.c_int64, ctypes.c_int32,
        ctypes.c_int32, _c_i32p, _c_i32p, _c_i8p, _c_f64p, _c_f64p, _c_i32p,
        ctypes.c_int]
    lib.sv_oracle_verify_probs.restype = ctypes.c_int
    lib.sv_oracle_verify_probs.argtypes = [
        ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
        ctypes.c_int64, ctypes.c_int32, ctypes.c_int32, _c_i32p, _c_i32p,
        _c_i8p, _c_f64p, _c_f64p, _c_i32p, ctypes.c_int]
    lib.sv_oracle_row_dists.restype = ctypes.c_double
    lib.sv_oracle_row_dists.argtypes = [
        ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p,
        ctypes.c_double, ctypes.c_int64, ctypes.c_int32, ctypes.c_int32,
        ctypes.c_int32, ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p,
        ctypes.c_void_p]
    lib.sv_oracle_filter_logits.restype = ctypes.c_int
    lib.sv_oracle_filter_logits.argtypes = [
        ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_int32, ctypes.c_double,
        ctypes.c_int32, ctypes.c_double, ctypes.c_void_p, _c_i32p, _c_i32p, ctypes.c_int]
    lib.sv_oracle_lm_head_entry.restype = ctypes.c_double
    lib.sv_oracle_lm_head_entry.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64,
                                            ctypes.c_int64]
    lib.sv_oracle_lm_head.restype = ctypes.c_int
    lib.sv_oracle_lm_head.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32,
                                      ctypes.c_int32, ctypes.c_void_p]
    lib.sv_oracle_bf16_round.restype = None
    lib.sv_oracle_bf16_round.argtypes = [ctypes.c_void_p, ctypes.c_int64, ctypes.c_void_p]
    lib.sv_oracle_tree_verify.restype = ctypes.c_int
    lib.sv_oracle_tree_verify.argtypes = [
        ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
        ctypes.c_double, ctypes.c_int64, ctypes.c_int32, ctypes.c_int32,
        ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p]
    lib.sv_oracle_tree_verify_probs.restype = ctypes.c_int
    lib.sv_oracle_tree_verify_probs.argtypes = [
        ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
        ctypes.c_int64, ctypes.c_int32, ctypes.c_int32,
        ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p]
    lib.sv_oracle_filter_order.restype = ctypes.c_int32
    lib.sv_oracle_filter_order.argtypes = [
        ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_int32, ctypes.c_double,
        ctypes.c_int32, ctypes.c_double, _c_i32p, _c_f64p, _c_i32p, _c_f64p]
    return lib


@dataclass
class FilterResult:
    logits: np.ndarray   # the filtered rows, same dtype and shape as the input
    kept: np.ndarray     # int32 [rows]: ids kept (0 for a bad row)
    status: np.ndarray   # int32 [rows]: ORC_BAD_ROW for a row copied unchanged


@dataclass
class FilterOrder:
    ids: np.ndarray      # int32 [n]: the finite ids in filter order
    cum: np.ndarray      # fp64 [n]: cumulative unnormalised mass in that order
    n_topk: int          # ids the top-k step keeps
    tau: float           # mass the top-p step must reach


_loaded: dict[str, "Oracle"] = {}


@dataclass
class OracleResult:
    out_tokens: np.ndarray     # int32 [B, K+1], -1 padded
    num_emitted: np.ndarray    # int32 [B], 0 for an invalid sequence
    accept_flags: np.ndarray   # int8  [B, K]: 1 accepted, 0 rejected, -1 not reached
    accept_prob: np.ndarray    # fp64  [B, K]: min(1, p(x)/q(x)) for every draft
    residual_mass: np.ndarray  # fp64  [B]: sum max(0, p-q) at the rejection, 0 on bonus
    status: np.ndarray         # int32 [B]: ORC_* bits


class Oracle:
    """ctypes handle on one compiled oracle library."""

    def __init__(self, path: str):
        self.path = path
        self.lib = _bind(ctypes.CDLL(path))

    @staticmethod
    def _outputs(B: int, K: int):
        return (np.empty((B, K + 1), np.int32), np.empty(B, np.int32),
                np.empty((B, K), np.int8), np.empty((B, K), np.float64),
                np.empty(B, np.float64), np.empty(B, np.int32))

    @staticmethod
    def _ptr(a, ct):
        return a.ctypes.data_as(ct)

    def verify(self, logits: np.ndarray, q: np.ndarray | None,
               tokens: np.ndarray, u: np.ndarray, T: float,
               nthreads: int = 1) -> OracleResult:
        """logits: [B,K+1,V] uint16 (bf16 bits) or float32; q: [B,K,V]
        float32 or None (one-hot drafts); tokens [B,K] int32; u [B,K+1] float32."""
        logits = np.ascontiguousarray(logits)
        if logits.dtype == np.uint16:
            dtype = 0
        elif logits.dtype == np.float32:
            dtype = 1
        else:
            raise TypeError("logits must be uint16 (bf16 bits) or float32")
        B, K1, V = logits.shape
        K = K1 - 1
        tokens = np.ascontiguousarray(tokens, dtype=np.int32).reshape(B, K)
        u = np.ascontiguousarray(u, dtype=np.float32).reshape(B, K + 1)
        if q is not None:
            q = np.ascontiguousarray(q, dtype=np.float32).reshape(B, K, V)
        outs = self._outputs(B, K)
        rc = self.lib.sv_oracle_verify(
            logits.ctypes.data, dtype, None if q is None else q.ctypes.data,
            tokens.ctypes.data, u.ctypes.data, float(T), B, K, V,
            self._ptr(outs[0], _c_i32p), self._ptr(outs[1], _c_i32p),
            self._ptr(outs[2], _c_i8p), self._ptr(outs[3], _c_f64p),
            self._ptr(outs[4], _c_f64p), self._ptr(outs[5], _c_i32p),
            int(nthreads))
        if rc != 0:
            raise RuntimeError("sv_oracle_verify failed")
        return OracleResult(*outs)

    def verify_probs(self, p: np.ndarray, q: np.ndarray | None,
                     tokens: np.ndarray, u: np.ndarray,
                     nthreads: int = 1) -> OracleResult:
        """p: [B,K+1,V] fp64 probabilities; q: [B,K,V] fp64 or None;
        tokens [B,K]; u [B,K+1] fp64."""
        p = np.ascontiguousarray(p, dtype=np.float64)
        B, K1, V = p.shape
        K = K1 - 1
        tokens = np.ascontiguousarray(tokens, dtype=np.int32).reshape(B, K)
        u = np.ascontiguousarray(u, dtype=np.float64).reshape(B, K + 1)
        if q is not None:
            q = np.ascontiguousarray(q, dtype=np.float64).reshape(B, K, V)
        outs = self._outputs(B, K)
        rc = self.lib.sv_oracle_verify_probs(
            p.ctypes.data, None if q is None else q.ctypes.data,
            tokens.ctypes.data, u.ctypes.data, B, K, V,
            self._ptr(outs[0], _c_i32p), self._ptr(outs[1], _c_i32p),
            self._ptr(outs[2], _c_i8p), self._ptr(outs[3], _c_f64p),
            self._ptr(outs[4], _c_f64p), self._ptr(outs[5], _c_i32p),
            int(nthreads))
        if rc != 0:
            raise RuntimeError("sv_oracle_verify_probs failed")
        return OracleResult(*outs)

    def row_dists(self, logits: np.ndarray, q: np.ndarray | None,
                  tokens: np.ndarray, T: float, b: int, j: int,
                  rejected: bool):
        """(p, w, cdf, Z) of row j of sequence b: the softmax, the normalised
        distribution the final token is drawn from (residual if `rejected`,
        else p), its running sum in id order, and the unnormalised mass."""
        logits = np.ascontiguousarray(logits)
        dtype = 0 if logits.dtype == np.uint16 else 1
        B, K1, V = logits.shape
        K = K1 - 1
        tokens = np.ascontiguousarray(tokens, dtype=np.int32).reshape(B, K)
        if q is not None:
            q = np.ascontiguousarray(q, dtype=np.float32).reshape(B, K, V)
        p = np.empty(V, np.float64)
        w = np.empty(V, np.float64)
        cdf = np.empty(V, np.float64)
        Z = self.lib.sv_oracle_row_dists(
            logits.ctypes.data, dtype, None if q is None else q.ctypes.data,
            tokens.ctypes.data, float(T), int(b), K, V, int(j),
            1 if rejected else 0, p.ctypes.data, w.ctypes.data,
            cdf.ctypes.data)
        if Z < 0:
            raise ValueError("invalid row")
        return p, w, cdf, Z


    @staticmethod
    def _dtype_of(logits: np.ndarray) -> int:
        if logits.dtype == np.uint16:
            return 0
        if logits.dtype == np.float32:
            return 1
        raise TypeError("logits must be uint16 (bf16 bits) or float32")

    def filter_logits(self, logits: np.ndarray, T: float, top_k: int = 0,
                      top_p: float = 1.0, nthreads: int = 1) -> FilterResult:
        """Top-k / top-p filtering of the rows of `logits` (last axis = V) at
        temperature T: the ids outside the kept set become -inf."""
        logits = np.ascontiguousarray(logits)
        dtype = self._dtype_of(logits)
        V = logits.shape[-1]
        rows = logits.size // V if V else 0
        out = np.empty_like(logits)
        kept = np.empty(rows, np.int32)
        status = np.empty(rows, np.int32)
        rc = self.lib.sv_oracle_filter_logits(
            logits.ctypes.data, dtype, rows, V, float(T), int(top_k), float(top_p),
            out.ctypes.data, self._ptr(kept, _c_i32p), self._ptr(status, _c_i32p), int(nthreads))
        if rc != 0:
            raise ValueError("sv_oracle_filter_logits rejected its arguments")
        return FilterResult(out, kept, status)

    def filter_order(self, logits: np.ndarray, row: int, T: float, top_k: int = 0,
                     top_p: float = 1.0) -> FilterOrder | None:
        """The filter order of one row (None for a bad row)."""
        logits = np.ascontiguousarray(logits)
        dtype = self._dtype_of(logits)
        V = logits.shape[-1]
        ids = np.empty(V, np.int32)
        cum = np.empty(V, np.float64)
        nk = ctypes.c_int32(0)
        tau = ctypes.c_double(0.0)
        n = self.lib.sv_oracle_filter_order(
            logits.ctypes.data, dtype, int(row), V, float(T), int(top_k), float(top_p),
            self._ptr(ids, _c_i32p), self._ptr(cum, _c_f64p), ctypes.byref(nk), ctypes.byref(tau))
        if n < 0:
            return None
        return FilterOrder(ids[:n].copy(), cum[:n].copy(), int(nk.value), float(tau.value))


def _lm_inputs(h: np.ndarray, W: np.ndarray):
    h = np.ascontiguousarray(h, dtype=np.uint16)
    W = np.ascontiguousarray(W, dtype=np.uint16)
    if h.ndim != 2 or W.ndim != 2 or h.shape[1] != W.shape[1]:
        raise ValueError("h [M, d] and W [V, d] bf16 bit patterns with the same d")
    return h, W


def _lm_head(self, h: np.ndarray, W: np.ndarray) -> np.ndarray:
    """logits = h W^T in fp64 from bf16 bit patterns h [M, d], W [V, d]."""
    h, W = _lm_inputs(h, W)
    M, d = h.shape
    V = W.shape[0]
    out = np.empty((M, V), np.float64)
    if self.lib.sv_oracle_lm_head(h.ctypes.data, W.ctypes.data, M, d, V, out.ctypes.data) != 0:
        raise RuntimeError("sv_oracle_lm_head failed")
    return out


def _lm_head_entries(self, h: np.ndarray, W: np.ndarray, rows, cols) -> np.ndarray:
    """The entries (rows[i], cols[i]) of h W^T, fp64."""
    h, W = _lm_inputs(h, W)
    d = h.shape[1]
    return np.array([self.lib.sv_oracle_lm_head_entry(h.ctypes.data, W.ctypes.data, d, int(r), int(c))
                     for r, c in zip(rows, cols)], np.float64)


def _bf16_round(self, x: np.ndarray) -> np.ndarray:
    """fp64 values rounded once to bf16 (nearest, ties to even); bit patterns."""
    x = np.ascontiguousarray(x, dtype=np.float64)
    out = np.empty(x.shape, np.uint16)
    self.lib.sv_oracle_bf16_round(x.ctypes.data, x.size, out.ctypes.data)
    return out


@dataclass
class TreeResult:
    out_tokens: np.ndarray   # [B, N] accepted path's tokens, then the final token, -1 padded
    out_nodes: np.ndarray    # [B, N] node ids of the accepted path, -1 padded
    num_emitted: np.ndarray  # [B]
    accept_prob: np.ndarray  # [B, N] min(1, r(x)/q(x)) of each tested node, -1 if not tested
    status: np.ndarray       # [B]


def _tree_out(B, N):
    return TreeResult(np.empty((B, N), np.int32), np.empty((B, N), np.int32), np.empty(B, np.int32),
                      np.empty((B, N), np.float64), np.empty(B, np.int32))


def _tree_call(fn, head, o: TreeResult, B, N, V):
    rc = fn(*head, B, N, V, o.out_tokens.ctypes.data, o.out_nodes.ctypes.data, o.num_emitted.ctypes.data,
            o.accept_prob.ctypes.data, o.status.ctypes.data)
    if rc != 0:
        raise ValueError(f"tree oracle refused the call ({rc})")
    return o


def _tree_verify(self, logits: np.ndarray, q: np.ndarray, parent: np.ndarray, tokens: np.ndarray,
                 u: np.ndarray, T: float) -> TreeResult:
    """Tree verification from logits [B, N, V] (bf16 bits or fp32), q fp32
    [B, N, V], parent / tokens int32 [B, N], u fp32 [B, N]."""
    logits = np.ascontiguousarray(logits)
    B, N, V = logits.shape
    q = np.ascontiguousarray(q, np.float32)
    parent = np.ascontiguousarray(parent, np.int32)
    tokens = np.ascontiguousarray(tokens, np.int32)
    u = np.ascontiguousarray(u, np.float32)
    assert q.shape == (B, N, V) and parent.shape == (B, N) and tokens.shape == (B, N) and u.shape == (B, N)
    head = (logits.ctypes.data, self._dtype_of(logits), q.ctypes.data, parent.ctypes.data, tokens.ctypes.data,
            u.ctypes.data, float(T))
    return _tree_call(self.lib.sv_oracle_tree_verify, head, _tree_out(B, N), B, N, V)


def _tree_verify_probs(self, p: np.ndarray, q: np.ndarray, parent: np.ndarray, tokens: np.ndarray,
                       u: np.ndarray) -> TreeResult:
    """Tree verification from probabilities p, q [B, N, V] fp64, u [B, N] fp64."""
    p = np.ascontiguousarray(p, np.float64)
    B, N, V = p.shape
    q = np.ascontiguousarray(q, np.float64)
    parent = np.ascontiguousarray(parent, np.int32)
    tokens = np.ascontiguousarray(tokens, np.int32)
    u = np.ascontiguousarray(u, np.float64)
    assert q.shape == (B, N, V) and parent.shape == (B, N) and tokens.shape == (B, N) and u.shape == (B, N)
    head = (p.ctypes.data, q.ctypes.data, parent.ctypes.data, tokens.ctypes.data, u.ctypes.data)
    return _tree_call(self.lib.sv_oracle_tree_verify_probs, head, _tree_out(B, N), B, N, V)


Oracle.tree_verify = _tree_verify
Oracle.tree_verify_probs = _tree_verify_probs
Oracle.lm_head = _lm_head
Oracle.lm_head_entries = _lm_head_entries
Oracle.bf16_round = _bf16_round


def load(path: str | None = None) -> Oracle:
    """The oracle library at `path` (default: build and load sv_oracle.c)."""
    path = path or build()
    if path not in _loaded:
        _loaded[path] = Oracle(path)
    return _loaded[path]
