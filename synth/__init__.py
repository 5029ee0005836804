"""Seeded synthetic inputs for the speculative-sampling verification step.

The generator (``synth.c``, Philox4x32-10, multithreaded) writes the same
host bytes that both the CUDA library and the oracle consume; it contains
none of the verification arithmetic.  Workloads follow the shapes and value
distributions of the five configurations the verification step is measured
on (see ``WORKLOADS``); the pages' own evaluation data (ShareGPT, GSM8K,
MBPP on DeepSeek-V4-Flash) is not available, and these distributions stand
in for it.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from dataclasses import dataclass, replace

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "synth.c")
_LIB = os.path.join(_HERE, "_build", "libsynth.so")

DEFAULT_SEED = 20261202


class _Cfg(ctypes.Structure):
    _fields_ = [("dtype", ctypes.c_int), ("K", ctypes.c_int32),
                ("V", ctypes.c_int32), ("sigma", ctypes.c_double),
                ("zipf_s", ctypes.c_double), ("T", ctypes.c_double),
                ("draft_sigma", ctypes.c_double), ("Tq", ctypes.c_double),
                ("top_p", ctypes.c_double), ("onehot_p", ctypes.c_double)]


@dataclass(frozen=True)
class Workload:
    """One input recipe.  dtype: "bf16" or "fp32"; Tq = 0 means one-hot
    drafts (no q tensor)."""
    name: str
    B: int
    K: int
    V: int
    dtype: str
    sigma: float
    zipf_s: float
    T: float
    draft_sigma: float
    Tq: float
    top_p: float = 0.0
    onehot_p: float = 0.0

    @property
    def onehot(self) -> bool:
        return self.Tq <= 0.0

    def with_(self, **kw) -> "Workload":
        return replace(self, **kw)


WORKLOADS = {
    # B=1, K=4, V=32000: fp32 logits N(0, 2^2); q = softmax(z + N(0, .5^2)); T=1
    "b1_k4_v32000_fp32": Workload("b1_k4_v32000_fp32", 1, 4, 32000, "fp32",
                                  2.0, 0.0, 1.0, 0.5, 1.0),
    # B=8, K=4, V=32000: bf16 N(0, 3^2) + Zipf(1.1); q from z + N(0, 1); T=.8 on both
    "b8_k4_v32000_bf16": Workload("b8_k4_v32000_bf16", 8, 4, 32000, "bf16",
                                  3.0, 1.1, 0.8, 1.0, 0.8),
    # B=64, K=5, V=128256: bf16 N(0, 3^2) + Zipf(1.1); q from z + N(0, .7^2);
    # T=1; top-p 0.9 on both p and q
    "b64_k5_v128256_bf16_topp": Workload("b64_k5_v128256_bf16_topp", 64, 5,
                                         128256, "bf16", 3.0, 1.1, 1.0, 0.7,
                                         1.0, top_p=0.9),
    # B=256, K=8, V=151936: bf16 N(0, 4^2) + Zipf(1.2); q from z + N(0, 1.5^2); T=.7
    "b256_k8_v151936_bf16": Workload("b256_k8_v151936_bf16", 256, 8, 151936,
                                     "bf16", 4.0, 1.2, 0.7, 1.5, 0.7),
    # B=128, K=8, V=128256: bf16 N(0, 3^2) + Zipf(1.1); T=.7; one-hot drafts:
    # the target argmax with probability 0.6, else uniform over V
    "b128_k8_v128256_bf16_onehot": Workload("b128_k8_v128256_bf16_onehot", 128,
                                            8, 128256, "bf16", 3.0, 1.1, 0.7,
                                            0.0, 0.0, onehot_p=0.6),
}
# the five configurations in their usual order
CONFIGS = list(WORKLOADS.values())


def compile_synth(out: str = _LIB) -> str:
    os.makedirs(os.path.dirname(out), exist_ok=True)
    subprocess.run(["gcc", "-O2", "-std=c11", "-fPIC", "-shared",
                    "-ffp-contract=off", "-pthread", "-o", out, _SRC, "-lm"],
                   check=True)
    return out


def build() -> str:
    if not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        compile_synth()
    return _LIB


_lib = None


def lib() -> ctypes.CDLL:
    global _lib
    if _lib is None:
        L = ctypes.CDLL(build())
        L.synth_generate.restype = ctypes.c_int
        L.synth_generate.argtypes = [ctypes.POINTER(_Cfg), ctypes.c_uint64,
                                     ctypes.c_int64, ctypes.c_int64,
                                     ctypes.c_void_p, ctypes.c_void_p,
                                     ctypes.c_void_p, ctypes.c_void_p,
                                     ctypes.c_int]
        L.synth_philox4x32_10.restype = None
        L.synth_philox4x32_10.argtypes = [ctypes.c_void_p, ctypes.c_void_p,
                                          ctypes.c_void_p]
        L.synth_f32_to_bf16.restype = None
        L.synth_f32_to_bf16.argtypes = [ctypes.c_void_p, ctypes.c_void_p,
                                        ctypes.c_int64]
        _lib = L
    return _lib


@dataclass
class Inputs:
    """Host inputs of one call.  logits: uint16 bf16 bits or float32."""
    workload: Workload
    logits: np.ndarray        # [B, K+1, V]
    q: np.ndarray | None      # [B, K, V] float32, None for one-hot drafts
    tokens: np.ndarray        # [B, K] int32
    u: np.ndarray             # [B, K+1] float32
    T: float
    b0: int = 0

    @property
    def B(self) -> int:
        return self.logits.shape[0]


def generate(w: Workload | str, seed: int = DEFAULT_SEED, b0: int = 0,
             nb: int | None = None, nthreads: int | None = None) -> Inputs:
    """Sequences [b0, b0+nb) of workload `w` for `seed` (default: all B)."""
    if isinstance(w, str):
        w = WORKLOADS[w]
    nb = w.B - b0 if nb is None else nb
    K, V = w.K, w.V
    cfg = _Cfg(0 if w.dtype == "bf16" else 1, K, V, w.sigma, w.zipf_s, w.T,
               w.draft_sigma, w.Tq, w.top_p, w.onehot_p)
    logits = np.empty((nb, K + 1, V), np.uint16 if w.dtype == "bf16" else np.float32)
    q = None if w.onehot else np.empty((nb, K, V), np.float32)
    tokens = np.empty((nb, K), np.int32)
    u = np.empty((nb, K + 1), np.float32)
    nthreads = nthreads or os.cpu_count() or 1
    rc = lib().synth_generate(ctypes.byref(cfg), seed, b0, nb, logits.ctypes.data,
                              None if q is None else q.ctypes.data,
                              tokens.ctypes.data, u.ctypes.data, int(nthreads))
    if rc != 0:
        raise RuntimeError("synth_generate failed")
    return Inputs(w, logits, q, tokens, u, w.T, b0)


def philox4x32_10(ctr, key) -> list[int]:
    c = (ctypes.c_uint32 * 4)(*ctr)
    k = (ctypes.c_uint32 * 2)(*key)
    o = (ctypes.c_uint32 * 4)()
    lib().synth_philox4x32_10(c, k, o)
    return list(o)


def f32_to_bf16(x: np.ndarray) -> np.ndarray:
    x = np.ascontiguousarray(x, np.float32)
    out = np.empty(x.shape, np.uint16)
    lib().synth_f32_to_bf16(x.ctypes.data, out.ctypes.data, x.size)
    return out


def bf16_to_f32(h: np.ndarray) -> np.ndarray:
    return (np.asarray(h, np.uint16).astype(np.uint32) << 16).view(np.float32)


def lm_head_inputs(M: int, d: int, V: int, seed: int = DEFAULT_SEED, dyadic: bool = False):
    """Seeded hidden states h [M, d] and output embedding W [V, d] as bf16 bit
    patterns (uint16), for the LM-head path.  dyadic=False: h ~ N(0, 1) and
    W ~ N(0, 1/d), rounded to bf16 (logits of order one).  dyadic=True: every
    entry is 0 or +-1/2, so every product is 0 or +-1/4 and every sum of up to
    2^24 of them is exact in fp32 as well as fp64."""
    rng = np.random.default_rng([seed, M, d, V, int(dyadic)])

    def bf16(a):  # round to nearest even
        u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32)
        return ((u + 0x7FFF + ((u >> 16) & 1)) >> 16).astype(np.uint16)

    if dyadic:
        vals = np.array([0xBF00, 0x0000, 0x3F00], np.uint16)   # -1/2, 0, +1/2
        return vals[rng.integers(0, 3, (M, d))], vals[rng.integers(0, 3, (V, d))]
    h = bf16(rng.standard_normal((M, d), dtype=np.float32))
    W = bf16(rng.standard_normal((V, d), dtype=np.float32) / np.float32(np.sqrt(d)))
    return h, W


def drafts_for(z: np.ndarray, T: float, draft_sigma: float, seed: int = DEFAULT_SEED,
               onehot_p: float | None = None):
    """Draft inputs for target logits z [B, K+1, V] (fp64 values) that are
    known only at run time (e.g. the LM head's).  Dense (onehot_p None):
    q = softmax((z + N(0, draft_sigma^2)) / T) over the first K positions,
    tokens drawn from q.  One-hot: tokens the target argmax with probability
    onehot_p, else uniform over V, and q None.  Uniforms U[0, 1) fp32 for
    all K+1 positions.  Returns (q fp32 | None, tokens int32, u fp32)."""
    z = np.asarray(z, np.float64)
    B, K1, V = z.shape
    K = K1 - 1
    rng = np.random.default_rng([seed, B, K, V, 0 if onehot_p is None else 1])
    u = rng.random((B, K1), dtype=np.float32)
    if onehot_p is not None:
        arg = z[:, :K].argmax(-1)
        rand = rng.integers(0, V, (B, K))
        tokens = np.where(rng.random((B, K)) < onehot_p, arg, rand).astype(np.int32)
        return None, tokens, u
    q = np.empty((B, K, V), np.float32)
    tokens = np.empty((B, K), np.int32)
    for b0 in range(0, B, 8):  # a few sequences at a time: bounded host memory
        b1 = min(B, b0 + 8)
        zq = (z[b0:b1, :K] + draft_sigma * rng.standard_normal((b1 - b0, K, V))) / T
        zq -= zq.max(-1, keepdims=True)
        e = np.exp(zq)
        qq = e / e.sum(-1, keepdims=True)
        cdf = np.cumsum(qq, -1)
        t = rng.random((b1 - b0, K, 1)) * cdf[..., -1:]
        tokens[b0:b1] = np.minimum((cdf <= t).sum(-1), V - 1)
        q[b0:b1] = qq
    return q, tokens, u


# Candidate-tree shapes (parent of each node; node 0 is the committed prefix).
TREE_SHAPES = {
    # 16 nodes, depth 5: the root has 3 children, its first child 3, ...
    "tree16": [-1, 0, 0, 0, 1, 1, 1, 2, 2, 3, 4, 4, 5, 7, 10, 14],
    "chain5": [-1, 0, 1, 2, 3],
    "star7": [-1, 0, 0, 0, 0, 0, 0],
}


def tree_inputs(w: Workload | str, parent, seed: int = DEFAULT_SEED, nb: int | None = None):
    """Inputs of a candidate-tree verification with the shapes and value
    distributions of workload `w` (dense drafts): logits [B, N, V] and the
    draft rows q [B, N, V] come from the workload's generator with K = N - 1
    (row i of q: the draft distribution at node i; the last node is always a
    leaf and its row is zero), each node's token is drawn from its parent's
    q row (siblings i.i.d.), uniforms [B, N].  Returns
    (logits, q, parent [B, N], tokens [B, N], u [B, N], T)."""
    if isinstance(w, str):
        w = WORKLOADS[w]
    parent = np.asarray(parent, np.int32)
    N = len(parent)
    inp = generate(w.with_(K=N - 1), seed=seed, nb=nb)
    B, V = inp.logits.shape[0], w.V
    q = np.concatenate([inp.q, np.zeros((B, 1, V), np.float32)], 1)
    rng = np.random.default_rng([seed, N, V, 7])
    tokens = np.zeros((B, N), np.int32)
    for v in sorted(set(parent[1:].tolist())):
        kids = np.nonzero(parent == v)[0]
        cdf = np.cumsum(q[:, v].astype(np.float64), -1)
        t = rng.random((B, len(kids))) * cdf[:, -1:]
        tokens[:, kids] = np.minimum(np.array([np.searchsorted(cdf[b], t[b], side="right") for b in range(B)]),
                                     V - 1)
    return inp.logits, q, np.tile(parent, (B, 1)), tokens, inp.u, w.T
