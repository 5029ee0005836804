#!/usr/bin/env python3
"""Benchmark of the speculative-sampling verification step on GB300.

One step = one spec_verify call over a whole batch: the row pass
(rows_kernel), the draw stream (survivor_kernel) and, when the draw stream
does not fill the GPU, the final draws (final_kernel); inputs resident in
HBM.  Prints ONE JSON line on rank 0.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
  python bench.py --impl reference ...   # the fp64 CPU oracle, timed on the host

Multi-GPU (torchrun): every rank verifies its own batch of B sequences (its
shard of a global batch); there is no collective on the data path, so the
scaling is weak; the step time is the max over ranks.
"""
from __future__ import annotations

import argparse
import ctypes
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "verified seqs/s and achieved HBM GB/s (% of GB300 peak) for spec_verify"
DEFAULT_WORKLOAD = "b256_k8_v151936_bf16"
GRAPH_STEPS = 10   # consecutive calls captured per CUDA graph in the timed region
NOMINAL_HBM_GBS = 8000.0
L2_BYTES = 129 * 1024 * 1024


def peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as fh:
            d = json.load(fh)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


# ----------------------------------------------------------- byte accounting

def rejected_rows_now(out: dict, K: int) -> int:
    """Sequences of the last call that rejected a draft (num_emitted <= K)."""
    return int((out["num_emitted"] <= K).sum().item())


def algorithmic_bytes(w, num_emitted: np.ndarray) -> dict:
    """Bytes each kernel must move for this batch (the algorithmic count).

    rows_kernel: every logit once, the q(x) gathers (one 32-byte sector each,
    dense drafts), the logit gathers z(x) (one sector each), the tokens and
    uniforms.  draw kernels (survivor_kernel + final_kernel): the surviving
    logit row once more and, after a rejection with dense q, that q row, plus
    the outputs."""
    B = len(num_emitted)
    K, V = w.K, w.V
    es = 2 if w.dtype == "bf16" else 4
    rows = B * (K + 1) * V * es
    rows += B * K * (4 + 32 + (0 if w.onehot else 32) + 4 + 1)   # tokens, z(x), q(x), a, flag
    rows += B * (K + 1) * 4 * 2 + B * 4                          # u, out_tokens, num_emitted
    rejected = int(np.sum(num_emitted <= K))
    surv = B * V * es + (0 if w.onehot else rejected * V * 4) + B * (4 + 4 + 4)
    return {"rows_kernel": rows, "draw_kernels": surv, "total": rows + surv, "rejected": rejected}


OWN_KERNEL_FILES = ("sv_filter.cuh", "sv_lmhead.cuh", "sv_tree.cuh")  # kernels of their own, hashed apart


def kernel_source_hash(only: str | None = None) -> str:
    """Hash of device code, with // comments, trailing blanks and empty lines
    removed (they do not change a kernel).  Default: the verification
    kernels, i.e. every .cuh file but those of the top-k / top-p filter, the
    LM head and the tree walk (the C ABI's host code in spec_verify.cu is
    left out).  only="sv_lmhead.cuh" (or another of those files): that file
    and the verification kernels it includes."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "speculative_decoding_sampling_gb300", "csrc")
    for f in sorted(os.listdir(csrc)):
        if f.endswith(".cuh") and (f not in OWN_KERNEL_FILES or f == only):
            with open(os.path.join(csrc, f), encoding="utf-8") as fh:
                lines = (line.split("//", 1)[0].rstrip() for line in fh.read().splitlines())
                code = "\n".join(line for line in lines if line)
            h.update(f.encode() + b"\0" + code.encode())
    return h.hexdigest()[:16]


def recorded_traffic(workload: str, kernel: str, only: str | None = None):
    """DRAM bytes per launch of `kernel` from the committed ncu summary
    (profiles/traffic.json), if it was taken on the current kernel source
    (kernel_source_hash(only)); else None."""
    try:
        with open(os.path.join(ROOT, "profiles", "traffic.json")) as fh:
            d = json.load(fh)
        e = d.get(workload)
        if e and e.get("source_hash") == kernel_source_hash(only):
            return e.get("dram_bytes_per_launch", {}).get(kernel)
    except Exception:
        pass
    return None


# ------------------------------------------------------------------- clocks

class ClockSampler:
    """nvidia-smi SM clock / throttle samples while the timed region runs."""
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.t0 = self.t1 = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            time.sleep(0.3)
        except Exception:
            self.proc = None

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.1)
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except Exception:
            self.proc.kill()
            out = ""
        sm, smax, reasons, watts = [], [], set(), []
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax.append(float(f[2]))
                watts.append(float(f[3]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        busy = [s for s in sm] or [None]
        return {"sm_mhz": statistics.median(busy) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "power_w_max": max(watts) if watts else None,
                "samples": len(sm), "reasons": sorted(reasons)}


# ----------------------------------------------------------------- GPU arm

def config_of(w, world: int, filt: bool) -> dict:
    """The `config` object of a bench line: what the workload is.  Both arms
    print it from here, so the same workload gives the same dict."""
    return {"workload": w.name, "B_per_gpu": w.B, "K": w.K, "V": w.V,
            "logits_dtype": w.dtype, "draft": "one-hot ids" if w.onehot else "dense q fp32",
            "temperature": w.T, "top_p": w.top_p or None,
            "top_p_applied": ("on the GPU (sv_filter_logits, raw logits in)" if filt else
                              ("by the input generator (masked logits in)" if w.top_p else None)),
            "parallelism": f"replicas x{world} (shard over sequences)"}


ROTATE_BYTES = 4 * L2_BYTES   # rotating copies: the bytes the steps between two uses of a copy read
FLUSH_BELOW = 16 << 20        # steps reading less than this: L2 flush between eager calls instead


class Rig:
    """Device inputs of one workload (one or several copies), the outputs,
    status, workspace and the public C-ABI call on a given copy."""

    def __init__(self, torch, w, inp, dev, copies: int, logits_override=None):
        import speculative_decoding_sampling_gb300 as sv
        from speculative_decoding_sampling_gb300 import _native as N
        self.torch, self.w, self.dev = torch, w, dev
        self.lib = N.lib()
        self.dt = N.SV_BF16 if w.dtype == "bf16" else N.SV_FP32
        B, K, V = w.B, w.K, w.V
        lg_host = inp.logits if logits_override is None else logits_override
        host_lg = torch.from_numpy(lg_host.view(np.int16) if w.dtype == "bf16" else lg_host)
        self.copies = []
        for _ in range(copies):
            lg = host_lg.to(dev)
            if w.dtype == "bf16":
                lg = lg.view(torch.bfloat16)
            q = None if inp.q is None else torch.from_numpy(inp.q).to(dev)
            self.copies.append((lg, q, torch.from_numpy(inp.tokens).to(dev), torch.from_numpy(inp.u).to(dev)))
        self.out = {"out_tokens": torch.empty((B, K + 1), dtype=torch.int32, device=dev),
                    "num_emitted": torch.empty((B,), dtype=torch.int32, device=dev),
                    "accept_flags": torch.empty((B, K), dtype=torch.int8, device=dev),
                    "accept_prob": torch.empty((B, K), dtype=torch.float32, device=dev),
                    "residual_mass": torch.empty((B,), dtype=torch.float32, device=dev)}
        self.status = torch.zeros(1, dtype=torch.int32, device=dev)
        self.need = sv.sv_workspace_bytes(B, K, V)
        self.ws = torch.zeros(self.need, dtype=torch.uint8, device=dev)
        self.sv = sv

    def args(self, i, stream, logits=None):
        lg, q, tok, u = self.copies[i]
        lg = lg if logits is None else logits
        w, o = self.w, self.out
        return (lg.data_ptr(), self.dt, None if q is None else q.data_ptr(), tok.data_ptr(),
                u.data_ptr(), ctypes.c_float(w.T), w.B, w.K, w.V, o["out_tokens"].data_ptr(),
                o["num_emitted"].data_ptr(), o["accept_flags"].data_ptr(), o["accept_prob"].data_ptr(),
                o["residual_mass"].data_ptr(), self.status.data_ptr(), self.ws.data_ptr(), self.need,
                stream.cuda_stream)

    def call(self, i, stream, logits=None):
        rc = self.lib.spec_verify(*self.args(i, stream, logits))
        if rc:
            raise RuntimeError(self.sv.sv_status_string(rc))

    def host_outputs(self):
        return {k: v.cpu().numpy() for k, v in self.out.items()}


def l2_rule(touched: int, flushed: bool, copies: int) -> str:
    if flushed:
        return (f"L2 flushed before every timed step (a {2 * L2_BYTES >> 20} MiB buffer written outside the "
                f"timed events; eager calls): a step reads {touched / 1e6:.1f} MB")
    if copies > 1:
        return (f"{copies} rotating input copies, step i reads copy i mod {copies}: {copies} x "
                f"{touched / 1e6:.0f} MB between two reads of a copy, over 4x the {L2_BYTES >> 20} MiB L2; "
                "no flush")
    return f"no flush: a step reads {touched / 1e6:.0f} MB, more than twice the {L2_BYTES >> 20} MiB L2"


def time_steps(torch, rig, steps: int, step_fn, flushed: bool, dev):
    """Device ms per step of `step_fn(i, stream)` (i = step number): CUDA
    graphs of whole rotations replayed back to back, or, with the flush,
    eager calls each between its own events."""
    stream = torch.cuda.current_stream(dev)
    n = len(rig.copies)
    if flushed:
        buf = torch.empty(2 * L2_BYTES // 4, dtype=torch.int32, device=dev)
        tev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
        for i, (e0, e1) in enumerate(tev):
            buf.fill_(1)
            e0.record(stream)
            step_fn(i % n, stream)
            e1.record(stream)
        torch.cuda.synchronize(dev)
        return sum(e0.elapsed_time(e1) for e0, e1 in tev) / steps
    per = n if n > 1 else GRAPH_STEPS
    gstream = torch.cuda.Stream(dev)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=gstream):
        for i in range(per):
            step_fn(i % n, gstream)
    rem = steps % per
    graph_r = None
    if rem:
        graph_r = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph_r, stream=gstream):
            for i in range(rem):
                step_fn(i % n, gstream)
    graph.replay()
    torch.cuda.synchronize(dev)
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(gstream):
        t0.record(gstream)
        for _ in range(steps // per):
            graph.replay()
        if graph_r is not None:
            graph_r.replay()
        t1.record(gstream)
    torch.cuda.synchronize(dev)
    return t0.elapsed_time(t1) / steps


def measure_workload(torch, dev, name: str, steps: int, cpu_threads: int) -> dict:
    """One of the five configurations: step time, algorithmic bytes, GB/s,
    roofline fractions, the L2 rule, and parity of the outputs against the
    fp64 oracle on the same inputs."""
    import synth
    import oracle
    from oracle import parity
    w = synth.WORKLOADS[name]
    inp = synth.generate(w)
    rig = Rig(torch, w, inp, dev, 1)
    stream = torch.cuda.current_stream(dev)
    for _ in range(3):
        rig.call(0, stream)
    torch.cuda.synchronize(dev)
    cand = rig.host_outputs()
    nb = algorithmic_bytes(w, cand["num_emitted"])
    touched = nb["total"]
    flushed = touched < FLUSH_BELOW
    copies = 1 if (flushed or touched >= 2 * L2_BYTES) else int(-(-ROTATE_BYTES // touched))
    if copies > 1:
        rig = Rig(torch, w, inp, dev, copies)
    for i in range(3 * len(rig.copies)):
        rig.call(i % len(rig.copies), stream)
    ms = time_steps(torch, rig, steps, rig.call, flushed, dev)
    # the small steps are also timed L2-warm (graph replay, no flush), as a second figure
    warm_ms = time_steps(torch, rig, steps, rig.call, False, dev) if flushed else None
    orc = oracle.load()
    rep = parity.compare(orc, inp.logits, inp.q, inp.tokens, inp.u, inp.T, rig.host_outputs(),
                         oracle_res=orc.verify(inp.logits, inp.q, inp.tokens, inp.u, inp.T, nthreads=cpu_threads))
    peak, _ = peaks()
    gbs = touched / (ms * 1e-3) / 1e9
    return {"step_us": ms * 1e3, "l2_warm_step_us": None if warm_ms is None else warm_ms * 1e3,
            "algorithmic_MB": touched / 1e6, "GB_per_s": gbs,
            "frac_of_measured": gbs / peak, "frac_of_8TBs": gbs / NOMINAL_HBM_GBS,
            "seqs_per_s": w.B / (ms * 1e-3), "launches_per_step": rig.sv.sv_kernel_launches(
                torch.bfloat16 if w.dtype == "bf16" else torch.float32, inp.q is not None, w.B, w.K, w.V),
            "l2": l2_rule(touched, flushed, len(rig.copies)), "steps": steps,
            "status_bits": int(rig.status.item()),
            "parity": {"ok": rep.ok(), "summary": rep.summary()}}


LM_SHAPE = (256, 8, 151936, 4096)  # B, K, V, d: the largest verification shape behind a 4096-wide LM head


def measure_lm_head(torch, dev, steps: int, shape=LM_SHAPE, check: bool = True) -> dict:
    """The LM head on the tensor cores (sv_lm_head_logits) and the whole
    fused step (spec_verify_lm_head: GEMM with the row statistics in its
    epilogue, merge, draws), each timed by CUDA-graph replay back to back.
    W alone is larger than L2.  Beside them, for context: a library GEMM
    (torch.matmul, cuBLAS) on the same operands followed by the unfused
    spec_verify.  Parity: sampled logits against the fp64 oracle."""
    import speculative_decoding_sampling_gb300 as sv
    B, K, V, d = shape
    M = B * (K + 1)
    g = torch.Generator(device=dev)
    g.manual_seed(4096)
    h = torch.randn(M, d, device=dev, generator=g).to(torch.bfloat16)
    W = (torch.randn(V, d, device=dev, generator=g) * d ** -0.5).to(torch.bfloat16)
    q = torch.softmax(torch.randn(B, K, V, device=dev, generator=g) * 3.0, -1)
    tok = torch.randint(0, V, (B, K), device=dev, dtype=torch.int32, generator=g)
    u = torch.rand(B, K + 1, device=dev, generator=g)
    logits = torch.empty(B, K + 1, V, dtype=torch.bfloat16, device=dev)
    ref = torch.empty(M, V, dtype=torch.bfloat16, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    ws = torch.zeros(sv.sv_lm_head_workspace_bytes(B, K, V), dtype=torch.uint8, device=dev)
    ws_v = ws[:sv.sv_workspace_bytes(B, K, V)]
    hid = h.view(B, K + 1, d)
    T = 0.7

    def gemm(s):
        sv.sv_lm_head_logits(h, W, out=logits.view(M, V), status=status, stream=s)

    def fused(s):
        sv.spec_verify_lm_head(hid, W, q, tok, u, T, logits_out=logits, workspace=ws, status=status, stream=s)

    def library(s):
        torch.matmul(h, W.t(), out=ref)
        sv.spec_verify(ref.view(B, K + 1, V), q, tok, u, T, workspace=ws_v, status=status, stream=s)

    def timed(fn, n):
        gs = torch.cuda.Stream(dev)
        with torch.cuda.stream(gs):
            for _ in range(3):
                fn(gs)
        torch.cuda.synchronize(dev)
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=gs):
            for _ in range(GRAPH_STEPS):
                fn(gs)
        graph.replay()
        torch.cuda.synchronize(dev)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        reps = max(1, n // GRAPH_STEPS)
        with torch.cuda.stream(gs):
            e0.record(gs)
            for _ in range(reps):
                graph.replay()
            e1.record(gs)
        torch.cuda.synchronize(dev)
        return e0.elapsed_time(e1) / (reps * GRAPH_STEPS)

    n = max(GRAPH_STEPS, min(steps, 200))
    gemm_ms = timed(gemm, n)
    fused_ms = timed(fused, n)
    lib_ms = timed(library, n)
    torch.cuda.synchronize(dev)
    flops = 2.0 * M * V * d
    with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as fh:
        pk = json.load(fh)
    tf_peak, tf_sus = float(pk["bf16_tflops"]), float(pk.get("bf16_tflops_sustained", pk["bf16_tflops"]))
    achieved = flops / (gemm_ms * 1e-3) / 1e12
    out = {
        "shape": {"B": B, "K": K, "V": V, "d": d, "M": M},
        "kernel": "lm_head_kernel",
        "gemm_us": gemm_ms * 1e3,
        "fused_step_us": fused_ms * 1e3,
        "fused_seqs_per_s": B / (fused_ms * 1e-3),
        "context_cublas_plus_spec_verify_us": lib_ms * 1e3,
        "roofline": {"bound": "tensor", "achieved": achieved, "peak": tf_peak, "unit": "TFLOP/s",
                     "frac": achieved / tf_peak, "frac_of_sustained": achieved / tf_sus,
                     "flops_per_launch": flops, "peak_source": "measured (MEASURED_PEAKS.json bf16_tflops burst)",
                     "algorithmic_dram_bytes": V * d * 2 + M * d * 2 + M * V * 2,
                     "traffic": recorded_traffic(f"lm_head_m{M}_v{V}_d{d}", "lm_head_kernel", "sv_lmhead.cuh")},
        "steps": n,
        "status_bits": int(status.item()),
        "timing": f"CUDA-graph replay of {GRAPH_STEPS} calls back to back; W ({V * d * 2 / 1e9:.2f} GB) alone "
                  "exceeds L2, so no flush",
    }
    if check:
        import oracle
        orc = oracle.load()
        rng = np.random.default_rng(1)
        rows, cols = rng.integers(0, M, 256), rng.integers(0, V, 256)
        gemm(torch.cuda.current_stream(dev))
        torch.cuda.synchronize(dev)
        hb = h.view(torch.int16).cpu().numpy().view(np.uint16)
        Wb = W.view(torch.int16).cpu().numpy().view(np.uint16)
        got = logits.view(M, V).view(torch.int16).cpu().numpy().view(np.uint16)[rows, cols]
        exact = orc.lm_head_entries(hb, Wb, rows, cols)
        gotv = (got.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
        absdot = np.array([np.abs((hb[r].astype(np.uint32) << 16).view(np.float32).astype(np.float64)) @
                           np.abs((Wb[c].astype(np.uint32) << 16).view(np.float32).astype(np.float64))
                           for r, c in zip(rows, cols)])
        bound = 2.0 ** -8 * np.abs(exact) + 2 * d * 2.0 ** -24 * absdot
        out["parity"] = {"sampled_logits": len(rows), "within_bound": int((np.abs(gotv - exact) <= bound).sum()),
                         "bit_equal_to_oracle_rounding": int((got == orc.bf16_round(exact)).sum()),
                         "bound": "2^-8 |exact| + 2 d 2^-24 sum|h W| (fp32 summation, one bf16 rounding)"}
    return out


TREE_WORKLOAD = ("b64_k5_v128256_bf16_topp", "tree16")  # B=64, V=128256 bf16 rows, the 16-node tree


def measure_tree(torch, dev, steps: int, check: bool = True) -> dict:
    """spec_verify_tree on B=64 sequences of a 16-node candidate tree over
    V=128256 (bf16 logits, dense fp32 drafts; the value distributions of the
    B=64, V=128256 configuration without its top-p): step time by CUDA-graph
    replay, algorithmic bytes (every node row once; for every rejection the
    node's p and q rows; a leaf's draw one more pass over its p row), and
    parity of sampled sequences against the fp64 oracle."""
    import synth
    import speculative_decoding_sampling_gb300 as sv
    wname, shape = TREE_WORKLOAD
    w = synth.WORKLOADS[wname].with_(top_p=0.0)
    logits, q, parent, tokens, u, T = synth.tree_inputs(w, synth.TREE_SHAPES[shape], seed=2026)
    B, N, V = logits.shape

    def dev_t(a):
        if a.dtype == np.uint16:
            return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(dev).view(torch.bfloat16)
        return torch.from_numpy(np.ascontiguousarray(a)).to(dev)

    d = [dev_t(a) for a in (logits, q, parent, tokens, u)]
    ws = torch.zeros(sv.sv_tree_workspace_bytes(B, N, V), dtype=torch.uint8, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    res = sv.spec_verify_tree(*d, T, workspace=ws, status=status)
    torch.cuda.synchronize(dev)
    out = {k: getattr(res, k).cpu().numpy() for k in ("out_tokens", "out_nodes", "num_emitted", "accept_prob")}
    tested = (out["accept_prob"] >= 0).sum(1)
    rejected = tested - (out["num_emitted"] - 1)
    # the final draw came from a leaf's p when the walk's last node has no children
    last = np.where(out["num_emitted"] > 1, out["out_nodes"][np.arange(B), np.maximum(out["num_emitted"] - 2, 0)], 0)
    has_child = np.array([(parent[b] == last[b]).any() for b in range(B)])
    nbytes = int(B * N * V * 2 + rejected.sum() * V * (2 + 4) + (~has_child).sum() * V * 2)
    n = max(GRAPH_STEPS, min(steps, 300))
    gs = torch.cuda.Stream(dev)
    with torch.cuda.stream(gs):
        for _ in range(3):
            sv.spec_verify_tree(*d, T, workspace=ws, status=status, stream=gs)
    torch.cuda.synchronize(dev)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=gs):
        for _ in range(GRAPH_STEPS):
            sv.spec_verify_tree(*d, T, workspace=ws, status=status, stream=gs)
    graph.replay()
    torch.cuda.synchronize(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    reps = max(1, n // GRAPH_STEPS)
    with torch.cuda.stream(gs):
        e0.record(gs)
        for _ in range(reps):
            graph.replay()
        e1.record(gs)
    torch.cuda.synchronize(dev)
    ms = e0.elapsed_time(e1) / (reps * GRAPH_STEPS)
    peak, _ = peaks()
    gbs = nbytes / (ms * 1e-3) / 1e9
    r = {"workload": f"{wname} rows without top-p, {shape} (N={N})", "B": B, "N": N, "V": V,
         "step_us": ms * 1e3, "seqs_per_s": B / (ms * 1e-3), "tokens_per_s": float(out["num_emitted"].sum()) /
         (ms * 1e-3), "mean_emitted": float(out["num_emitted"].mean()), "algorithmic_MB": nbytes / 1e6,
         "GB_per_s": gbs, "frac_of_measured": gbs / peak, "launches_per_step": 2, "status_bits": int(status.item()),
         "timing": f"CUDA-graph replay of {GRAPH_STEPS} calls back to back; the logits "
                   f"({B * N * V * 2 / 1e6:.0f} MB) exceed L2"}
    if check:
        import oracle
        from oracle import parity
        rep = parity.compare_tree(oracle.load(), logits, q, parent, tokens, u, T, out, seqs=[0, 21, 42, 63])
        r["parity"] = {"ok": rep.ok(), "summary": rep.summary()}
    return r


def run_gpu(args):
    import torch
    import torch.distributed as dist

    import synth
    import speculative_decoding_sampling_gb300 as sv

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    w = synth.WORKLOADS[args.workload]
    if args.batch:
        w = w.with_(B=args.batch)
    B, K, V = w.B, w.K, w.V

    # this rank's shard of the global batch: sequences [rank*B, (rank+1)*B)
    inp = synth.generate(w, b0=rank * B, nb=B)
    filt = bool(args.filter_top_p)
    raw = None
    if filt:
        # the target's top-p applied on the GPU: raw logits in, the draft's
        # processed q, tokens and uniforms as generated
        if not w.top_p:
            raise SystemExit("--filter-top-p needs a workload with top-p")
        raw = synth.generate(w.with_(top_p=0.0), b0=rank * B, nb=B).logits
    rig = Rig(torch, w, inp, dev, 1, logits_override=raw)
    stream = torch.cuda.current_stream(dev)
    top_p32 = float(np.float32(w.top_p)) if filt else 1.0
    d_filt = torch.empty_like(rig.copies[0][0]) if filt else None
    d_kept = torch.empty(B * (K + 1), dtype=torch.int32, device=dev) if filt else None

    def filter_call(i, s):
        rc = rig.lib.sv_filter_logits(rig.copies[i][0].data_ptr(), rig.dt, B * (K + 1), V, ctypes.c_float(w.T), 0,
                                      ctypes.c_float(top_p32), d_filt.data_ptr(), d_kept.data_ptr(),
                                      rig.status.data_ptr(), s.cuda_stream)
        if rc:
            raise RuntimeError(sv.sv_status_string(rc))

    def step(i, s):
        # one step = the public call: the row pass, the draw stream and, unless
        # the draw stream makes them, the final draws, each chained to the one
        # before by programmatic dependent launch; with --filter-top-p the
        # filter launch comes first
        if filt:
            filter_call(i, s)
            rig.call(i, s, logits=d_filt)
        else:
            rig.call(i, s)

    def barrier():
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize(dev)

    for _ in range(max(args.warmup, 3)):
        step(0, stream)
    barrier()

    # bytes one step reads: every logit, the surviving rows again, the
    # rejected rows' draft probabilities (and the filter's read and write)
    touched = algorithmic_bytes(w, rig.out["num_emitted"].cpu().numpy())["total"]
    if filt:
        touched += 2 * B * (K + 1) * V * (2 if w.dtype == "bf16" else 4)
    flushed = {"auto": touched < FLUSH_BELOW, "on": True, "off": False}[args.l2_flush]
    copies = 1 if (flushed or touched >= 2 * L2_BYTES or args.l2_flush == "off") else int(-(-ROTATE_BYTES // touched))
    if copies > 1:
        rig = Rig(torch, w, inp, dev, copies, logits_override=raw)
        for i in range(3 * copies):
            step(i % copies, stream)
    launches_per_step = sv.sv_kernel_launches(
        torch.bfloat16 if w.dtype == "bf16" else torch.float32, inp.q is not None, B, K, V) + (1 if filt else 0)
    barrier()

    # ---- timed region: exactly K steps of the public call
    clocks = ClockSampler(local)
    clocks.start()
    barrier()
    ms_step = time_steps(torch, rig, args.steps, step, flushed, dev)
    barrier()

    # the same K steps as eager calls from the host (for reference)
    e_start = torch.cuda.Event(enable_timing=True)
    e_end = torch.cuda.Event(enable_timing=True)
    e_start.record(stream)
    for i in range(args.steps):
        step(i % copies, stream)
    e_end.record(stream)
    barrier()
    ms_step_eager = e_start.elapsed_time(e_end) / args.steps

    # ---- per-kernel durations: the stages through their own entry points,
    # events between them (this breaks the launch chaining there, so it is
    # used for per-kernel durations only)
    n_k = max(20, min(args.steps, 500))
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(n_k)]
    fevs = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(n_k)] if filt else None
    for i in range(n_k):
        c = i % copies
        if filt:
            fevs[i][0].record(stream)
            filter_call(c, stream)
            fevs[i][1].record(stream)
        a = rig.args(c, stream, logits=d_filt if filt else None)
        evs[i][0].record(stream)
        rc = rig.lib.sv_verify_rows(*a)
        evs[i][1].record(stream)
        rc |= rig.lib.sv_sample_survivors(*a)
        evs[i][2].record(stream)
        if rc:
            raise RuntimeError(sv.sv_status_string(rc))
    barrier()
    clk = clocks.stop()
    rows_ms = sum(e[0].elapsed_time(e[1]) for e in evs) / n_k
    surv_ms = sum(e[1].elapsed_time(e[2]) for e in evs) / n_k
    filt_ms = sum(e[0].elapsed_time(e[1]) for e in fevs) / n_k if filt else None
    if world > 1:
        t = torch.tensor([ms_step], device=dev)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        ms_step = float(t.item())

    num_emitted = rig.out["num_emitted"].cpu().numpy()
    st = int(rig.status.item())
    tokens_per_step = int(num_emitted.sum())
    nbytes = algorithmic_bytes(w, num_emitted)
    if filt:   # the filter reads every logit once and writes every logit once
        nbytes["filter_kernel"] = 2 * B * (K + 1) * V * (2 if w.dtype == "bf16" else 4)
        nbytes["total"] += nbytes["filter_kernel"]
    peak, peak_kind = peaks()
    rows_gbs = nbytes["rows_kernel"] / (rows_ms * 1e-3) / 1e9
    surv_gbs = nbytes["draw_kernels"] / (surv_ms * 1e-3) / 1e9
    step_gbs = nbytes["total"] / (ms_step * 1e-3) / 1e9

    e2e = None if args.no_e2e else run_e2e(torch, w, inp, rig, raw, filt, top_p32, d_kept, dev, args, world)

    result = None
    if rank == 0:
        seqs = B * world
        cpu = None
        parity_note = None
        out_host = rig.host_outputs()
        if not args.no_cpu_baseline:
            fl = None
            if filt:
                f = d_filt.cpu()
                f = f.view(torch.int16).numpy().view(np.uint16) if w.dtype == "bf16" else f.numpy()
                fl = (f, d_kept.cpu().numpy())
            cpu, parity_note = cpu_baseline_and_check(w, inp, out_host, args.cpu_seconds,
                                                      top_p=top_p32 if filt else None, filtered=fl,
                                                      raw_logits=raw)
        workloads = None
        if args.workloads:
            cores = os.cpu_count() or 1
            workloads = {}
            for name in synth.WORKLOADS:
                workloads[name] = measure_workload(torch, dev, name, min(args.steps, 300), cores)
        lm = measure_lm_head(torch, dev, args.steps) if args.lm_head == "on" else None
        tree = measure_tree(torch, dev, args.steps) if (args.workloads and args.tree == "on") else None
        config = config_of(w, world, filt)
        result = {
            "metric": METRIC,
            "value": seqs / (ms_step * 1e-3),
            "unit": "seqs/s",
            "n_gpus": world,
            "steps": args.steps,
            "warmup": args.warmup,
            "ms_per_step": ms_step,
            "higher_is_better": True,
            "scaling": "weak",
            "vs_baseline": None,
            "dtype": "f32",
            "data": "synthetic (seeded Philox4x32-10 generator; shapes and value "
                    "distributions of the workload; no model weights or datasets)",
            "config": config,
            "l2": l2_rule(touched, flushed, copies),
            "tokens_per_s": tokens_per_step * world / (ms_step * 1e-3),
            "hbm_gbs_step": step_gbs,
            "hbm_frac_step": {"of_measured": step_gbs / peak, "of_8tbs_nominal": step_gbs / NOMINAL_HBM_GBS},
            "ms_per_step_eager": ms_step_eager,
            "timing": (("the public C-ABI call issued from the host, each call between its own CUDA "
                        "events, the L2 flush before each (enqueued while the flush runs)") if flushed else
                       ("CUDA-graph replay of the public C-ABI call, back to back (one graph holds a whole "
                        "rotation of input copies, or %d calls)" % GRAPH_STEPS)) +
                      "; ms_per_step_eager: the same K calls issued back to back from the host",
            "kernels_ms": {"rows_kernel": rows_ms, "survivor_kernel+final_kernel": surv_ms,
                           "source": f"{n_k} staged calls with CUDA events between the row pass and the draws"},
            "kernels_gbs": {"rows_kernel": rows_gbs, "survivor_kernel+final_kernel": surv_gbs},
            "filter": ({"kernel": "filter_kernel", "top_p": top_p32, "top_k": 0, "ms": filt_ms,
                        "algorithmic_bytes": nbytes["filter_kernel"],
                        "achieved": nbytes["filter_kernel"] / (filt_ms * 1e-3) / 1e9, "peak": peak,
                        "unit": "GB/s", "frac": nbytes["filter_kernel"] / (filt_ms * 1e-3) / 1e9 / peak,
                        "kept_mean": float(d_kept.float().mean().item())} if filt else None),
            "algorithmic_bytes": nbytes,
            "roofline": {"bound": "hbm", "kernel": "rows_kernel",
                         "achieved": rows_gbs, "peak": peak, "unit": "GB/s",
                         "frac": rows_gbs / peak, "peak_source": peak_kind,
                         "traffic": recorded_traffic(w.name, "rows_kernel")},
            "e2e": e2e,
            "gpu_launches": launches_per_step * args.steps,
            "gpu_launches_per_step": launches_per_step,
            "clocks": clk,
            "status_bits": st,
            "cpu_baseline": cpu,
            "parity": parity_note,
            "workloads": workloads,
            "lm_head": lm,
            "tree": tree,
        }
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()
    return result


def run_e2e(torch, w, inp, rig, raw, filt, top_p32, d_kept, dev, args, world):
    """The same metric end to end through the Python API from pinned host
    buffers: every step copies its logits, tokens and uniforms host -> device
    and its results device -> host; q stays in page-locked memory and the
    kernels read it in place (only the rejected rows and the drafted entries
    cross the link).  Two device input buffers alternate, so step i+1's
    copy (on a copy stream) overlaps step i's verification and result copy."""
    import speculative_decoding_sampling_gb300 as sv
    B, K = w.B, w.K
    steps = max(3, min(args.steps, 20))
    lg_np = inp.logits if raw is None else raw
    host_lg = torch.from_numpy(lg_np.view(np.int16) if w.dtype == "bf16" else lg_np).pin_memory()
    pin = {"logits": host_lg, "tokens": torch.from_numpy(inp.tokens).pin_memory(),
           "u": torch.from_numpy(inp.u).pin_memory(),
           "q": None if inp.q is None else torch.from_numpy(inp.q).pin_memory()}
    h_out = [{"out_tokens": torch.empty((B, K + 1), dtype=torch.int32).pin_memory(),
              "num_emitted": torch.empty((B,), dtype=torch.int32).pin_memory()} for _ in range(2)]
    h2d = sum(pin[k].numel() * pin[k].element_size() for k in ("logits", "tokens", "u"))
    if pin["q"] is not None:   # q bytes read in place: rejected rows, one sector per drafted entry
        h2d += int((rig.out["num_emitted"] <= K).sum().item()) * w.V * 4 + B * K * 32
    d2h = sum(v.numel() * v.element_size() for v in h_out[0].values())
    bufs = [{"logits": torch.empty_like(host_lg, device=dev), "tokens": torch.empty_like(pin["tokens"], device=dev),
             "u": torch.empty_like(pin["u"], device=dev)} for _ in range(2)]
    outs = [{k: torch.empty_like(v) for k, v in rig.out.items()} for _ in range(2)]
    ws = [rig.ws, torch.zeros_like(rig.ws)]
    comp = torch.cuda.current_stream(dev)
    cps = torch.cuda.Stream(dev)
    copied = [torch.cuda.Event() for _ in range(2)]
    consumed = [torch.cuda.Event() for _ in range(2)]

    def e2e_step(i):
        sl = i % 2
        cps.wait_event(consumed[sl])           # the verification two steps back is done with this buffer
        with torch.cuda.stream(cps):
            for k in ("logits", "tokens", "u"):
                bufs[sl][k].copy_(pin[k], non_blocking=True)
            copied[sl].record(cps)
        comp.wait_event(copied[sl])
        lg = bufs[sl]["logits"].view(torch.bfloat16) if w.dtype == "bf16" else bufs[sl]["logits"]
        if filt:
            sv.sv_filter_logits(lg, w.T, 0, top_p32, out=lg, kept=d_kept, status=rig.status)
        o = outs[sl]
        sv.spec_verify(lg, pin["q"], bufs[sl]["tokens"], bufs[sl]["u"], w.T, workspace=ws[sl],
                       status=rig.status, out=o)
        h_out[sl]["out_tokens"].copy_(o["out_tokens"], non_blocking=True)
        h_out[sl]["num_emitted"].copy_(o["num_emitted"], non_blocking=True)
        consumed[sl].record(comp)

    for i in range(4):   # the host pages read in place get their device mappings on first touch
        e2e_step(i)
    torch.cuda.synchronize(dev)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(comp)
    cps.wait_event(e0)
    for i in range(steps):
        e2e_step(i)
    e1.record(comp)
    torch.cuda.synchronize(dev)
    ms = e0.elapsed_time(e1) / steps
    # the link on its own: the step's logits copied host -> device, pinned
    c0 = torch.cuda.Event(enable_timing=True)
    c1 = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(cps):
        c0.record(cps)
        for _ in range(3):
            bufs[0]["logits"].copy_(pin["logits"], non_blocking=True)
        c1.record(cps)
    torch.cuda.synchronize(dev)
    link_peak = 3 * pin["logits"].numel() * pin["logits"].element_size() / (c0.elapsed_time(c1) * 1e-3) / 1e9
    link = h2d / (ms * 1e-3) / 1e9
    if world > 1:
        import torch.distributed as dist
        t = torch.tensor([ms], device=dev)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        ms = float(t.item())
    return {"value": B * world / (ms * 1e-3), "unit": "seqs/s", "ms_per_step": ms,
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": steps,
            "link_gbs": link, "link_peak_gbs": link_peak, "link_frac": link / link_peak,
            "how": "two alternating device input buffers: step i+1's host->device copy on a copy stream "
                   "overlaps step i's verification and result copy; link_peak_gbs = the same logits "
                   "copied host->device alone"}


def cpu_model() -> str:
    """The host CPU's model name (lscpu, else /proc/cpuinfo), for the CPU-baseline record."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.strip().startswith("Model name:"):
                return line.split(":", 1)[1].strip()
    except Exception:
        pass
    try:
        with open("/proc/cpuinfo") as fh:
            for line in fh:
                if line.lower().startswith(("model name", "cpu part")):
                    return line.split(":", 1)[1].strip()
    except Exception:
        pass
    return "unknown"


def cpu_baseline_and_check(w, inp, out, seconds, top_p=None, filtered=None, raw_logits=None):
    """Time the oracle as it stands on this host's cores over the whole batch
    (repeated until `seconds` elapse) and check the GPU outputs against it.
    With `top_p`, the oracle filters the raw logits first (part of the timed
    step) and the GPU's filtered logits `filtered` are checked too."""
    import oracle
    from oracle import parity
    orc = oracle.load()
    cores = os.cpu_count() or 1
    t0 = time.perf_counter()
    passes = 0
    ref = None
    logits = inp.logits
    raw = inp.logits if raw_logits is None else raw_logits
    while True:
        if top_p is not None:
            logits = orc.filter_logits(raw, inp.T, 0, top_p, nthreads=cores).logits
        ref = orc.verify(logits, inp.q, inp.tokens, inp.u, inp.T, nthreads=cores)
        passes += 1
        if time.perf_counter() - t0 >= seconds:
            break
    el = time.perf_counter() - t0
    # the same, single-threaded, for about half as long
    t1 = time.perf_counter()
    passes1 = 0
    while True:
        lg1 = inp.logits
        if top_p is not None:
            lg1 = orc.filter_logits(raw, inp.T, 0, top_p, nthreads=1).logits
        orc.verify(lg1, inp.q, inp.tokens, inp.u, inp.T, nthreads=1)
        passes1 += 1
        if time.perf_counter() - t1 >= seconds / 2:
            break
    el1 = time.perf_counter() - t1
    cand = {k: (out[k].cpu().numpy() if hasattr(out[k], "cpu") else np.asarray(out[k])) for k in out}
    note = {}
    if top_p is not None:
        frep = parity.compare_filter(orc, raw, inp.T, 0, top_p, filtered[0], filtered[1])
        note["filter"] = {"ok": frep.ok(), "summary": frep.summary()}
        if frep.excused:   # verify what the GPU actually filtered
            logits = filtered[0].reshape(logits.shape)
            ref = None
    rep = parity.compare(orc, logits, inp.q, inp.tokens, inp.u, inp.T, cand, oracle_res=ref)
    cpu = {"value": passes * inp.B / el, "unit": "seqs/s", "cores": cores, "kind": "oracle",
           "cpu_model": cpu_model(),
           "sample": f"all {inp.B} sequences of the workload, {passes} passes, {el:.1f} s wall"
                     + (" (top-p filter included)" if top_p is not None else ""),
           "single_thread": {"value": passes1 * inp.B / el1, "unit": "seqs/s", "cores": 1,
                             "sample": f"all {inp.B} sequences, {passes1} passes, {el1:.1f} s wall"}}
    ok = rep.ok() and all(v["ok"] for v in note.values())
    return cpu, dict(ok=ok, summary=rep.summary(), **note)


# ------------------------------------------------------------ reference arm

def run_reference(args):
    """The fp64 CPU oracle, timed as it stands on the host cores."""
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    if rank != 0:
        return None
    import oracle
    import synth
    w = synth.WORKLOADS[args.workload]
    orc = oracle.load()
    cores = os.cpu_count() or 1
    # calibrate, then size each step's sample so the whole run stays ~60 s
    calib = synth.generate(w, nb=min(w.B, cores))
    t0 = time.perf_counter()
    orc.verify(calib.logits, calib.q, calib.tokens, calib.u, calib.T, nthreads=cores)
    rate = calib.B / max(time.perf_counter() - t0, 1e-6)
    n_steps = args.steps + args.warmup
    per_step = max(1, min(w.B, int(rate * 60.0 / max(n_steps, 1))))
    inp = synth.generate(w, nb=per_step)
    for _ in range(args.warmup):
        orc.verify(inp.logits, inp.q, inp.tokens, inp.u, inp.T, nthreads=cores)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        orc.verify(inp.logits, inp.q, inp.tokens, inp.u, inp.T, nthreads=cores)
    el = time.perf_counter() - t0
    ms = el * 1e3 / args.steps
    value = per_step / (el / args.steps)
    sample = (f"first {per_step} of the {w.B} sequences of the workload per step, "
              f"fp64 oracle, {cores} threads")
    return {
        "impl": "reference",
        "metric": METRIC, "value": value, "unit": "seqs/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f64", "data": "synthetic",
        "config": config_of(w, world, bool(args.filter_top_p)),
        "cpu_baseline": {"value": value, "unit": "seqs/s", "cores": cores, "kind": "oracle",
                         "cpu_model": cpu_model(), "sample": sample},
        "e2e": {"value": value, "unit": "seqs/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=3000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true", help="skip the host-buffer end-to-end timing")
    ap.add_argument("--batch", type=int, default=0, help="override B (profiling runs)")
    ap.add_argument("--filter-top-p", action="store_true",
                    help="top-p workloads: raw logits, the target's top-p applied by sv_filter_logits in the step")
    ap.add_argument("--l2-flush", default="auto", choices=["auto", "on", "off"],
                    help="auto: steps reading under 16 MB flush L2 between eager calls, steps reading under "
                         "2x L2 rotate input copies (4x L2 between two reads of a copy), larger steps neither; "
                         "on: always flush; off: neither")
    ap.add_argument("--no-workloads", dest="workloads", action="store_false",
                    help="skip the per-configuration `workloads` object (all five configs, parity included)")
    ap.add_argument("--lm-head", default="on", choices=["on", "off", "only"],
                    help="the LM-head leg (GEMM and fused step); only: that leg alone (profiling runs)")
    ap.add_argument("--lm-shape", default=",".join(map(str, LM_SHAPE)),
                    help="B,K,V,d of the LM-head leg with --lm-head only (profiling runs)")
    ap.add_argument("--tree", default="on", choices=["on", "off", "only"],
                    help="the tree-verification leg; only: that leg alone, without the oracle check (profiling runs)")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.tree == "only" and args.impl != "reference":
        import torch
        print(json.dumps({"tree": measure_tree(torch, torch.device("cuda", 0), args.steps, check=False)}),
              flush=True)
        return
    if args.lm_head == "only" and args.impl != "reference":
        import torch
        dev = torch.device("cuda", 0)
        shape = tuple(int(x) for x in args.lm_shape.split(","))
        print(json.dumps({"lm_head": measure_lm_head(torch, dev, args.steps, shape, check=False)}), flush=True)
        return
    res = run_reference(args) if args.impl == "reference" else run_gpu(args)
    if res is not None:
        print(json.dumps(res), flush=True)


if __name__ == "__main__":
    main()
