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


def kernel_source_hash() -> str:
    """Hash of the code the verification kernels and their launches are
    built from: every .cu/.cuh file but the top-k / top-p filter's, with
    // comments, trailing blanks and empty lines removed (they do not change
    a kernel)."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "speculative_decoding_sampling_gb300", "csrc")
    for f in sorted(os.listdir(csrc)):
        if f.endswith((".cu", ".cuh")) and f != "sv_filter.cuh":
            with open(os.path.join(csrc, f), encoding="utf-8") as fh:
                lines = (line.split("//", 1)[0].rstrip() for line in fh.read().splitlines())
                code = "\n".join(line for line in lines if line)
            h.update(f.encode() + b"\0" + code.encode())
    return h.hexdigest()[:16]


def recorded_traffic(workload: str, kernel: str):
    """DRAM bytes per launch of `kernel` from the committed ncu summary
    (profiles/traffic.json), if it was taken on the current kernel source;
    else None."""
    try:
        with open(os.path.join(ROOT, "profiles", "traffic.json")) as fh:
            d = json.load(fh)
        e = d.get(workload)
        if e and e.get("source_hash") == kernel_source_hash():
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

def run_gpu(args):
    import torch
    import torch.distributed as dist

    import synth
    import speculative_decoding_sampling_gb300 as sv
    from speculative_decoding_sampling_gb300 import _native as N

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
    if filt:
        # the target's top-p applied on the GPU: raw logits in, the draft's
        # processed q, tokens and uniforms as generated
        if not w.top_p:
            raise SystemExit("--filter-top-p needs a workload with top-p")
        inp.logits = synth.generate(w.with_(top_p=0.0), b0=rank * B, nb=B).logits
    host = {"logits": torch.from_numpy(inp.logits.view(np.int16) if w.dtype == "bf16" else inp.logits),
            "q": None if inp.q is None else torch.from_numpy(inp.q),
            "tokens": torch.from_numpy(inp.tokens), "u": torch.from_numpy(inp.u)}
    d_logits = host["logits"].to(dev)
    if w.dtype == "bf16":
        d_logits = d_logits.view(torch.bfloat16)
    d_q = None if host["q"] is None else host["q"].to(dev)
    d_tok = host["tokens"].to(dev)
    d_u = host["u"].to(dev)
    out = {"out_tokens": torch.empty((B, K + 1), dtype=torch.int32, device=dev),
           "num_emitted": torch.empty((B,), dtype=torch.int32, device=dev),
           "accept_flags": torch.empty((B, K), dtype=torch.int8, device=dev),
           "accept_prob": torch.empty((B, K), dtype=torch.float32, device=dev),
           "residual_mass": torch.empty((B,), dtype=torch.float32, device=dev)}
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    need = sv.sv_workspace_bytes(B, K, V)
    ws = torch.zeros(need, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    lib = N.lib()
    dt = N.SV_BF16 if w.dtype == "bf16" else N.SV_FP32

    def args_for(logits, q, tok, u, o):
        return (logits.data_ptr(), dt, None if q is None else q.data_ptr(), tok.data_ptr(),
                u.data_ptr(), ctypes.c_float(w.T), B, K, V, o["out_tokens"].data_ptr(),
                o["num_emitted"].data_ptr(), o["accept_flags"].data_ptr(),
                o["accept_prob"].data_ptr(), o["residual_mass"].data_ptr(), status.data_ptr(),
                ws.data_ptr(), need, stream.cuda_stream)

    d_filt = torch.empty_like(d_logits) if filt else None
    d_kept = torch.empty(B * (K + 1), dtype=torch.int32, device=dev) if filt else None
    top_p32 = float(np.float32(w.top_p)) if filt else 1.0
    cargs = args_for(d_filt if filt else d_logits, d_q, d_tok, d_u, out)

    def filter_call(s):
        rc = lib.sv_filter_logits(d_logits.data_ptr(), dt, B * (K + 1), V, ctypes.c_float(w.T), 0,
                                  ctypes.c_float(top_p32), d_filt.data_ptr(), d_kept.data_ptr(),
                                  status.data_ptr(), s.cuda_stream)
        if rc:
            raise RuntimeError(sv.sv_status_string(rc))

    def step(s):
        # one call = the launches of the path (row pass, draw stream and,
        # unless the draw stream makes them, the final draws), each chained
        # to the one before by programmatic dependent launch; with
        # --filter-top-p the filter launch comes first
        if filt:
            filter_call(s)
        rc = lib.spec_verify(*cargs[:-1], s.cuda_stream)
        if rc:
            raise RuntimeError(sv.sv_status_string(rc))

    def staged_step(evs, fev=None):
        # the same launches through the per-stage entry points, with events
        # between the row pass and the draws (this breaks the launch chaining
        # there, so it is used for per-kernel durations only)
        if fev is not None:
            fev[0].record(stream)
            filter_call(stream)
            fev[1].record(stream)
        evs[0].record(stream)
        rc = lib.sv_verify_rows(*cargs)
        evs[1].record(stream)
        rc |= lib.sv_sample_survivors(*cargs)
        evs[2].record(stream)
        if rc:
            raise RuntimeError(sv.sv_status_string(rc))

    def barrier():
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize(dev)

    # warm-up
    for _ in range(max(args.warmup, 3)):
        step(stream)
    barrier()

    # bytes one step reads: every logit, the surviving rows again, the
    # rejected rows' draft probabilities.  Below twice the L2 size, the L2 is
    # flushed before every timed step, outside the timed events, so no step
    # finds its inputs cached by the step before.
    touched = algorithmic_bytes(w, out["num_emitted"].cpu().numpy())["total"]
    flush_l2 = {"auto": touched < 2 * L2_BYTES, "on": True, "off": False}[args.l2_flush]
    flush_buf = torch.empty(2 * L2_BYTES // 4, dtype=torch.int32, device=dev) if flush_l2 else None

    def flush(s):
        # write a buffer of twice the L2: no input of the step stays cached
        if flush_buf is not None:
            with torch.cuda.stream(s):
                flush_buf.fill_(1)
    launches_per_step = sv.sv_kernel_launches(
        torch.bfloat16 if w.dtype == "bf16" else torch.float32, d_q is not None, B, K, V) + (1 if filt else 0)

    # the public call captured in CUDA graphs, GRAPH_STEPS consecutive calls
    # (steps) per graph plus a one-call graph for the remainder: the timed
    # region replays them, so host launch overhead and the gap between graph
    # launches stay out of the device timing
    gstream = torch.cuda.Stream(dev)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=gstream):
        for _ in range(GRAPH_STEPS):
            step(gstream)
    graph1 = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph1, stream=gstream):
        step(gstream)
    graph.replay()
    graph1.replay()
    barrier()

    # ---- timed region: exactly K steps of the public call (graph replays;
    # with the L2 flush, eager calls, each between its own events)
    clocks = ClockSampler(local)
    clocks.start()
    barrier()
    if flush_l2:
        tev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(args.steps)]
        # eager calls: the host enqueues each call while the flush before it
        # runs, so the events see the call's device time alone
        for e0, e1 in tev:
            flush(stream)
            e0.record(stream)
            step(stream)
            e1.record(stream)
        barrier()
        ms_step = sum(e0.elapsed_time(e1) for e0, e1 in tev) / args.steps
    else:
        t_start = torch.cuda.Event(enable_timing=True)
        t_end = torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(gstream):
            t_start.record(gstream)
            for _ in range(args.steps // GRAPH_STEPS):
                graph.replay()
            for _ in range(args.steps % GRAPH_STEPS):
                graph1.replay()
            t_end.record(gstream)
        barrier()
        ms_step = t_start.elapsed_time(t_end) / args.steps

    # the same K steps as eager calls from the host (for reference)
    e_start = torch.cuda.Event(enable_timing=True)
    e_end = torch.cuda.Event(enable_timing=True)
    e_start.record(stream)
    for _ in range(args.steps):
        step(stream)
    e_end.record(stream)
    barrier()
    ms_step_eager = e_start.elapsed_time(e_end) / args.steps

    # ---- per-kernel durations: the same launches, events between them
    n_k = max(20, min(args.steps, 500))
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(n_k)]
    fevs = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(n_k)] if filt else None
    for i in range(n_k):
        flush(stream)
        staged_step(evs[i], fevs[i] if filt else None)
    barrier()
    clk = clocks.stop()
    rows_ms = sum(e[0].elapsed_time(e[1]) for e in evs) / n_k
    surv_ms = sum(e[1].elapsed_time(e[2]) for e in evs) / n_k
    filt_ms = sum(e[0].elapsed_time(e[1]) for e in fevs) / n_k if filt else None
    if world > 1:
        t = torch.tensor([ms_step], device=dev)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        ms_step = float(t.item())

    num_emitted = out["num_emitted"].cpu().numpy()
    st = int(status.item())
    tokens_per_step = int(num_emitted.sum())
    nbytes = algorithmic_bytes(w, num_emitted)
    if filt:   # the filter reads every logit once and writes every logit once
        nbytes["filter_kernel"] = 2 * B * (K + 1) * V * (2 if w.dtype == "bf16" else 4)
        nbytes["total"] += nbytes["filter_kernel"]
    peak, peak_kind = peaks()
    rows_gbs = nbytes["rows_kernel"] / (rows_ms * 1e-3) / 1e9
    surv_gbs = nbytes["draw_kernels"] / (surv_ms * 1e-3) / 1e9
    step_gbs = nbytes["total"] / (ms_step * 1e-3) / 1e9

    # ---- end to end through the public call with pinned host buffers: the
    # logits (every one is read), tokens and uniforms are copied to the device
    # each step; the draft probabilities stay in page-locked host memory and
    # the kernels read them in place, so only the rejected rows and the
    # drafted entries cross the host link
    e2e_steps = 0 if args.no_e2e else max(3, min(args.steps, 20))
    pin = {k: (v.pin_memory() if (v is not None and e2e_steps) else v) for k, v in host.items()}
    h_out = {"out_tokens": torch.empty((B, K + 1), dtype=torch.int32).pin_memory(),
             "num_emitted": torch.empty((B,), dtype=torch.int32).pin_memory()}
    h2d = sum(pin[k].numel() * pin[k].element_size() for k in ("logits", "tokens", "u"))
    if pin.get("q") is not None:   # q bytes read in place: rejected rows, one sector per drafted entry
        h2d += rejected_rows_now(out, K) * V * 4 + B * K * 32
    d2h = sum(v.numel() * v.element_size() for v in h_out.values())
    e_logits = torch.empty_like(host["logits"], device=dev) if e2e_steps else None
    e_tok = torch.empty_like(d_tok)
    e_u = torch.empty_like(d_u)

    def e2e_step():
        e_logits.copy_(pin["logits"], non_blocking=True)
        e_tok.copy_(pin["tokens"], non_blocking=True)
        e_u.copy_(pin["u"], non_blocking=True)
        lg = e_logits.view(torch.bfloat16) if w.dtype == "bf16" else e_logits
        if filt:
            sv.sv_filter_logits(lg, w.T, 0, top_p32, out=lg, kept=d_kept, status=status)
        res = sv.spec_verify(lg, pin.get("q"), e_tok, e_u, w.T, out=out, workspace=ws, status=status)
        h_out["out_tokens"].copy_(res.out_tokens, non_blocking=True)
        h_out["num_emitted"].copy_(res.num_emitted, non_blocking=True)

    e2e_ms = float("nan")
    if e2e_steps:
        for _ in range(3):   # the host pages read in place get their device mappings on first touch
            e2e_step()
        barrier()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(e2e_steps):
            e2e_step()
        e1.record(stream)
        barrier()
        e2e_ms = e0.elapsed_time(e1) / e2e_steps
    if world > 1:
        t = torch.tensor([e2e_ms], device=dev)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        e2e_ms = float(t.item())

    result = None
    if rank == 0:
        seqs = B * world
        cpu = None
        parity_note = None
        if not args.no_cpu_baseline:
            fl = None
            if filt:
                f = d_filt.cpu()
                f = f.view(torch.int16).numpy().view(np.uint16) if w.dtype == "bf16" else f.numpy()
                fl = (f, d_kept.cpu().numpy())
            cpu, parity_note = cpu_baseline_and_check(w, inp, out, args.cpu_seconds,
                                                      top_p=top_p32 if filt else None, filtered=fl)
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
            "config": {"workload": w.name, "B_per_gpu": B, "K": K, "V": V,
                       "logits_dtype": w.dtype, "draft": "one-hot ids" if w.onehot else "dense q fp32",
                       "temperature": w.T, "top_p": w.top_p or None,
                       "top_p_applied": ("on the GPU (sv_filter_logits, raw logits in)" if filt else
                                         ("by the input generator (masked logits in)" if w.top_p else None)),
                       "l2": (f"L2 flushed before every timed step (a {2 * L2_BYTES >> 20} MiB buffer written "
                              f"outside the timed events): a step reads {touched / 1e6:.0f} MB, "
                              f"under twice the {L2_BYTES >> 20} MiB L2") if flush_l2 else
                             (f"no flush: a step reads {touched / 1e6:.0f} MB, "
                              + ("more than twice" if touched >= 2 * L2_BYTES else "UNDER twice (flush off by flag)")
                              + f" the {L2_BYTES >> 20} MiB L2"),
                       "parallelism": f"replicas x{world} (shard over sequences)"},
            "tokens_per_s": tokens_per_step * world / (ms_step * 1e-3),
            "hbm_gbs_step": step_gbs,
            "hbm_frac_step": {"of_measured": step_gbs / peak, "of_8tbs_nominal": step_gbs / NOMINAL_HBM_GBS},
            "ms_per_step_eager": ms_step_eager,
            "timing": (("the public C-ABI call issued from the host, each call between its own CUDA "
                        "events, the L2 flush before each (enqueued while the flush runs)") if flush_l2 else
                       (f"CUDA-graph replay of the public C-ABI call ({GRAPH_STEPS} consecutive calls per "
                        "replay, the remainder one call per replay)")) +
                      "; ms_per_step_eager: the same K calls issued back to back from the host, no flush",
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
            "e2e": ({"value": seqs / (e2e_ms * 1e-3), "unit": "seqs/s",
                     "ms_per_step": e2e_ms, "h2d_bytes_per_step": h2d,
                     "d2h_bytes_per_step": d2h, "steps": e2e_steps} if e2e_steps else None),
            "gpu_launches": launches_per_step * args.steps,
            "gpu_launches_per_step": launches_per_step,
            "clocks": clk,
            "status_bits": st,
            "cpu_baseline": cpu,
            "parity": parity_note,
        }
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()
    return result


def cpu_baseline_and_check(w, inp, out, seconds, top_p=None, filtered=None):
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
    while True:
        if top_p is not None:
            logits = orc.filter_logits(inp.logits, inp.T, 0, top_p, nthreads=cores).logits
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
            lg1 = orc.filter_logits(inp.logits, inp.T, 0, top_p, nthreads=1).logits
        orc.verify(lg1, inp.q, inp.tokens, inp.u, inp.T, nthreads=1)
        passes1 += 1
        if time.perf_counter() - t1 >= seconds / 2:
            break
    el1 = time.perf_counter() - t1
    cand = {k: (out[k].cpu().numpy() if hasattr(out[k], "cpu") else np.asarray(out[k])) for k in out}
    note = {}
    if top_p is not None:
        frep = parity.compare_filter(orc, inp.logits, inp.T, 0, top_p, filtered[0], filtered[1])
        note["filter"] = {"ok": frep.ok(), "summary": frep.summary()}
        if frep.excused:   # verify what the GPU actually filtered
            logits = filtered[0].reshape(logits.shape)
            ref = None
    rep = parity.compare(orc, logits, inp.q, inp.tokens, inp.u, inp.T, cand, oracle_res=ref)
    cpu = {"value": passes * inp.B / el, "unit": "seqs/s", "cores": cores, "kind": "oracle",
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
        "config": {"workload": w.name, "B_per_gpu": w.B, "K": w.K, "V": w.V,
                   "logits_dtype": w.dtype, "draft": "one-hot ids" if w.onehot else "dense q fp32"},
        "cpu_baseline": {"value": value, "unit": "seqs/s", "cores": cores, "kind": "oracle",
                         "sample": sample},
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
                    help="flush L2 before every timed step (auto: when a step reads under 2x L2)")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    res = run_reference(args) if args.impl == "reference" else run_gpu(args)
    if res is not None:
        print(json.dumps(res), flush=True)


if __name__ == "__main__":
    main()
