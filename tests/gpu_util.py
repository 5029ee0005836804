"""Helpers for the GPU tests: move generated inputs to the device and run
the C-ABI library through its binding."""
from __future__ import annotations

import numpy as np
import torch

import speculative_decoding_sampling_gb300 as sv


def to_device(inp, dev="cuda:0"):
    """(logits, q, tokens, u) device tensors for generated host inputs."""
    if inp.logits.dtype == np.uint16:
        logits = torch.from_numpy(inp.logits.view(np.int16)).to(dev).view(torch.bfloat16)
    else:
        logits = torch.from_numpy(inp.logits).to(dev)
    q = None if inp.q is None else torch.from_numpy(inp.q).to(dev)
    tok = torch.from_numpy(inp.tokens).to(dev)
    u = torch.from_numpy(inp.u).to(dev)
    return logits, q, tok, u


def host_logits_tensor(logits_np, dev="cuda:0"):
    if logits_np.dtype == np.uint16:
        return torch.from_numpy(logits_np.view(np.int16)).to(dev).view(torch.bfloat16)
    return torch.from_numpy(np.ascontiguousarray(logits_np)).to(dev)


def run(logits, q, tok, u, T, **kw):
    status = torch.zeros(1, dtype=torch.int32, device=logits.device)
    res = sv.spec_verify(logits, q, tok, u, T, status=status, **kw)
    torch.cuda.synchronize()
    cand = {k: getattr(res, k).cpu().numpy() for k in
            ("out_tokens", "num_emitted", "accept_flags", "accept_prob", "residual_mass")}
    cand["status"] = int(status.item())
    return cand


def run_inputs(inp, **kw):
    return run(*to_device(inp), inp.T, **kw)
