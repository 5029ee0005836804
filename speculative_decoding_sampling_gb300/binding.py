"""PyTorch binding of the C ABI: argument marshalling only.

Every step of the verification runs in the CUDA kernels of
libspecverify.so; this module checks shapes and dtypes, allocates outputs
and the workspace through PyTorch, and passes raw device pointers and the
current CUDA stream.  The function names are those of the C ABI.
"""
from __future__ import annotations

import threading
from dataclasses import dataclass

import torch

from . import _native as N


class SpecVerifyError(RuntimeError):
    def __init__(self, code: int):
        self.code = code
        super().__init__(sv_status_string(code))


def sv_status_string(code: int) -> str:
    return N.lib().sv_status_string(int(code)).decode()


def sv_workspace_bytes(B: int, K: int, V: int) -> int:
    return int(N.lib().sv_workspace_bytes(int(B), int(K), int(V)))


def sv_kernel_launches(logits_dtype: torch.dtype, dense: bool, B: int, K: int, V: int) -> int:
    """Kernels one spec_verify call with these arguments launches on the
    current device (2 or 3; 0 for B == 0)."""
    import ctypes
    dt = N.SV_BF16 if logits_dtype == torch.bfloat16 else N.SV_FP32
    if logits_dtype not in (torch.bfloat16, torch.float32):
        raise SpecVerifyError(N.SV_EINVAL)
    n = ctypes.c_int32(-1)
    rc = N.lib().sv_kernel_launches(dt, 1 if dense else 0, int(B), int(K), int(V), ctypes.byref(n))
    if rc != N.SV_OK:
        raise SpecVerifyError(rc)
    return int(n.value)


def sv_filter_logits(logits: torch.Tensor, temperature: float, top_k: int = 0, top_p: float = 1.0, *,
                     out: torch.Tensor | None = None, kept: torch.Tensor | None = None,
                     status: torch.Tensor | None = None) -> tuple[torch.Tensor, torch.Tensor]:
    """Top-k / top-p filtering of logit rows (last axis = V) at `temperature`:
    every id outside the kept set becomes -inf.  `out` may be `logits`
    itself (in place).  Returns (filtered logits, kept ids per row)."""
    if logits.dtype not in (torch.bfloat16, torch.float32):
        raise SpecVerifyError(N.SV_EINVAL)
    if not logits.is_cuda or not logits.is_contiguous() or logits.dim() < 1:
        raise ValueError("logits must be a contiguous CUDA tensor")
    V = logits.shape[-1]
    rows = logits.numel() // V if V else 0
    if out is None:
        out = torch.empty_like(logits)
    if out.shape != logits.shape or out.dtype != logits.dtype or not out.is_contiguous() \
            or out.device != logits.device:
        raise ValueError("out must match logits")
    if kept is None:
        kept = torch.empty(logits.shape[:-1], dtype=torch.int32, device=logits.device)
    if kept.numel() != rows or kept.dtype != torch.int32 or not kept.is_contiguous() \
            or kept.device != logits.device:
        raise ValueError("kept must be a contiguous int32 tensor with one entry per row on the logits' device")
    if status is not None:
        _check(status, "status", torch.int32, (1,), logits.device)
    dt = N.SV_BF16 if logits.dtype == torch.bfloat16 else N.SV_FP32
    stream = torch.cuda.current_stream(logits.device).cuda_stream
    rc = N.lib().sv_filter_logits(logits.data_ptr(), dt, rows, V, float(temperature), int(top_k),
                                  float(top_p), out.data_ptr(), kept.data_ptr(),
                                  None if status is None else status.data_ptr(), stream)
    if rc != N.SV_OK:
        raise SpecVerifyError(rc)
    return out, kept


_ws_lock = threading.Lock()
_ws_cache: dict[int, torch.Tensor] = {}


def default_workspace(device: torch.device, nbytes: int) -> torch.Tensor:
    """A zero-filled workspace of at least `nbytes` on `device`, shared by the
    calls that do not pass their own.  The kernels leave it zero-filled, so
    calls ordered on one stream may reuse it; calls that may overlap (other
    streams) must pass distinct workspaces."""
    idx = device.index if device.index is not None else torch.cuda.current_device()
    with _ws_lock:
        ws = _ws_cache.get(idx)
        if ws is None or ws.numel() < nbytes:
            ws = torch.zeros(max(nbytes, 256), dtype=torch.uint8, device=f"cuda:{idx}")
            _ws_cache[idx] = ws
        return ws


@dataclass
class SpecVerifyResult:
    out_tokens: torch.Tensor            # int32 [B, K+1], -1 padded
    num_emitted: torch.Tensor           # int32 [B]
    accept_flags: torch.Tensor          # int8  [B, K]
    accept_prob: torch.Tensor | None    # fp32  [B, K]
    residual_mass: torch.Tensor | None  # fp32  [B]
    status: torch.Tensor | None         # int32 [1], OR of SV_BAD_* bits


def _ptr(t: torch.Tensor | None) -> int | None:
    return None if t is None else t.data_ptr()


def _check(t: torch.Tensor, name: str, dtype, shape, device, host_ok: bool = False):
    if t.dtype != dtype:
        raise TypeError(f"{name}: expected {dtype}, got {t.dtype}")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name}: expected shape {tuple(shape)}, got {tuple(t.shape)}")
    if t.device != device and not (host_ok and _pinned(t)):
        raise ValueError(f"{name}: expected device {device}" + (" or page-locked host memory" if host_ok else "")
                         + f", got {t.device}")
    if not t.is_contiguous():
        raise ValueError(f"{name}: must be contiguous")


def _exec_device(target_logits: torch.Tensor) -> torch.device:
    """The GPU a call runs on: the logits' own, or the current one for
    page-locked host logits."""
    if target_logits.is_cuda:
        return target_logits.device
    if _pinned(target_logits):
        return torch.device("cuda", torch.cuda.current_device())
    raise ValueError("target_logits must be a CUDA tensor or page-locked host memory")


def _pinned(t: torch.Tensor) -> bool:
    """A page-locked CPU tensor: mapped into every device's address space, so
    the kernels read it in place (only the bytes they touch cross the link)."""
    return t.device.type == "cpu" and t.is_pinned()


def _call(fn_name: str, target_logits, draft_probs, draft_tokens, uniforms,
          temperature, out_tokens, num_emitted, accept_flags, accept_prob,
          residual_mass, status, workspace, stream, stats=None):
    dev = _exec_device(target_logits)
    if target_logits.dim() != 3:
        raise ValueError("target_logits must be [B, K+1, V]")
    B, K1, V = target_logits.shape
    K = K1 - 1
    if K < 0:
        raise ValueError("target_logits needs K+1 >= 1 rows per sequence")
    if target_logits.dtype == torch.bfloat16:
        dt = N.SV_BF16
    elif target_logits.dtype == torch.float32:
        dt = N.SV_FP32
    else:
        raise TypeError("target_logits must be bfloat16 or float32")
    if not target_logits.is_contiguous():
        raise ValueError("target_logits must be contiguous")
    if draft_probs is not None:
        _check(draft_probs, "draft_probs", torch.float32, (B, K, V), dev, host_ok=True)
    if draft_tokens is None:
        if K > 0:
            raise ValueError("draft_tokens required when K > 0")
    else:
        _check(draft_tokens, "draft_tokens", torch.int32, (B, K), dev, host_ok=True)
    _check(uniforms, "uniforms", torch.float32, (B, K + 1), dev, host_ok=True)
    for name, t, dtype, shape in (("out_tokens", out_tokens, torch.int32, (B, K + 1)),
                                  ("num_emitted", num_emitted, torch.int32, (B,)),
                                  ("accept_flags", accept_flags, torch.int8, (B, K)),
                                  ("accept_prob", accept_prob, torch.float32, (B, K)),
                                  ("residual_mass", residual_mass, torch.float32, (B,)),
                                  ("status", status, torch.int32, (1,))):
        if t is not None:
            _check(t, name, dtype, shape, dev)
    need = sv_workspace_bytes(B, K, V)
    if need == 0 and B > 0:
        raise SpecVerifyError(N.SV_EUNSUPPORTED)
    if stream is None:
        stream = torch.cuda.current_stream(dev)
    if workspace is None:
        workspace = default_workspace(dev, need)
        # the shared workspace was allocated on the stream current at the time;
        # when this call runs on another one, the caching allocator must not
        # hand the memory out again (after a larger workspace replaces it)
        # before this call's kernels are done with it
        if stream != torch.cuda.current_stream(dev):
            workspace.record_stream(stream)
    elif workspace.device != dev or workspace.numel() * workspace.element_size() < need:
        raise ValueError(f"workspace must hold {need} bytes on {dev}")
    args = [target_logits.data_ptr(), dt, _ptr(draft_probs), _ptr(draft_tokens),
            uniforms.data_ptr(), float(temperature), B, K, V, _ptr(out_tokens),
            _ptr(num_emitted), _ptr(accept_flags), _ptr(accept_prob),
            _ptr(residual_mass), _ptr(status), workspace.data_ptr(),
            workspace.numel() * workspace.element_size()]
    if stats is not None:
        _check(stats, "stats", torch.int64, (N.stats_words(K),), dev)
        fn_name = "spec_verify_stats"
        args.append(stats.data_ptr())
    rc = getattr(N.lib(), fn_name)(*args, stream.cuda_stream)
    if rc != N.SV_OK:
        raise SpecVerifyError(rc)


def _outputs(target_logits, want_probs, out):
    B, K1, V = target_logits.shape
    K = K1 - 1
    dev = _exec_device(target_logits)
    o = dict(out or {})
    o.setdefault("out_tokens", torch.empty((B, K + 1), dtype=torch.int32, device=dev))
    o.setdefault("num_emitted", torch.empty((B,), dtype=torch.int32, device=dev))
    o.setdefault("accept_flags", torch.empty((B, K), dtype=torch.int8, device=dev))
    if want_probs:
        o.setdefault("accept_prob", torch.empty((B, K), dtype=torch.float32, device=dev))
        o.setdefault("residual_mass", torch.empty((B,), dtype=torch.float32, device=dev))
    o.setdefault("accept_prob", None)
    o.setdefault("residual_mass", None)
    o.setdefault("status", None)
    return o


def spec_verify(target_logits: torch.Tensor, draft_probs: torch.Tensor | None,
                draft_tokens: torch.Tensor | None, uniforms: torch.Tensor,
                temperature: float, *, want_probs: bool = True,
                out: dict | None = None, status: torch.Tensor | None = None,
                workspace: torch.Tensor | None = None,
                stream: torch.cuda.Stream | None = None,
                stats: torch.Tensor | None = None) -> SpecVerifyResult:
    """Verify a batch of drafts against target logits on the GPU.

    target_logits [B, K+1, V] bf16/fp32; draft_probs [B, K, V] fp32 or None
    (one-hot drafts); draft_tokens [B, K] int32; uniforms [B, K+1] fp32 in
    [0, 1) with uniforms[:, K] the final draw; temperature > 0.  The inputs
    may be CUDA tensors or page-locked (pinned) CPU tensors, which the
    kernels read in place: a pinned draft_probs sends only the rows the
    draws use (the rejected ones) and the drafted entries over the link.
    `out` may supply preallocated output tensors by name; `status` an int32
    [1] device tensor that receives SV_BAD_* bits; `stats` an int64
    [SV_STATS_WORDS(K)] device tensor the verdicts add the call's acceptance
    counters to (spec_verify_stats).  Runs asynchronously on `stream`
    (default: the current stream)."""
    o = _outputs(target_logits, want_probs, out)
    if status is not None:
        o["status"] = status
    _call("spec_verify", target_logits, draft_probs, draft_tokens, uniforms,
          temperature, o["out_tokens"], o["num_emitted"], o["accept_flags"],
          o["accept_prob"], o["residual_mass"], o["status"], workspace, stream, stats)
    return SpecVerifyResult(o["out_tokens"], o["num_emitted"], o["accept_flags"],
                            o["accept_prob"], o["residual_mass"], o["status"])


def sv_verify_rows(target_logits, draft_probs, draft_tokens, uniforms,
                   temperature, *, out: dict, workspace: torch.Tensor,
                   stream=None) -> None:
    """First stage of spec_verify (see the C header); `out` as returned in
    the fields of a SpecVerifyResult."""
    _call("sv_verify_rows", target_logits, draft_probs, draft_tokens, uniforms,
          temperature, out["out_tokens"], out["num_emitted"],
          out.get("accept_flags"), out.get("accept_prob"),
          out.get("residual_mass"), out.get("status"), workspace, stream)


def sv_sample_survivors(target_logits, draft_probs, draft_tokens, uniforms,
                        temperature, *, out: dict, workspace: torch.Tensor,
                        stream=None) -> None:
    """Second stage of spec_verify; must follow sv_verify_rows on the same
    stream, workspace and inputs."""
    _call("sv_sample_survivors", target_logits, draft_probs, draft_tokens,
          uniforms, temperature, out["out_tokens"], out["num_emitted"],
          out.get("accept_flags"), out.get("accept_prob"),
          out.get("residual_mass"), out.get("status"), workspace, stream)


# ------------------------------------------------------------- LM head

def sv_lm_head_workspace_bytes(B: int, K: int, V: int) -> int:
    return int(N.lib().sv_lm_head_workspace_bytes(int(B), int(K), int(V)))


def _lm_check(hidden, lm_head):
    if hidden.dtype != torch.bfloat16 or lm_head.dtype != torch.bfloat16:
        raise TypeError("hidden and lm_head must be bfloat16")
    if not (hidden.is_cuda and lm_head.is_cuda and hidden.is_contiguous() and lm_head.is_contiguous()):
        raise ValueError("hidden and lm_head must be contiguous CUDA tensors")
    if hidden.device != lm_head.device or lm_head.dim() != 2 or hidden.shape[-1] != lm_head.shape[1]:
        raise ValueError("lm_head must be [V, d] on the hidden states' device, d their last dimension")


def sv_lm_head_logits(hidden: torch.Tensor, lm_head: torch.Tensor, *, out: torch.Tensor | None = None,
                      status: torch.Tensor | None = None,
                      stream: torch.cuda.Stream | None = None) -> torch.Tensor:
    """logits = hidden @ lm_head.T on the tensor cores, bf16 out: hidden
    [..., d] bf16, lm_head [V, d] bf16 -> [..., V] bf16.  status: optional
    int32 [1] device tensor that receives SV_INTERNAL_TIMEOUT."""
    _lm_check(hidden, lm_head)
    V, d = lm_head.shape
    M = hidden.numel() // d if d else 0
    if out is None:
        out = torch.empty(hidden.shape[:-1] + (V,), dtype=torch.bfloat16, device=hidden.device)
    if out.dtype != torch.bfloat16 or out.numel() != M * V or not out.is_contiguous() or out.device != hidden.device:
        raise ValueError("out must be a contiguous bf16 [..., V] tensor on the hidden states' device")
    if status is not None:
        _check(status, "status", torch.int32, (1,), hidden.device)
    stream = stream or torch.cuda.current_stream(hidden.device)
    rc = N.lib().sv_lm_head_logits(hidden.data_ptr(), lm_head.data_ptr(), M, d, V, out.data_ptr(),
                                   _ptr(status), stream.cuda_stream)
    if rc != N.SV_OK:
        raise SpecVerifyError(rc)
    return out


def spec_verify_lm_head(hidden: torch.Tensor, lm_head: torch.Tensor, draft_probs: torch.Tensor | None,
                        draft_tokens: torch.Tensor, uniforms: torch.Tensor, temperature: float, *,
                        logits_out: torch.Tensor | None = None, want_probs: bool = True,
                        workspace: torch.Tensor | None = None, status: torch.Tensor | None = None,
                        stream: torch.cuda.Stream | None = None):
    """spec_verify on logits computed in the same step by the target's LM
    head: hidden [B, K+1, d] bf16, lm_head [V, d] bf16.  Returns
    (SpecVerifyResult, logits [B, K+1, V] bf16)."""
    _lm_check(hidden, lm_head)
    if hidden.dim() != 3:
        raise ValueError("hidden must be [B, K+1, d]")
    B, K1, d = hidden.shape
    K = K1 - 1
    V = lm_head.shape[0]
    dev = hidden.device
    if logits_out is None:
        logits_out = torch.empty((B, K1, V), dtype=torch.bfloat16, device=dev)
    if logits_out.shape != (B, K1, V) or logits_out.dtype != torch.bfloat16 or not logits_out.is_contiguous():
        raise ValueError("logits_out must be a contiguous bf16 [B, K+1, V] tensor")
    if draft_probs is not None:
        _check(draft_probs, "draft_probs", torch.float32, (B, K, V), dev)
    _check(draft_tokens, "draft_tokens", torch.int32, (B, K), dev)
    _check(uniforms, "uniforms", torch.float32, (B, K + 1), dev)
    need = sv_lm_head_workspace_bytes(B, K, V)
    if need == 0 and B > 0:
        raise SpecVerifyError(N.SV_EUNSUPPORTED)
    stream = stream or torch.cuda.current_stream(dev)
    if workspace is None:
        workspace = default_workspace(dev, need)
        if stream != torch.cuda.current_stream(dev):
            workspace.record_stream(stream)
    elif workspace.device != dev or workspace.numel() * workspace.element_size() < need:
        raise ValueError(f"workspace must hold {need} bytes on {dev}")
    res = SpecVerifyResult(
        out_tokens=torch.empty((B, K1), dtype=torch.int32, device=dev),
        num_emitted=torch.empty((B,), dtype=torch.int32, device=dev),
        accept_flags=torch.empty((B, K), dtype=torch.int8, device=dev),
        accept_prob=torch.empty((B, K), dtype=torch.float32, device=dev) if want_probs else None,
        residual_mass=torch.empty((B,), dtype=torch.float32, device=dev) if want_probs else None,
        status=status)
    if status is not None:
        _check(status, "status", torch.int32, (1,), dev)
    rc = N.lib().spec_verify_lm_head(
        hidden.data_ptr(), lm_head.data_ptr(), d, _ptr(draft_probs), draft_tokens.data_ptr(),
        uniforms.data_ptr(), float(temperature), B, K, V, logits_out.data_ptr(), res.out_tokens.data_ptr(),
        res.num_emitted.data_ptr(), res.accept_flags.data_ptr(), _ptr(res.accept_prob),
        _ptr(res.residual_mass), _ptr(status), workspace.data_ptr(),
        workspace.numel() * workspace.element_size(), stream.cuda_stream)
    if rc != N.SV_OK:
        raise SpecVerifyError(rc)
    return res, logits_out


# ------------------------------------------------------------- trees

@dataclass
class TreeResult:
    out_tokens: torch.Tensor           # [B, N] int32: the accepted path's tokens, the final token, then -1
    out_nodes: torch.Tensor            # [B, N] int32: the accepted path's node ids, then -1
    num_emitted: torch.Tensor          # [B] int32
    accept_prob: torch.Tensor | None   # [B, N] fp32: min(1, r(x)/q(x)) of each tested node, -1 otherwise
    status: torch.Tensor | None = None


def sv_tree_workspace_bytes(B: int, nodes: int, V: int) -> int:
    return int(N.lib().sv_tree_workspace_bytes(int(B), int(nodes), int(V)))


def spec_verify_tree(logits: torch.Tensor, draft_probs: torch.Tensor, parent: torch.Tensor, tokens: torch.Tensor,
                     uniforms: torch.Tensor, temperature: float, *, want_probs: bool = True,
                     workspace: torch.Tensor | None = None, status: torch.Tensor | None = None,
                     stream: torch.cuda.Stream | None = None) -> TreeResult:
    """Verification of a candidate tree (multi-step speculative sampling):
    logits [B, N, V] bf16 / fp32 (row i: the target after node i's path),
    draft_probs [B, N, V] fp32 (row i: the draft distribution of node i's
    children), parent / tokens [B, N] int32, uniforms [B, N] fp32."""
    if logits.dim() != 3:
        raise ValueError("logits must be [B, N, V]")
    B, Nn, V = logits.shape
    dev = logits.device
    dt = N.SV_BF16 if logits.dtype == torch.bfloat16 else (N.SV_FP32 if logits.dtype == torch.float32 else None)
    if dt is None:
        raise TypeError("logits must be bfloat16 or float32")
    _check(logits, "logits", logits.dtype, (B, Nn, V), dev)
    _check(draft_probs, "draft_probs", torch.float32, (B, Nn, V), dev)
    _check(parent, "parent", torch.int32, (B, Nn), dev)
    _check(tokens, "tokens", torch.int32, (B, Nn), dev)
    _check(uniforms, "uniforms", torch.float32, (B, Nn), dev)
    need = sv_tree_workspace_bytes(B, Nn, V)
    if need == 0 and B > 0:
        raise SpecVerifyError(N.SV_EUNSUPPORTED)
    stream = stream or torch.cuda.current_stream(dev)
    if workspace is None:
        workspace = default_workspace(dev, need)
        if stream != torch.cuda.current_stream(dev):
            workspace.record_stream(stream)
    elif workspace.device != dev or workspace.numel() * workspace.element_size() < need:
        raise ValueError(f"workspace must hold {need} bytes on {dev}")
    if status is not None:
        _check(status, "status", torch.int32, (1,), dev)
    res = TreeResult(out_tokens=torch.empty((B, Nn), dtype=torch.int32, device=dev),
                     out_nodes=torch.empty((B, Nn), dtype=torch.int32, device=dev),
                     num_emitted=torch.empty((B,), dtype=torch.int32, device=dev),
                     accept_prob=torch.empty((B, Nn), dtype=torch.float32, device=dev) if want_probs else None,
                     status=status)
    rc = N.lib().spec_verify_tree(
        logits.data_ptr(), dt, draft_probs.data_ptr(), parent.data_ptr(), tokens.data_ptr(), uniforms.data_ptr(),
        float(temperature), B, Nn, V, res.out_tokens.data_ptr(), res.out_nodes.data_ptr(),
        res.num_emitted.data_ptr(), _ptr(res.accept_prob), _ptr(status), workspace.data_ptr(),
        workspace.numel() * workspace.element_size(), stream.cuda_stream)
    if rc != N.SV_OK:
        raise SpecVerifyError(rc)
    return res
