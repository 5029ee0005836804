"""The C ABI without a GPU: the library loads, exports every function the
header declares, and rejects bad arguments on the host before any launch."""
import ctypes
import os
import re

import pytest

import speculative_decoding_sampling_gb300 as sv
from speculative_decoding_sampling_gb300 import _native as N

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    names = []
    inc = os.path.join(ROOT, "include")
    for f in sorted(os.listdir(inc)):
        if f.endswith(".h"):
            text = open(os.path.join(inc, f), encoding="utf-8").read()
            text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
            names += re.findall(r"^\s*(?:const\s+)?[a-z_][a-z0-9_]*\s*\**\s*([a-z_][a-z0-9_]*)\s*\(",
                                text, flags=re.M)
    return names


def test_library_exports_every_declared_function():
    lib = N.lib()
    names = declared_functions()
    assert "spec_verify" in names and "sv_workspace_bytes" in names
    for name in names:
        assert hasattr(lib, name), name
    # the binding's list covers the header's original entry points
    for name in N.EXPORTS:
        assert name in names


def test_status_strings():
    for code in (N.SV_OK, N.SV_EINVAL, N.SV_ECUDA, N.SV_EUNSUPPORTED):
        assert sv.sv_status_string(code).startswith("SV_")
    assert "unknown" in sv.sv_status_string(99)


def test_workspace_size_is_a_function_of_shape():
    a = sv.sv_workspace_bytes(256, 8, 151936)
    assert a > 0 and a % 256 == 0
    assert a == sv.sv_workspace_bytes(256, 8, 151936)
    assert sv.sv_workspace_bytes(0, 4, 100) >= 0
    assert sv.sv_workspace_bytes(-1, 4, 100) == 0
    assert sv.sv_workspace_bytes(1, 4, 0) == 0
    assert sv.sv_workspace_bytes(1, 4, N.SV_MAX_V + 1) == 0


def _call(**kw):
    """spec_verify with plausible (fake, never dereferenced) device pointers."""
    fake = 1 << 40
    args = dict(logits=fake, dtype=N.SV_BF16, q=fake, tok=fake, u=fake, T=1.0, B=4, K=3,
                V=1000, out=fake, n=fake, flags=None, prob=None, mass=None, status=None,
                ws=fake, ws_bytes=1 << 20, stream=None)
    args.update(kw)
    return N.lib().spec_verify(args["logits"], args["dtype"], args["q"], args["tok"],
                               args["u"], ctypes.c_float(args["T"]), args["B"], args["K"],
                               args["V"], args["out"], args["n"], args["flags"],
                               args["prob"], args["mass"], args["status"], args["ws"],
                               args["ws_bytes"], args["stream"])


@pytest.mark.parametrize("kw", [
    dict(logits=None), dict(u=None), dict(out=None), dict(n=None), dict(ws=None),
    dict(tok=None), dict(T=0.0), dict(T=-1.0), dict(T=float("nan")), dict(T=float("inf")),
    dict(T=1e-45), dict(B=-1), dict(K=-1), dict(V=0), dict(dtype=7),
    dict(logits=(1 << 40) + 1), dict(ws=(1 << 40) + 16), dict(u=(1 << 40) + 2),
    dict(ws_bytes=16),
], ids=lambda d: ",".join(f"{k}" for k in d))
def test_host_checks_reject_without_launching(kw):
    # every case returns before any CUDA call, so no GPU is needed
    assert _call(**kw) == N.SV_EINVAL


def test_unsupported_sizes():
    assert _call(V=N.SV_MAX_V + 1) == N.SV_EUNSUPPORTED


def test_empty_batch_is_a_noop():
    assert _call(B=0, ws_bytes=0) == N.SV_OK


def _launches(dtype=N.SV_BF16, dense=1, B=4, K=3, V=1000, out=True):
    n = ctypes.c_int32(-7)
    rc = N.lib().sv_kernel_launches(dtype, dense, B, K, V, ctypes.byref(n) if out else None)
    return rc, n.value


@pytest.mark.parametrize("kw", [dict(out=False), dict(B=-1), dict(K=-1), dict(V=0), dict(dtype=7)],
                         ids=lambda d: ",".join(d))
def test_kernel_launches_host_checks(kw):
    # rejected before the device is queried
    assert _launches(**kw)[0] == N.SV_EINVAL


def test_kernel_launches_sizes_and_empty_batch():
    assert _launches(V=N.SV_MAX_V + 1)[0] == N.SV_EUNSUPPORTED
    assert _launches(B=0) == (N.SV_OK, 0)


def _filter(**kw):
    fake = 1 << 40
    a = dict(logits=fake, dtype=N.SV_BF16, rows=4, V=1000, T=1.0, k=0, p=0.9, out=fake, kept=None,
             status=None, stream=None)
    a.update(kw)
    return N.lib().sv_filter_logits(a["logits"], a["dtype"], a["rows"], a["V"], ctypes.c_float(a["T"]),
                                    a["k"], ctypes.c_float(a["p"]), a["out"], a["kept"], a["status"],
                                    a["stream"])


@pytest.mark.parametrize("kw", [
    dict(logits=None), dict(out=None), dict(rows=-1), dict(V=0), dict(dtype=5), dict(T=0.0),
    dict(T=float("nan")), dict(T=float("inf")), dict(p=0.0), dict(p=-0.5), dict(p=float("nan")),
    dict(logits=(1 << 40) + 1), dict(out=(1 << 40) + 1), dict(kept=(1 << 40) + 2),
], ids=lambda d: ",".join(d))
def test_filter_host_checks(kw):
    # rejected before any CUDA call
    assert _filter(**kw) == N.SV_EINVAL


def test_filter_sizes_and_empty():
    assert _filter(V=N.SV_MAX_V + 1) == N.SV_EUNSUPPORTED
    assert _filter(rows=0) == N.SV_OK
    assert _filter(rows=0, logits=None, out=None) == N.SV_OK


def test_filter_binding_rejects_bad_tensors():
    # checked in Python before the library is called: no GPU needed
    import torch
    x = torch.zeros(2, 8)                       # not a CUDA tensor
    with pytest.raises(ValueError):
        sv.sv_filter_logits(x, 1.0, 0, 0.9)
    with pytest.raises(sv.SpecVerifyError):
        sv.sv_filter_logits(torch.zeros(2, 8, dtype=torch.float16), 1.0, 0, 0.9)


# ----------------------------------------------------------------- LM head

def _lm_logits(**kw):
    fake = 1 << 40
    a = dict(h=fake, W=fake, M=256, d=4096, V=1000, out=fake, status=None, stream=None)
    a.update(kw)
    return N.lib().sv_lm_head_logits(a["h"], a["W"], a["M"], a["d"], a["V"], a["out"], a["status"], a["stream"])


@pytest.mark.parametrize("kw", [
    dict(h=None), dict(W=None), dict(out=None), dict(M=-1), dict(d=0), dict(d=12), dict(d=4),
    dict(V=0), dict(h=(1 << 40) + 8), dict(W=(1 << 40) + 2), dict(out=(1 << 40) + 1),
    dict(status=(1 << 40) + 2),
], ids=lambda d: ",".join(f"{k}={v}" for k, v in d.items()))
def test_lm_head_host_checks(kw):
    assert _lm_logits(**kw) == N.SV_EINVAL


def test_lm_head_sizes():
    assert _lm_logits(V=N.SV_MAX_V + 1) == N.SV_EUNSUPPORTED
    assert _lm_logits(M=(1 << 30) + 1) == N.SV_EUNSUPPORTED
    assert _lm_logits(M=0) == N.SV_OK  # nothing to do, nothing launched
    ws = sv.sv_lm_head_workspace_bytes(256, 8, 151936)
    # the verification's workspace plus one (max, normaliser) pair per row and 256-id tile
    assert ws >= sv.sv_workspace_bytes(256, 8, 151936) + 256 * 9 * 594 * 8
    assert sv.sv_lm_head_workspace_bytes(-1, 8, 100) == 0


def _lm_verify(**kw):
    fake = 1 << 40
    a = dict(h=fake, W=fake, d=256, q=fake, tok=fake, u=fake, T=1.0, B=4, K=3, V=1000, logits=fake,
             out=fake, n=fake, flags=None, prob=None, mass=None, status=None, ws=fake, ws_bytes=1 << 24,
             stream=None)
    a.update(kw)
    return N.lib().spec_verify_lm_head(a["h"], a["W"], a["d"], a["q"], a["tok"], a["u"], ctypes.c_float(a["T"]),
                                       a["B"], a["K"], a["V"], a["logits"], a["out"], a["n"], a["flags"],
                                       a["prob"], a["mass"], a["status"], a["ws"], a["ws_bytes"], a["stream"])


@pytest.mark.parametrize("kw", [
    dict(h=None), dict(W=None), dict(logits=None), dict(u=None), dict(out=None), dict(tok=None),
    dict(d=10), dict(B=-1), dict(K=-1), dict(T=0.0), dict(T=float("nan")), dict(ws_bytes=64),
    dict(ws=None), dict(h=(1 << 40) + 4), dict(logits=(1 << 40) + 1),
], ids=lambda d: ",".join(f"{k}={v}" for k, v in d.items()))
def test_lm_head_verify_host_checks(kw):
    # every case returns before the GEMM is launched
    assert _lm_verify(**kw) == N.SV_EINVAL


def test_lm_head_verify_empty_batch():
    assert _lm_verify(B=0) == N.SV_OK


# ----------------------------------------------------------------- trees

def _tree(**kw):
    fake = 1 << 40
    a = dict(logits=fake, dtype=N.SV_BF16, q=fake, parent=fake, tok=fake, u=fake, T=1.0, B=4, N=16, V=1000,
             out=fake, nodes=None, n=fake, prob=None, status=None, ws=fake, ws_bytes=1 << 24, stream=None)
    a.update(kw)
    return N.lib().spec_verify_tree(a["logits"], a["dtype"], a["q"], a["parent"], a["tok"], a["u"],
                                    ctypes.c_float(a["T"]), a["B"], a["N"], a["V"], a["out"], a["nodes"], a["n"],
                                    a["prob"], a["status"], a["ws"], a["ws_bytes"], a["stream"])


@pytest.mark.parametrize("kw", [
    dict(logits=None), dict(q=None), dict(parent=None), dict(tok=None), dict(u=None), dict(out=None),
    dict(n=None), dict(ws=None), dict(N=0), dict(B=-1), dict(V=0), dict(T=0.0), dict(T=float("nan")),
    dict(dtype=5), dict(logits=(1 << 40) + 1), dict(parent=(1 << 40) + 2), dict(ws=(1 << 40) + 8),
    dict(nodes=(1 << 40) + 1), dict(ws_bytes=100),
], ids=lambda d: ",".join(f"{k}={v}" for k, v in d.items()))
def test_tree_host_checks(kw):
    assert _tree(**kw) == N.SV_EINVAL


def test_tree_sizes():
    assert _tree(N=N.SV_MAX_TREE_NODES + 1) == N.SV_EUNSUPPORTED
    assert _tree(V=N.SV_MAX_V + 1) == N.SV_EUNSUPPORTED
    assert _tree(B=0) == N.SV_OK
    assert sv.sv_tree_workspace_bytes(64, 16, 128256) == sv.sv_workspace_bytes(64, 15, 128256)
    assert sv.sv_tree_workspace_bytes(4, 0, 100) == 0
    assert sv.sv_tree_workspace_bytes(4, N.SV_MAX_TREE_NODES + 1, 100) == 0
