"""spec_verify_noalloc: the allocation-free entry point, for callers that
cannot allocate device memory (a server whose memory is reserved up front by
its own pool, a plugin interface that hands out only input and output
buffers).  Called through the C ABI and compared with the fp64 oracle and
with spec_verify, the entry point that takes a caller workspace, on calls
made back to back and on a run of different shapes sharing the one static
scratch array.

This file is collected last on purpose, so that a run stopping at its first
failure has already run every other test."""
import ctypes

import numpy as np
import pytest
import torch

import synth
from oracle import parity
import speculative_decoding_sampling_gb300 as sv
from speculative_decoding_sampling_gb300 import _native as N

import gpu_util as G

pytestmark = pytest.mark.gpu

TOL = 1e-5  # the probability tolerance of the parity tests


def _entry():
    fn = N.lib().spec_verify_noalloc
    fn.restype = ctypes.c_int
    fn.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p,
                   ctypes.c_void_p, ctypes.c_float, ctypes.c_int64, ctypes.c_int32,
                   ctypes.c_int32] + [ctypes.c_void_p] * 7
    return fn


def _outputs(B, K, dev):
    """Output buffers filled with a value no call writes."""
    return {"out_tokens": torch.full((B, K + 1), -7, dtype=torch.int32, device=dev),
            "num_emitted": torch.full((B,), -7, dtype=torch.int32, device=dev),
            "accept_flags": torch.full((B, K), -7, dtype=torch.int8, device=dev),
            "accept_prob": torch.full((B, K), -7.0, dtype=torch.float32, device=dev),
            "residual_mass": torch.full((B,), -7.0, dtype=torch.float32, device=dev),
            "status": torch.zeros(1, dtype=torch.int32, device=dev)}


def _launch_noalloc(logits, q, tok, u, T, out):
    """One allocation-free call into preallocated outputs (no sync)."""
    B, K1, V = logits.shape
    dt = N.SV_BF16 if logits.dtype == torch.bfloat16 else N.SV_FP32
    rc = _entry()(logits.data_ptr(), dt, None if q is None else q.data_ptr(), tok.data_ptr(),
                  u.data_ptr(), float(T), B, K1 - 1, V, out["out_tokens"].data_ptr(),
                  out["num_emitted"].data_ptr(), out["accept_flags"].data_ptr(),
                  out["accept_prob"].data_ptr(), out["residual_mass"].data_ptr(),
                  out["status"].data_ptr(), torch.cuda.current_stream(logits.device).cuda_stream)
    assert rc == N.SV_OK, sv.sv_status_string(rc)


def _host(out):
    res = {k: v.cpu().numpy() for k, v in out.items() if k != "status"}
    res["status"] = int(out["status"].item())
    return res


def _call_noalloc(logits, q, tok, u, T):
    B, K1, V = logits.shape
    out = _outputs(B, K1 - 1, logits.device)
    _launch_noalloc(logits, q, tok, u, T, out)
    torch.cuda.synchronize()
    return _host(out)


def _oracle_ok(orc, inp, cand):
    rep = parity.compare(orc, inp.logits, inp.q, inp.tokens, inp.u, inp.T, cand)
    assert rep.ok(), rep.summary()


def _same(a, b):
    for k in ("out_tokens", "num_emitted", "accept_flags"):
        assert np.array_equal(a[k], b[k]), k
    for k in ("accept_prob", "residual_mass"):
        assert np.max(np.abs(a[k].astype(np.float64) - b[k])) <= TOL, k
    assert a["status"] == b["status"]


@pytest.mark.parametrize("name,nb", [("b256_k8_v151936_bf16", 256),
                                     ("b128_k8_v128256_bf16_onehot", 64),
                                     ("b1_k4_v32000_fp32", 1)])
def test_noalloc_matches_spec_verify_on_consecutive_calls(orc, name, nb):
    inp = synth.generate(name, nb=nb)
    d = G.to_device(inp)
    ref = G.run(*d, inp.T)               # spec_verify with a caller workspace
    first = _call_noalloc(*d, inp.T)     # two allocation-free calls in a row
    second = _call_noalloc(*d, inp.T)
    _oracle_ok(orc, inp, first)          # against the fp64 oracle
    _oracle_ok(orc, inp, second)
    _same(first, ref)
    _same(second, ref)


def test_noalloc_shapes_in_sequence_allocate_nothing(orc):
    """A run of different shapes on the one static scratch array -- a dense
    batch, a single fp32 sequence, a one-hot batch, then the first again --
    each checked against the oracle; after a first call has warmed the
    library up, the calls change neither PyTorch's allocated bytes nor the
    device's free memory."""
    runs = [("b256_k8_v151936_bf16", 256), ("b1_k4_v32000_fp32", 1),
            ("b128_k8_v128256_bf16_onehot", 128), ("b256_k8_v151936_bf16", 256)]
    cases = []
    for name, nb in runs:
        inp = synth.generate(name, nb=nb)
        d = G.to_device(inp)
        cases.append((inp, d, _outputs(*inp.tokens.shape, d[0].device)))
    inp0, d0, o0 = cases[0]
    _launch_noalloc(*d0, inp0.T, o0)      # warm-up: loads the device code
    torch.cuda.synchronize()
    alloc0 = torch.cuda.memory_allocated()
    free0, _ = torch.cuda.mem_get_info()
    for inp, d, o in cases:
        _launch_noalloc(*d, inp.T, o)
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert torch.cuda.memory_allocated() == alloc0
    assert free1 == free0
    for inp, d, o in cases:
        cand = _host(o)
        assert cand["status"] == 0
        _oracle_ok(orc, inp, cand)


def test_noalloc_rejects_batches_beyond_its_scratch():
    B, K, V = 100000, 8, 1000
    assert sv.sv_workspace_bytes(B, K, V) > (4 << 20)   # SV_NOALLOC_SCRATCH_BYTES
    fake = 1 << 40
    rc = _entry()(fake, N.SV_BF16, None, fake, fake, 1.0, B, K, V, fake, fake, None, None,
                  None, None, None)
    assert rc == N.SV_EUNSUPPORTED
