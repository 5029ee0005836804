"""Guard regions around every buffer the library writes (GPU).

Each output, the status word, the statistics counters and the workspace sit
between two 4 KiB guards of a known byte pattern; after the call the guards
must be untouched, the inputs unchanged and the workspace back to zero.  The
results themselves are checked against the oracle as in the parity tests.
This stands in for a device memory checker on shapes that end in ragged
groups, chunks and spans."""
import numpy as np
import pytest
import torch

import synth
from oracle import parity

import filter_rows
import gpu_util as G

pytestmark = pytest.mark.gpu

GUARD = 4096
PATTERN = 0xA5


class Guarded:
    """A tensor of `shape`/`dtype` inside a byte buffer with guards."""

    def __init__(self, shape, dtype, fill=None):
        n = int(np.prod(shape)) * torch.tensor([], dtype=dtype).element_size()
        body = (n + 255) // 256 * 256
        self.buf = torch.full((GUARD + body + GUARD,), PATTERN, dtype=torch.uint8, device="cuda:0")
        self.n = n
        if fill is not None:
            self.buf[GUARD:GUARD + n].fill_(fill)
        self.t = self.buf[GUARD:GUARD + n].view(dtype).view(shape)

    def guards_intact(self) -> bool:
        """Every byte outside the tensor (guards and padding) still holds the pattern."""
        b = self.buf.cpu().numpy()
        return bool((b[:GUARD] == PATTERN).all() and (b[GUARD + self.n:] == PATTERN).all())


CASES = [("b8_k4_v32000_bf16", dict(B=5, V=4097)), ("b8_k4_v32000_bf16", dict(B=3, V=1025, K=0)),
         ("b1_k4_v32000_fp32", dict(B=4, V=3001)), ("b128_k8_v128256_bf16_onehot", dict(B=6, V=2049)),
         ("b256_k8_v151936_bf16", dict(B=40, V=151936)), ("b64_k5_v128256_bf16_topp", dict(B=9, V=7777))]


@pytest.mark.parametrize("name,kw", CASES, ids=[f"{n}_{'_'.join(f'{k}{v}' for k, v in kw.items())}"
                                               for n, kw in CASES])
def test_spec_verify_writes_only_its_buffers(orc, name, kw):
    import speculative_decoding_sampling_gb300 as sv
    w = synth.WORKLOADS[name].with_(**kw)
    inp = synth.generate(w, seed=91)
    lg, q, tok, u = G.to_device(inp)
    ins = [t.clone() for t in (lg, tok, u) + ((q,) if q is not None else ())]
    B, K = inp.tokens.shape
    out = {"out_tokens": Guarded((B, K + 1), torch.int32), "num_emitted": Guarded((B,), torch.int32),
           "accept_flags": Guarded((B, K), torch.int8), "accept_prob": Guarded((B, K), torch.float32),
           "residual_mass": Guarded((B,), torch.float32)}
    status = Guarded((1,), torch.int32, fill=0)
    stats = Guarded((4 + K + 1,), torch.int64, fill=0)
    ws = Guarded((sv.sv_workspace_bytes(B, K, w.V),), torch.uint8, fill=0)
    for _ in range(2):   # the second call runs on the workspace the first one left
        res = sv.spec_verify(lg, q, tok, u, inp.T, out={k: g.t for k, g in out.items()},
                             status=status.t, workspace=ws.t, stats=stats.t)
    torch.cuda.synchronize()
    for name_, g in list(out.items()) + [("status", status), ("stats", stats), ("workspace", ws)]:
        assert g.guards_intact(), f"{name_}: a guard byte changed"
    assert int(ws.t.count_nonzero().item()) == 0, "workspace not returned to zero"
    for a, b in zip(ins, [t for t in (lg, tok, u, q) if t is not None]):
        assert torch.equal(a.view(torch.uint8) if a.dtype == torch.bfloat16 else a,
                           b.view(torch.uint8) if b.dtype == torch.bfloat16 else b), "an input changed"
    cand = {k: getattr(res, k).cpu().numpy() for k in
            ("out_tokens", "num_emitted", "accept_flags", "accept_prob", "residual_mass")}
    rep = parity.compare(orc, inp.logits, inp.q, inp.tokens, inp.u, inp.T, cand)
    assert rep.ok(), rep.summary()


@pytest.mark.parametrize("V,dtype", [(4099, "bf16"), (3001, "fp32"), (32000, "bf16")])
def test_filter_writes_only_its_buffers(orc, V, dtype):
    import speculative_decoding_sampling_gb300 as sv
    z = filter_rows.rows(V, 5, V, dtype)
    x = G.host_logits_tensor(z)
    x0 = x.clone()
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    o = Guarded((5, V), tdt)
    kept = Guarded((5,), torch.int32)
    status = Guarded((1,), torch.int32, fill=0)
    top_p = float(np.float32(0.9))
    sv.sv_filter_logits(x, 1.0, 50, top_p, out=o.t, kept=kept.t, status=status.t)
    torch.cuda.synchronize()
    assert o.guards_intact() and kept.guards_intact() and status.guards_intact()
    assert torch.equal(x.view(torch.uint8) if dtype == "bf16" else x,
                       x0.view(torch.uint8) if dtype == "bf16" else x0)
    got = o.t.cpu()
    got = got.view(torch.int16).numpy().view(np.uint16) if dtype == "bf16" else got.numpy()
    rep = parity.compare_filter(orc, z, 1.0, 50, top_p, got, kept.t.cpu().numpy())
    assert rep.ok(), rep.summary()
