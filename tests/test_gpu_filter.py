"""sv_filter_logits (through the C ABI) against the fp64 oracle's filter."""
import numpy as np
import pytest
import torch

import synth
from oracle import parity

import filter_rows
import gpu_util as G

pytestmark = pytest.mark.gpu


def _gpu_filter(z_np, T, top_k, top_p, in_place=False):
    import speculative_decoding_sampling_gb300 as sv
    x = G.host_logits_tensor(z_np)
    status = torch.zeros(1, dtype=torch.int32, device="cuda:0")
    out, kept = sv.sv_filter_logits(x, T, top_k, top_p, out=x if in_place else None, status=status)
    torch.cuda.synchronize()
    o = out.cpu()
    o = o.view(torch.int16).numpy().view(np.uint16) if o.dtype == torch.bfloat16 else o.numpy()
    return o, kept.cpu().numpy(), int(status.item())


def _check(orc, z, T, top_k, top_p, **kw):
    # the kernel takes top_p as fp32: the oracle gets the same value
    top_p = float(np.float32(top_p))
    out, kept, st = _gpu_filter(z, T, top_k, top_p, **kw)
    rep = parity.compare_filter(orc, z, T, top_k, top_p, out, kept)
    assert rep.ok(), rep.summary()
    return out, kept, st


SHAPES = [(1, 6), (7, 6), (1000, 6), (4099, 6), (32000, 4)]


@pytest.mark.parametrize("V,n", SHAPES, ids=[f"V{v}" for v, _ in SHAPES])
@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
def test_filter_parity(orc, V, n, dtype):
    z = filter_rows.rows(V + n, n, V, dtype)
    for top_k in (0, 1, 5, V - 1, V + 3):
        for top_p in (0.3, 0.9, 0.99, 1.0):
            for T in (0.7, 1.3):
                _check(orc, z, T, top_k, top_p)


@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
def test_filter_wide_nucleus(orc, dtype):
    """Nearly flat rows: the top-p set holds thousands of ids, more than the
    fast path's shared-memory list, so the exact fallback decides."""
    z = filter_rows.rows(11, 4, 32000, dtype, sigma=0.2)
    for top_p in (0.5, 0.9):
        _, kept, _ = _check(orc, z, 1.0, 0, top_p)
        assert kept.max() > 2048
        _check(orc, z, 1.0, 3000, top_p)   # top-k set larger than the list as well


def test_filter_ties_flat_rows(orc):
    # every id the same value: the cuts fall among ties, decided by id
    z = np.zeros((3, 100000), np.float32)
    out, kept, _ = _check(orc, z, 1.0, 777, 1.0)
    assert list(kept) == [777] * 3 and np.isfinite(out[:, :777]).all() and np.isinf(out[:, 777:]).all()
    out, kept, _ = _check(orc, z, 1.0, 0, 0.5)
    assert list(kept) == [50000] * 3
    zb = synth.f32_to_bf16(np.full((2, 70001), 1.5, np.float32))
    _check(orc, zb, 0.8, 0, 0.25)
    _check(orc, zb, 0.8, 123, 0.5)


def test_filter_bad_rows_and_in_place(orc):
    z = filter_rows.rows(5, 5, 3000, "fp32")
    z[1, 17] = np.nan
    z[2, 5] = np.inf
    z[3, :] = -np.inf
    out, kept, st = _check(orc, z.copy(), 1.0, 40, 0.9)
    assert st == 8 and kept[1] == kept[2] == kept[3] == 0
    out2, kept2, _ = _gpu_filter(z.copy(), 1.0, 40, float(np.float32(0.9)), in_place=True)
    assert np.array_equal(out2.view(np.uint32), out.view(np.uint32)) and np.array_equal(kept2, kept)


def test_filter_matches_generator_nucleus_full_size(orc):
    """The 64-sequence workload's recipe: top-p 0.9 on p at T = 1 over
    V = 128256.  Raw logits filtered on the GPU equal the generator's
    masked logits (and the oracle's) except for excused rows."""
    w = synth.WORKLOADS["b64_k5_v128256_bf16_topp"]
    raw = synth.generate(w.with_(top_p=0.0)).logits
    masked = synth.generate(w).logits
    out, kept, st = _check(orc, raw, w.T, 0, w.top_p)
    assert st == 0
    same = np.all(out.reshape(-1, w.V) == masked.reshape(-1, w.V), axis=1)
    assert same.mean() > 0.99


def test_filter_then_verify(orc):
    """Filter on the GPU, then verify the filtered logits: the same outputs
    as the oracle verifying the oracle-filtered logits."""
    import speculative_decoding_sampling_gb300 as sv
    w = synth.WORKLOADS["b64_k5_v128256_bf16_topp"].with_(B=16, V=20000)
    inp = synth.generate(w)
    raw = synth.generate(w.with_(top_p=0.0)).logits
    top_p = float(np.float32(w.top_p))
    lg = G.host_logits_tensor(raw)
    filt, kept = sv.sv_filter_logits(lg, w.T, 0, top_p)
    _, q, tok, u = G.to_device(inp)
    cand = G.run(filt, q, tok, u, inp.T)
    ref = orc.filter_logits(raw, w.T, 0, top_p)
    got = filt.cpu().view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(got, ref.logits)
    rep = parity.compare(orc, ref.logits, inp.q, inp.tokens, inp.u, inp.T, cand)
    assert rep.ok(), rep.summary()


@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
def test_filter_in_place_scalar_path(orc, dtype):
    # V odd: rows are not 16-byte groups, element loads; in place
    z = filter_rows.rows(21, 6, 5001, dtype)
    top_p = float(np.float32(0.9))
    out_a, kept_a, _ = _gpu_filter(z.copy(), 0.8, 17, top_p)
    out_b, kept_b, _ = _gpu_filter(z.copy(), 0.8, 17, top_p, in_place=True)
    assert np.array_equal(out_a.view(np.uint8), out_b.view(np.uint8)) and np.array_equal(kept_a, kept_b)
    rep = parity.compare_filter(orc, z, 0.8, 17, top_p, out_b, kept_b)
    assert rep.ok(), rep.summary()


def test_filter_largest_vocabulary(orc):
    import speculative_decoding_sampling_gb300 as sv
    V = sv.SV_MAX_V
    z = filter_rows.rows(5, 2, V, "bf16")
    _check(orc, z, 1.0, 0, 0.9)
    _check(orc, z, 0.7, 1000, 0.95)
