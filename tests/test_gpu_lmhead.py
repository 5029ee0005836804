"""The LM head on the tensor cores (logits = h W^T, bf16 out) and the
verification fused behind it, through the C ABI, against the fp64 oracle."""
import numpy as np
import pytest
import torch

import speculative_decoding_sampling_gb300 as sv
import synth
from oracle import parity

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


def _dev_bf16(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to(DEV).view(torch.bfloat16)


def _host_bits(t):
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


def _value(bits):
    return (np.asarray(bits, np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def _gpu_logits(h, W):
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    out = sv.sv_lm_head_logits(_dev_bf16(h), _dev_bf16(W), status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    return _host_bits(out)


def _bound(h, W, exact):
    """|bf16(fp32 sum) - exact| <= 2^-8 |exact| + 2 err32, err32 the fp32
    summation bound d 2^-24 sum_k |h_k W_k| (any summation order)."""
    d = h.shape[1]
    absdot = np.abs(_value(h)) @ np.abs(_value(W)).T
    return 2.0**-8 * np.abs(exact) + 2 * d * 2.0**-24 * absdot + 1e-30


# (M, d, V): tiles of 128 x 256 x 64 with ragged edges on every axis: d below
# one 64-wide slice, d not a multiple of 64, V below one tile, V odd (scalar
# stores), V a multiple of 8 with an 8-wide last tile (vector stores), a long
# hidden loop that wraps the 4-stage ring many times
GEMM_SHAPES = [(1, 64, 256), (5, 8, 7), (130, 72, 300), (257, 192, 1001), (384, 512, 2056),
               (128, 4096, 512), (3, 136, 520)]


@pytest.mark.parametrize("M,d,V", GEMM_SHAPES, ids=[f"M{m}_d{d}_V{v}" for m, d, v in GEMM_SHAPES])
def test_logits_against_oracle(orc, M, d, V):
    h, W = synth.lm_head_inputs(M, d, V, seed=31 + M + d + V)
    exact = orc.lm_head(h, W)
    got = _value(_gpu_logits(h, W))
    err = np.abs(got - exact)
    bound = _bound(h, W, exact)
    bad = np.argwhere(err > bound)
    assert bad.size == 0, (bad[:5], got[tuple(bad[0])], exact[tuple(bad[0])])
    # most entries are the oracle's correctly rounded value itself
    assert (_gpu_logits(h, W) == orc.bf16_round(exact.ravel()).reshape(M, V)).mean() > 0.95


@pytest.mark.parametrize("M,d,V", [(300, 320, 1000), (129, 1024, 777), (64, 64, 4096)])
def test_logits_dyadic_bit_exact(orc, M, d, V):
    """Entries in {0, +-1/2}: every partial sum is exact in fp32, so the bf16
    logits are the oracle's rounding of the exact dot products, bit for bit."""
    h, W = synth.lm_head_inputs(M, d, V, seed=5, dyadic=True)
    want = orc.bf16_round(orc.lm_head(h, W).ravel()).reshape(M, V)
    assert np.array_equal(_gpu_logits(h, W), want)


def test_logits_empty_and_errors():
    h, W = synth.lm_head_inputs(4, 64, 100, seed=1)
    hd, Wd = _dev_bf16(h), _dev_bf16(W)
    out = sv.sv_lm_head_logits(hd[:0], Wd)
    assert out.shape == (0, 100)
    with pytest.raises(ValueError):
        sv.sv_lm_head_logits(hd, Wd[:, :32])
    with pytest.raises(sv.SpecVerifyError):  # d not a multiple of 8
        sv.sv_lm_head_logits(_dev_bf16(h[:, :12].copy()), _dev_bf16(W[:, :12].copy()))


def _fused(h, W, B, K, q, tokens, u, T, d):
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    hid = _dev_bf16(h).view(B, K + 1, d)
    res, logits = sv.spec_verify_lm_head(
        hid, _dev_bf16(W), None if q is None else torch.from_numpy(q).to(DEV),
        torch.from_numpy(tokens).to(DEV), torch.from_numpy(u).to(DEV), T, status=status)
    torch.cuda.synchronize()
    cand = {k: getattr(res, k).cpu().numpy() for k in
            ("out_tokens", "num_emitted", "accept_flags", "accept_prob", "residual_mass")}
    cand["status"] = int(status.item())
    return cand, logits


FUSED = [(24, 3, 1000, 256), (24, 0, 4097, 128), (17, 8, 32000, 256), (5, 4, 130, 64), (40, 1, 257, 192)]


@pytest.mark.parametrize("onehot", [False, True], ids=["dense", "onehot"])
@pytest.mark.parametrize("B,K,V,d", FUSED, ids=[f"B{b}_K{k}_V{v}_d{d}" for b, k, v, d in FUSED])
def test_fused_verify_against_oracle(orc, B, K, V, d, onehot):
    """Dyadic h and W make the logits exact, so the oracle verifies the very
    logits the kernels see: logits bit-exact, then the verification under the
    usual parity rule."""
    T = 0.8
    M = B * (K + 1)
    h, W = synth.lm_head_inputs(M, d, V, seed=B + 7 * K + V, dyadic=True)
    z_bits = orc.bf16_round(orc.lm_head(h, W).ravel()).reshape(B, K + 1, V)
    q, tokens, u = synth.drafts_for(_value(z_bits), T, 1.0, seed=V + K, onehot_p=0.6 if onehot else None)
    cand, logits = _fused(h, W, B, K, q, tokens, u, T, d)
    assert cand["status"] == 0
    assert np.array_equal(_host_bits(logits), z_bits)
    rep = parity.compare(orc, z_bits, q, tokens, u, T, cand)
    assert rep.ok(), rep.summary()


def test_fused_matches_unfused_on_random_weights(orc):
    """Random (non-dyadic) h and W: the logits stay within the rounding bound
    of the oracle's, and the fused call agrees with the unfused spec_verify on
    the logits the LM head wrote: the same tokens, counts and flags, and
    probabilities within 1e-5 (the fused path merges each row's softmax
    statistics from 256-id tiles, in another order than the row pass)."""
    B, K, V, d, T = 32, 4, 5000, 512, 0.7
    h, W = synth.lm_head_inputs(B * (K + 1), d, V, seed=77)
    exact = orc.lm_head(h, W)
    q, tokens, u = synth.drafts_for(exact.reshape(B, K + 1, V), T, 1.0, seed=78)
    cand, logits = _fused(h, W, B, K, q, tokens, u, T, d)
    assert cand["status"] == 0
    got = _value(_host_bits(logits)).reshape(B * (K + 1), V)
    assert (np.abs(got - exact) <= _bound(h, W, exact)).all()
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    ref = sv.spec_verify(logits, torch.from_numpy(q).to(DEV), torch.from_numpy(tokens).to(DEV),
                         torch.from_numpy(u).to(DEV), T, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    for k in ("out_tokens", "num_emitted", "accept_flags"):
        assert np.array_equal(cand[k], getattr(ref, k).cpu().numpy()), k
    for k in ("accept_prob", "residual_mass"):
        assert np.abs(cand[k] - getattr(ref, k).cpu().numpy()).max() <= 1e-5, k


def test_fused_full_size_sampled(orc):
    """B=256, K=8, V=151936, d=4096 (the large verification shape behind an
    LM head of hidden size 4096), launched as the benchmark launches it: the
    logits bit-exact against the oracle on sampled entries (dyadic inputs),
    and the whole verification of two sampled sequences against the oracle."""
    B, K, V, d, T = 256, 8, 151936, 4096, 0.7
    M = B * (K + 1)
    h, W = synth.lm_head_inputs(M, d, V, seed=4096, dyadic=True)
    rng = np.random.default_rng(9)
    seqs = np.array([3, 200])
    rows = (seqs[:, None] * (K + 1) + np.arange(K + 1)[None]).ravel()
    z_rows = orc.bf16_round(orc.lm_head(h[rows], W).ravel()).reshape(len(seqs), K + 1, V)
    # drafts: from the sampled sequences' own logits, the rest from fresh
    # Gaussian logits (any valid draft input is fine for the other sequences)
    z_all = rng.standard_normal((B, K + 1, V)).astype(np.float32) * 3
    z_all[seqs] = _value(z_rows)
    q, tokens, u = synth.drafts_for(z_all, T, 1.5, seed=10)
    cand, logits = _fused(h, W, B, K, q, tokens, u, T, d)
    assert cand["status"] == 0
    lbits = _host_bits(logits).reshape(M, V)
    r = rng.integers(0, M, 4000)
    c = rng.integers(0, V, 4000)
    want = orc.bf16_round(orc.lm_head_entries(h, W, r, c))
    assert np.array_equal(lbits[r, c], want)
    assert np.array_equal(lbits[rows].reshape(len(seqs), K + 1, V), z_rows)
    sub = {k: (v[seqs] if isinstance(v, np.ndarray) else v) for k, v in cand.items()}
    rep = parity.compare(orc, z_rows, q[seqs], tokens[seqs], u[seqs], T, sub)
    assert rep.ok(), rep.summary()


def test_fused_returns_workspace_to_zero():
    """Every byte of the workspace (the GEMM's per-tile statistics included)
    is zero again after a call, as spec_verify's rule requires."""
    B, K, V, d = 9, 3, 3000, 128
    h, W = synth.lm_head_inputs(B * (K + 1), d, V, seed=12, dyadic=True)
    z = np.zeros((B, K + 1, V))
    q, tokens, u = synth.drafts_for(z, 1.0, 1.0, seed=3)
    ws = torch.zeros(sv.sv_lm_head_workspace_bytes(B, K, V), dtype=torch.uint8, device=DEV)
    sv.spec_verify_lm_head(_dev_bf16(h).view(B, K + 1, d), _dev_bf16(W), torch.from_numpy(q).to(DEV),
                           torch.from_numpy(tokens).to(DEV), torch.from_numpy(u).to(DEV), 1.0, workspace=ws)
    torch.cuda.synchronize()
    assert int(ws.count_nonzero().item()) == 0
