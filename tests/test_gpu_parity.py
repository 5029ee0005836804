"""GPU path (through the C ABI) against the fp64 oracle on seeded inputs."""
import numpy as np
import pytest
import torch

import synth
from oracle import parity

import gpu_util as G

pytestmark = pytest.mark.gpu


def _check(orc, inp, cand, seqs=None):
    rep = parity.compare(orc, inp.logits, inp.q, inp.tokens, inp.u, inp.T, cand, seqs=seqs)
    assert rep.ok(), rep.summary()
    return rep


@pytest.mark.parametrize("name", list(synth.WORKLOADS))
def test_config_full_size(orc, name):
    """Each of the five configurations at full size, every sequence checked."""
    inp = synth.generate(name)
    cand = G.run_inputs(inp)
    assert cand["status"] == 0
    rep = _check(orc, inp, cand)
    print(name, rep.summary())


SHAPES = [(1, 1), (3, 0), (7, 1), (8, 4), (9, 2), (31, 16), (257, 8), (4097, 4),
          (16385, 3), (40000, 5)]


@pytest.mark.parametrize("V,K", SHAPES, ids=[f"V{v}_K{k}" for v, k in SHAPES])
@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
@pytest.mark.parametrize("onehot", [False, True], ids=["dense", "onehot"])
def test_shapes(orc, V, K, dtype, onehot):
    """Ragged vocabularies (scalar heads and tails, several tiles, one to
    eight cluster CTAs), K from 0 to 16, both dtypes and both draft modes."""
    base = synth.WORKLOADS["b8_k4_v32000_bf16"]
    w = base.with_(name="shape", B=24, K=K, V=V, dtype=dtype,
                   Tq=0.0 if onehot else 0.8, onehot_p=0.5 if onehot else 0.0)
    inp = synth.generate(w, seed=1000 + V + 17 * K)
    cand = G.run_inputs(inp)
    assert cand["status"] == 0
    _check(orc, inp, cand)


def test_topp_masked_rows_and_zero_mass_drafts(orc):
    """-inf (masked) logits everywhere outside a nucleus, and drafts whose
    target probability is exactly 0 (always rejected)."""
    w = synth.WORKLOADS["b64_k5_v128256_bf16_topp"].with_(B=16, V=5000)
    inp = synth.generate(w, seed=7)
    masked = inp.logits == 0xFF80
    assert masked.mean() > 0.5
    # point some drafts at masked tokens: p(x) = 0, q(x) > 0
    rng = np.random.default_rng(3)
    for b in range(0, 16, 2):
        k = rng.integers(0, w.K)
        cand_ids = np.nonzero(masked[b, k] & (inp.q[b, k] > 0))[0]
        if len(cand_ids):
            inp.tokens[b, k] = cand_ids[0]
        else:
            x = np.nonzero(masked[b, k])[0][0]
            inp.q[b, k, x] = 1e-3
            inp.tokens[b, k] = x
    cand = G.run_inputs(inp)
    _check(orc, inp, cand)


def test_extreme_uniforms(orc):
    """u = 0 and u = the largest float below 1, for accept tests and the draw."""
    w = synth.WORKLOADS["b8_k4_v32000_bf16"].with_(B=32, V=3000)
    inp = synth.generate(w, seed=8)
    top = np.nextafter(np.float32(1), np.float32(0))
    inp.u[::2] = 0.0
    inp.u[1::2] = top
    cand = G.run_inputs(inp)
    _check(orc, inp, cand)


def test_p_equals_q_all_accepted(orc):
    """q(x) = p(x) exactly: one finite logit per row and one-hot q give
    p = q = 1 at the draft, so every draft is accepted."""
    B, K, V = 16, 6, 777
    rng = np.random.default_rng(9)
    logits = np.full((B, K + 1, V), -np.inf, np.float32)
    ids = rng.integers(0, V, size=(B, K + 1))
    for b in range(B):
        for j in range(K + 1):
            logits[b, j, ids[b, j]] = 0.5
    q = np.zeros((B, K, V), np.float32)
    for b in range(B):
        for k in range(K):
            q[b, k, ids[b, k]] = 1.0
    tok = ids[:, :K].astype(np.int32)
    u = rng.random((B, K + 1)).astype(np.float32)
    inp = synth.Inputs(None, logits, q, tok, u, 1.3)
    cand = G.run_inputs(inp)
    assert (cand["num_emitted"] == K + 1).all()
    assert (cand["out_tokens"] == ids).all()
    _check(orc, inp, cand)


@pytest.mark.parametrize("V", [128000, 128001], ids=["whole_groups", "ragged"])
@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
@pytest.mark.parametrize("onehot", [False, True], ids=["dense", "onehot"])
def test_stream_filling_shapes(orc, V, dtype, onehot):
    """Enough chunks (B = 24, about 125 a sequence) for the draw stream to
    fill every SM while each sequence keeps its own warps: the last of them
    makes the sequence's final draw.  An odd V puts rows off 16-byte
    boundaries, so the chunks are loaded element by element."""
    base = synth.WORKLOADS["b8_k4_v32000_bf16"]
    w = base.with_(name="fill", B=24, K=3, V=V, dtype=dtype,
                   Tq=0.0 if onehot else 0.8, onehot_p=0.5 if onehot else 0.0)
    inp = synth.generate(w, seed=31 + V % 7)
    cand = G.run_inputs(inp)
    assert cand["status"] == 0
    _check(orc, inp, cand)


@pytest.mark.parametrize("B,V", [(8, 777), (16, 128000)])
def test_degenerate_residual_draws_from_p(orc, B, V):
    """q = 1.001 p at every id (q is not renormalised): the first draft is
    rejected once u >= 1/1.001, max(p - q, 0) is 0 everywhere, so the token
    is drawn from p itself and the status says so.  The larger shape fills
    the draw stream, which then makes the final draw itself; the smaller one
    leaves it to the final pass."""
    import speculative_decoding_sampling_gb300 as sv
    K, T = 2, 1.0
    rng = np.random.default_rng(21)
    logits = rng.normal(0.0, 2.0, (B, K + 1, V)).astype(np.float32)
    z = logits.astype(np.float64) / T
    p = np.exp(z - z.max(-1, keepdims=True))
    p /= p.sum(-1, keepdims=True)
    q = (p[:, :K] * 1.001).astype(np.float32)
    tok = rng.integers(0, V, (B, K)).astype(np.int32)
    u = rng.random((B, K + 1)).astype(np.float32)
    u[:, 0] = 0.9995
    inp = synth.Inputs(None, logits, q, tok, u, T)
    cand = G.run_inputs(inp)
    assert cand["status"] == sv.SV_DEGENERATE_RESIDUAL, cand["status"]
    assert (cand["num_emitted"] == 1).all()
    assert (cand["residual_mass"] == 0.0).all()
    _check(orc, inp, cand)


def test_bad_inputs_report_and_emit_nothing(orc):
    """Bad data sets status bits, that sequence emits nothing, others are unaffected."""
    import speculative_decoding_sampling_gb300 as sv
    w = synth.WORKLOADS["b8_k4_v32000_bf16"].with_(B=8, V=1000)
    inp = synth.generate(w, seed=10)
    inp.u[1, 2] = 1.0                       # bad uniform
    inp.tokens[2, 1] = 1000                 # token out of range
    inp.q[3, 0, inp.tokens[3, 0]] = 0.0     # q(x) = 0
    inp.logits[4, 3, :] = 0xFF80            # row all -inf
    inp.logits[5, 0, 17] = 0x7FC0           # NaN logit
    inp.u[6, 4] = np.nan                    # bad final draw
    cand = G.run_inputs(inp)
    want = sv.SV_BAD_U | sv.SV_BAD_TOKEN | sv.SV_BAD_Q | sv.SV_BAD_ROW
    assert cand["status"] == want, cand["status"]
    for b in range(1, 7):
        assert cand["num_emitted"][b] == 0 and (cand["out_tokens"][b] == -1).all()
    _check(orc, inp, cand)


def test_deterministic_and_workspace_reuse(orc):
    """One workspace reused across calls of different shapes gives the same
    results as a fresh one: every call returns its counters to zero."""
    import speculative_decoding_sampling_gb300 as sv
    inp1 = synth.generate("b64_k5_v128256_bf16_topp", nb=12)
    inp2 = synth.generate("b128_k8_v128256_bf16_onehot", nb=20)
    d1, d2 = G.to_device(inp1), G.to_device(inp2)
    need = max(sv.sv_workspace_bytes(12, 5, 128256), sv.sv_workspace_bytes(20, 8, 128256))
    ws = torch.zeros(need, dtype=torch.uint8, device="cuda:0")
    a = G.run(*d1, inp1.T, workspace=ws)
    assert int(ws.count_nonzero().item()) == 0
    b = G.run(*d2, inp2.T, workspace=ws)
    assert int(ws.count_nonzero().item()) == 0
    a2 = G.run(*d1, inp1.T, workspace=ws)
    b2 = G.run(*d2, inp2.T, workspace=torch.zeros_like(ws))
    for k in ("out_tokens", "num_emitted", "accept_flags", "accept_prob", "residual_mass"):
        assert np.array_equal(a[k], a2[k]), k
        assert np.array_equal(b[k], b2[k]), k
    _check(orc, inp1, a)
    _check(orc, inp2, b)


def test_stages_equal_whole_call(orc):
    import speculative_decoding_sampling_gb300 as sv
    inp = synth.generate("b128_k8_v128256_bf16_onehot", nb=16)
    logits, q, tok, u = G.to_device(inp)
    whole = G.run(logits, q, tok, u, inp.T)
    B, K = inp.tokens.shape
    V = inp.logits.shape[2]
    dev = logits.device
    out = {"out_tokens": torch.empty((B, K + 1), dtype=torch.int32, device=dev),
           "num_emitted": torch.empty((B,), dtype=torch.int32, device=dev),
           "accept_flags": torch.empty((B, K), dtype=torch.int8, device=dev),
           "accept_prob": torch.empty((B, K), dtype=torch.float32, device=dev),
           "residual_mass": torch.empty((B,), dtype=torch.float32, device=dev)}
    ws = torch.zeros(sv.sv_workspace_bytes(B, K, V), dtype=torch.uint8, device=dev)
    sv.sv_verify_rows(logits, q, tok, u, inp.T, out=out, workspace=ws)
    sv.sv_sample_survivors(logits, q, tok, u, inp.T, out=out, workspace=ws)
    torch.cuda.synchronize()
    for k in out:
        assert np.array_equal(out[k].cpu().numpy(), whole[k]), k


def test_misaligned_base_pointers(orc):
    """Tensors that start off a 16-byte boundary take the scalar paths."""
    w = synth.WORKLOADS["b8_k4_v32000_bf16"].with_(B=6, V=2051)
    inp = synth.generate(w, seed=12)
    B, K1, V = inp.logits.shape
    flat = torch.empty(B * K1 * V + 3, dtype=torch.bfloat16, device="cuda:0")
    logits = flat[3:].view(B, K1, V)
    logits.copy_(G.host_logits_tensor(inp.logits))
    qflat = torch.empty(B * (K1 - 1) * V + 1, dtype=torch.float32, device="cuda:0")
    q = qflat[1:].view(B, K1 - 1, V)
    q.copy_(torch.from_numpy(inp.q))
    tok = torch.from_numpy(inp.tokens).cuda()
    u = torch.from_numpy(inp.u).cuda()
    cand = G.run(logits, q, tok, u, inp.T)
    _check(orc, inp, cand)


@pytest.mark.parametrize("onehot", [False, True], ids=["dense", "onehot"])
def test_many_short_sequences(orc, onehot):
    """More sequences than draw warps (B = 5000, V = 300): each warp's chunk
    range then spans several sequences, each with its own verdict."""
    base = synth.WORKLOADS["b8_k4_v32000_bf16"]
    w = base.with_(name="many", B=5000, K=2, V=300, Tq=0.0 if onehot else 0.8,
                   onehot_p=0.5 if onehot else 0.0)
    inp = synth.generate(w, seed=31 + int(onehot))
    cand = G.run_inputs(inp)
    assert cand["status"] == 0
    _check(orc, inp, cand)


@pytest.mark.parametrize("onehot", [False, True], ids=["dense", "onehot"])
def test_largest_vocabulary(orc, onehot):
    """V = SV_MAX_V (2^21): 2048 draw chunks per row, 22 fraction bits for
    the largest fixed-point totals."""
    from speculative_decoding_sampling_gb300 import _native as N
    base = synth.WORKLOADS["b8_k4_v32000_bf16"]
    w = base.with_(name="maxv", B=3, K=2, V=N.SV_MAX_V, Tq=0.0 if onehot else 0.8,
                   onehot_p=0.5 if onehot else 0.0)
    inp = synth.generate(w, seed=41 + int(onehot))
    cand = G.run_inputs(inp)
    assert cand["status"] == 0
    _check(orc, inp, cand)


@pytest.mark.parametrize("where", ["q_pinned", "all_pinned"])
def test_pinned_host_inputs_read_in_place(orc, where):
    """Page-locked host inputs are read in place by the kernels and give the
    same results as device-resident ones."""
    import speculative_decoding_sampling_gb300 as sv
    w = synth.WORKLOADS["b64_k5_v128256_bf16_topp"].with_(B=12, V=20000)
    inp = synth.generate(w, seed=51)
    lg, q, tok, u = G.to_device(inp)
    ref = G.run(lg, q, tok, u, inp.T)
    hq = q.cpu().pin_memory()
    if where == "all_pinned":
        hlg = lg.cpu().pin_memory()
        htok, hu = tok.cpu().pin_memory(), u.cpu().pin_memory()
    else:
        hlg, htok, hu = lg, tok, u
    status = torch.zeros(1, dtype=torch.int32, device="cuda:0")
    res = sv.spec_verify(hlg, hq, htok, hu, inp.T, status=status)
    torch.cuda.synchronize()
    got = {"out_tokens": res.out_tokens.cpu().numpy(), "num_emitted": res.num_emitted.cpu().numpy(),
           "accept_flags": res.accept_flags.cpu().numpy(), "accept_prob": res.accept_prob.cpu().numpy(),
           "residual_mass": res.residual_mass.cpu().numpy(), "status": int(status.item())}
    for k in ("out_tokens", "num_emitted", "accept_flags", "accept_prob", "residual_mass"):
        assert np.array_equal(got[k], ref[k]), k
    assert got["status"] == ref["status"]
    _check(orc, inp, got)


def test_acceptance_statistics_counters(orc):
    """spec_verify_stats: the verdicts' counters equal those counted from the
    fp64 oracle's outputs on the same inputs, add up over calls, and leave
    out sequences with bad data."""
    import speculative_decoding_sampling_gb300 as sv
    from speculative_decoding_sampling_gb300.adaptive import RoundStats, stats_buffer
    w = synth.WORKLOADS["b8_k4_v32000_bf16"].with_(B=40, V=3000)
    inp = synth.generate(w, seed=61)
    inp.u[3, 0] = 1.5                       # a bad uniform: sequence 3 emits nothing
    lg, q, tok, u = G.to_device(inp)
    B, K = inp.tokens.shape
    stats = stats_buffer(K)
    status = torch.zeros(1, dtype=torch.int32, device="cuda:0")
    res = sv.spec_verify(lg, q, tok, u, inp.T, status=status, stats=stats)
    sv.spec_verify(lg, q, tok, u, inp.T, status=status, stats=stats)
    torch.cuda.synchronize()
    ref = orc.verify(inp.logits, inp.q, inp.tokens, inp.u, inp.T)
    rep = parity.compare(orc, inp.logits, inp.q, inp.tokens, inp.u, inp.T,
                         {"out_tokens": res.out_tokens.cpu().numpy(), "num_emitted": res.num_emitted.cpu().numpy(),
                          "accept_flags": res.accept_flags.cpu().numpy(),
                          "accept_prob": res.accept_prob.cpu().numpy(),
                          "residual_mass": res.residual_mass.cpu().numpy()}, oracle_res=ref)
    assert rep.ok() and rep.excused == 0, rep.summary()   # every accept test decided as the oracle did
    n = ref.num_emitted.astype(np.int64)                  # the counts come from the oracle's outputs
    ok = n > 0
    assert not ok[3] and ok.sum() == B - 1
    s = RoundStats.from_counters(stats.cpu())
    assert s.sequences == 2 * ok.sum()
    assert s.proposed == 2 * K * ok.sum()
    assert s.accepted == 2 * (n[ok] - 1).sum()
    assert s.emitted == 2 * n[ok].sum()
    assert s.accepted_hist == tuple(2 * int(((n - 1) == a)[ok].sum()) for a in range(K + 1))
    _check(orc, inp, {"out_tokens": res.out_tokens.cpu().numpy(), "num_emitted": n,
                      "accept_flags": res.accept_flags.cpu().numpy(),
                      "accept_prob": res.accept_prob.cpu().numpy(),
                      "residual_mass": res.residual_mass.cpu().numpy(), "status": int(status.item())})


def test_kernel_launch_count():
    """sv_kernel_launches: a draw stream that fills the GPU makes its own
    final draws (2 kernels); a small one leaves them to the final kernel (3)."""
    import speculative_decoding_sampling_gb300 as sv
    assert sv.sv_kernel_launches(torch.bfloat16, True, 256, 8, 151936) == 2
    assert sv.sv_kernel_launches(torch.bfloat16, False, 128, 8, 128256) == 2
    assert sv.sv_kernel_launches(torch.bfloat16, True, 8, 4, 32000) == 3
    assert sv.sv_kernel_launches(torch.float32, True, 1, 4, 32000) == 3
    assert sv.sv_kernel_launches(torch.bfloat16, True, 0, 4, 32000) == 0


def test_worked_example_on_the_gpu(orc):
    """The pages' worked example ("推测解码：草稿、验证与实际加速", section
    算完三个 token 的全部概率) through the CUDA path: logits = ln p at T = 1,
    p = (1/2, 3/10, 1/5) and q = (3/5, 1/10, 3/10) at every position, drafts
    A, C, B, draws 7/10, 9/10, 1/5 and final draw 1/5: A passes at 5/6, C fails
    at 2/3, B is never reached, and the correction from the residual (0, 1, 0)
    is B -- [A, B] emitted (tests/golden/worked_example.txt)."""
    from fractions import Fraction as F
    from oracle_pins import read_golden
    g = read_golden("worked_example.txt")
    ids = {name: i for i, name in enumerate(g["tokens"])}
    p = np.array([float(F(x)) for x in g["p"]])
    q = np.array([float(F(x)) for x in g["q"]], np.float32)
    draft = [ids[x] for x in g["draft"]]
    K = len(draft)
    u = np.array([[float(F(x)) for x in g["draws"]] + [float(F(g["final_draw"][0]))]], np.float32)
    logits = np.log(p).astype(np.float32)[None, None].repeat(K + 1, 1)
    inp = synth.Inputs(None, logits, q[None, None].repeat(K, 1).copy(), np.array([draft], np.int32), u, 1.0)
    cand = G.run_inputs(inp)
    emit = [ids[x] for x in g["emit"]]
    assert cand["status"] == 0
    assert cand["num_emitted"][0] == len(emit)
    assert list(cand["out_tokens"][0]) == emit + [-1] * (K + 1 - len(emit))
    assert list(cand["accept_flags"][0]) == [1, 0, -1]
    a = [float(F(x)) for x in g["accept_prob_per_token"]]   # per token A, B, C
    assert abs(cand["accept_prob"][0, 0] - a[ids["A"]]) < 1e-5
    assert abs(cand["accept_prob"][0, 1] - a[ids["C"]]) < 1e-5
    assert abs(cand["residual_mass"][0] - (1 - float(F(g["acceptance"][0])))) < 1e-5
    _check(orc, inp, cand)


def test_p_equals_q_on_random_rows(orc):
    """q = fp32 of the fp64 softmax of the target row at every drafted
    position (p = q up to rounding): every draft is accepted in at least
    99.999 % of the sequences, and the outputs match the oracle."""
    B, K, V, T = 20000, 4, 256, 1.0
    rng = np.random.default_rng(77)
    z = rng.normal(0.0, 2.0, (B, K + 1, V)).astype(np.float32)
    p = np.exp(z.astype(np.float64) - z.max(-1, keepdims=True))
    p /= p.sum(-1, keepdims=True)
    q = p[:, :K].astype(np.float32)
    tok = np.empty((B, K), np.int32)
    for k in range(K):   # drafts drawn from q by the inverse CDF of seeded uniforms
        c = np.cumsum(q[:, k].astype(np.float64), -1)
        r = rng.random(B) * c[:, -1]
        tok[:, k] = np.minimum((c < r[:, None]).sum(-1), V - 1)
    u = rng.random((B, K + 1)).astype(np.float32)
    inp = synth.Inputs(None, z, q, tok, u, T)
    cand = G.run_inputs(inp)
    assert cand["status"] == 0
    full = (cand["num_emitted"] == K + 1).mean()
    assert full >= 1 - 1e-5, full
    _check(orc, inp, cand)
