"""Candidate-tree verification (multi-step speculative sampling) through the
C ABI against the fp64 oracle."""
import numpy as np
import pytest
import torch

import speculative_decoding_sampling_gb300 as sv
import synth
from oracle import parity

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


def _dev(a):
    if a.dtype == np.uint16:
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(DEV).view(torch.bfloat16)
    return torch.from_numpy(np.ascontiguousarray(a)).to(DEV)


def _run(logits, q, parent, tokens, u, T):
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    res = sv.spec_verify_tree(_dev(logits), _dev(q), _dev(parent), _dev(tokens), _dev(u), T, status=status)
    torch.cuda.synchronize()
    cand = {k: getattr(res, k).cpu().numpy() for k in ("out_tokens", "out_nodes", "num_emitted", "accept_prob")}
    cand["status"] = int(status.item())
    return cand


CASES = [("tree16", 3000, "bf16"), ("tree16", 7, "fp32"), ("chain5", 40000, "bf16"), ("star7", 300, "fp32"),
         ("star7", 32000, "bf16"), ("tree16", 2049, "fp32")]


@pytest.mark.parametrize("shape,V,dtype", CASES, ids=[f"{s}_V{v}_{d}" for s, v, d in CASES])
def test_tree_against_oracle(orc, shape, V, dtype):
    """Ragged vocabularies (one chunk, several, a 1-id tail), both dtypes,
    chains, stars and a 16-node tree."""
    w = synth.WORKLOADS["b8_k4_v32000_bf16"].with_(B=48, V=V, dtype=dtype)
    logits, q, parent, tokens, u, T = synth.tree_inputs(w, synth.TREE_SHAPES[shape], seed=V + len(shape))
    cand = _run(logits, q, parent, tokens, u, T)
    assert cand["status"] == 0
    rep = parity.compare_tree(orc, logits, q, parent, tokens, u, T, cand)
    assert rep.ok(), rep.summary()
    assert cand["num_emitted"].min() >= 1


def test_tree_low_acceptance_many_rejections(orc):
    """Drafts far from the target (large draft noise): most siblings are
    rejected, so the residual is rebuilt many times per node."""
    w = synth.WORKLOADS["b256_k8_v151936_bf16"].with_(B=40, V=5000, draft_sigma=4.0)
    logits, q, parent, tokens, u, T = synth.tree_inputs(w, [-1] + [0] * 12 + [1, 1, 2], seed=5)
    cand = _run(logits, q, parent, tokens, u, T)
    rep = parity.compare_tree(orc, logits, q, parent, tokens, u, T, cand)
    assert rep.ok(), rep.summary()
    assert (cand["accept_prob"][:, 1:13] >= 0).sum() > 40 * 4  # many siblings were tested


def test_tree_invalid_inputs(orc):
    w = synth.WORKLOADS["b8_k4_v32000_bf16"].with_(B=6, V=500)
    logits, q, parent, tokens, u, T = synth.tree_inputs(w, synth.TREE_SHAPES["star7"], seed=9)
    parent[0, 3] = 3          # a node that is its own parent
    tokens[1, 2] = 500        # a token outside [0, V)
    q[2, 0, tokens[2, 1]] = 0  # a drafted token of zero draft probability
    u[3, 4] = 1.0             # a uniform outside [0, 1)
    cand = _run(logits, q, parent, tokens, u, T)
    assert cand["status"] & (sv.SV_BAD_U | sv.SV_BAD_TOKEN | sv.SV_BAD_Q) == (sv.SV_BAD_U | sv.SV_BAD_TOKEN | sv.SV_BAD_Q)
    assert cand["status"] & 64
    for b in range(4):
        assert cand["num_emitted"][b] == 0 and (cand["out_tokens"][b] == -1).all()
    rep = parity.compare_tree(orc, logits, q, parent, tokens, u, T, cand)
    assert rep.ok(), rep.summary()


def test_tree_single_node_is_a_plain_draw(orc):
    """N = 1 (no drafts): one token drawn from p_0."""
    w = synth.WORKLOADS["b8_k4_v32000_bf16"].with_(B=30, V=1000)
    logits, q, parent, tokens, u, T = synth.tree_inputs(w, [-1], seed=2)
    cand = _run(logits, q, parent, tokens, u, T)
    assert (cand["num_emitted"] == 1).all()
    rep = parity.compare_tree(orc, logits, q, parent, tokens, u, T, cand)
    assert rep.ok(), rep.summary()


def test_tree_full_size_sampled(orc):
    """B=64, V=128256 bf16, the 16-node tree: sampled sequences against the
    oracle."""
    w = synth.WORKLOADS["b64_k5_v128256_bf16_topp"].with_(top_p=0.0)
    logits, q, parent, tokens, u, T = synth.tree_inputs(w, synth.TREE_SHAPES["tree16"], seed=11)
    cand = _run(logits, q, parent, tokens, u, T)
    assert cand["status"] == 0
    rep = parity.compare_tree(orc, logits, q, parent, tokens, u, T, cand, seqs=[0, 17, 40, 63])
    assert rep.ok(), rep.summary()


def test_tree_returns_workspace_to_zero():
    """The workspace follows spec_verify's rule (zero before, zero after), so
    the default workspace can serve tree and chain calls of any shape."""
    w = synth.WORKLOADS["b8_k4_v32000_bf16"].with_(B=20, V=4000)
    logits, q, parent, tokens, u, T = synth.tree_inputs(w, synth.TREE_SHAPES["tree16"], seed=4)
    ws = torch.zeros(sv.sv_tree_workspace_bytes(20, 16, 4000), dtype=torch.uint8, device=DEV)
    sv.spec_verify_tree(_dev(logits), _dev(q), _dev(parent), _dev(tokens), _dev(u), T, workspace=ws)
    torch.cuda.synchronize()
    assert int(ws.count_nonzero().item()) == 0


@pytest.mark.parametrize("N,V,seed", [(256, 500, 1), (40, 20000, 2), (97, 4097, 3)])
def test_tree_random_topologies(orc, N, V, seed):
    """Random trees (each node's parent drawn uniformly from the nodes before
    it), up to the largest tree a call takes (SV_MAX_TREE_NODES = 256)."""
    rng = np.random.default_rng(seed)
    parent = [-1] + [int(rng.integers(0, i)) for i in range(1, N)]
    w = synth.WORKLOADS["b8_k4_v32000_bf16"].with_(B=12, V=V)
    logits, q, par, tokens, u, T = synth.tree_inputs(w, parent, seed=seed)
    cand = _run(logits, q, par, tokens, u, T)
    assert cand["status"] == 0
    rep = parity.compare_tree(orc, logits, q, par, tokens, u, T, cand)
    assert rep.ok(), rep.summary()
    # the path follows parent links from the root
    for b in range(12):
        n = int(cand["num_emitted"][b]) - 1
        prev = 0
        for k in range(n):
            node = int(cand["out_nodes"][b, k])
            assert par[b, node] == prev
            prev = node


def test_tree_too_many_nodes_is_refused():
    w = synth.WORKLOADS["b8_k4_v32000_bf16"].with_(B=2, V=100)
    logits, q, par, tokens, u, T = synth.tree_inputs(w, [-1] + [0] * 256, seed=1)
    with pytest.raises(sv.SpecVerifyError):
        _run(logits, q, par, tokens, u, T)
