"""The seeded input generator (CPU)."""
import numpy as np
import pytest

import synth


def test_philox_known_answers():
    """Known-answer vectors of Philox4x32-10 (Salmon et al., SC'11)."""
    assert synth.philox4x32_10([0, 0, 0, 0], [0, 0]) == [0x6627e8d5, 0xe169c58d, 0xbc57ac4c, 0x9b00dbd8]
    assert synth.philox4x32_10([0xffffffff] * 4, [0xffffffff] * 2) == \
        [0x408f276d, 0x41c83b0e, 0xa20bc7c6, 0x6d5451fd]
    assert synth.philox4x32_10([0x243f6a88, 0x85a308d3, 0x13198a2e, 0x03707344],
                               [0xa4093822, 0x299f31d0]) == \
        [0xd16cfe09, 0x94fdcceb, 0x5001e420, 0x24126ea1]


def test_bf16_round_to_nearest_even():
    bits = np.array([0x3F800000, 0x3F808000, 0x3F818000, 0x3F808001, 0xFF800000,
                     0x7F800000, 0x7FC00001, 0x00000000, 0x80000000, 0x3F7FFFFF], np.uint32)
    out = synth.f32_to_bf16(bits.view(np.float32))
    assert list(out[:6]) == [0x3F80, 0x3F80, 0x3F82, 0x3F81, 0xFF80, 0x7F80]
    assert (out[6] & 0x7F80) == 0x7F80 and (out[6] & 0x7F) != 0   # NaN stays NaN
    assert list(out[7:]) == [0x0000, 0x8000, 0x3F80]


def test_uniforms_and_shapes():
    inp = synth.generate("b8_k4_v32000_bf16")
    assert inp.logits.shape == (8, 5, 32000) and inp.logits.dtype == np.uint16
    assert inp.q.shape == (8, 4, 32000) and inp.tokens.shape == (8, 4)
    assert ((inp.u >= 0) & (inp.u < 1)).all()
    assert np.all((inp.u * 2 ** 24) == np.floor(inp.u * 2 ** 24))


def test_normals_and_bias():
    w = synth.WORKLOADS["b1_k4_v32000_fp32"]
    inp = synth.generate(w)
    z = inp.logits.astype(np.float64).ravel()
    assert abs(z.mean()) < 0.03 and abs(z.std() - 2.0) < 0.03
    w2 = w.with_(zipf_s=1.1, sigma=0.0)
    z2 = synth.generate(w2).logits[0, 0].astype(np.float64)
    assert np.allclose(z2, (-1.1 * np.log(np.arange(32000) + 1.0)).astype(np.float32))


def test_q_rows_and_drafts():
    inp = synth.generate("b8_k4_v32000_bf16")
    s = inp.q.astype(np.float64).sum(-1)
    assert np.allclose(s, 1.0, atol=1e-5)
    qx = np.take_along_axis(inp.q, inp.tokens[..., None], -1)
    assert (qx > 0).all()


def test_top_p_nucleus():
    w = synth.WORKLOADS["b64_k5_v128256_bf16_topp"].with_(B=3, V=4000)
    inp = synth.generate(w)
    raw = synth.generate(w.with_(top_p=0.0, Tq=w.Tq))
    for b in range(3):
        for j in range(w.K + 1):
            z = synth.bf16_to_f32(raw.logits[b, j]).astype(np.float64) / w.T
            p = np.exp(z - z.max()); p /= p.sum()
            keep = inp.logits[b, j] != 0xFF80
            assert p[keep].sum() >= 0.9
            assert p[keep].sum() - p[keep].min() < 0.9     # smallest such set
            assert p[keep].min() >= p[~keep].max()
        for k in range(w.K):
            qk = inp.q[b, k]
            assert abs(qk.astype(np.float64).sum() - 1) < 1e-5


def test_onehot_drafts():
    w = synth.WORKLOADS["b128_k8_v128256_bf16_onehot"].with_(V=500)
    inp = synth.generate(w)
    assert inp.q is None
    z = synth.bf16_to_f32(inp.logits[:, :w.K])
    frac = (inp.tokens == z.argmax(-1)).mean()
    assert 0.55 < frac < 0.66


def test_exponential_race_draws_follow_q():
    from scipy.stats import chisquare
    w = synth.WORKLOADS["b8_k4_v32000_bf16"].with_(B=4000, K=1, V=6, sigma=1.0, zipf_s=0.0,
                                                   draft_sigma=0.3)
    inp = synth.generate(w)
    counts = np.bincount(inp.tokens[:, 0], minlength=6)
    expect = inp.q[:, 0].astype(np.float64).sum(0)
    expect *= counts.sum() / expect.sum()
    assert chisquare(counts, expect).pvalue > 1e-3
