"""Pins for the oracle's attention, RoPE, norms, LoRA, MLP, branching and readout (CPU only)."""
import json
import math
import os

import numpy as np
import pytest
import torch

from oracle import model as om
from prefill_only_decision_gb300 import configs, synth

GOLD = os.path.join(os.path.dirname(__file__), "golden")


# -- attention ------------------------------------------------------------------
@pytest.mark.parametrize("Tq,Tk,Hq,Hkv", [(7, 7, 4, 2), (5, 12, 6, 3), (1, 9, 2, 1), (16, 16, 8, 8)])
def test_attention_vs_torch_sdpa(Tq, Tk, Hq, Hkv):
    """Brute force vs torch's scaled_dot_product_attention (library routine)."""
    g = np.random.default_rng(Tq * 100 + Tk)
    hd = 16
    q = g.standard_normal((Tq, Hq, hd)); k = g.standard_normal((Tk, Hkv, hd)); v = g.standard_normal((Tk, Hkv, hd))
    q_pos = np.arange(Tk - Tq, Tk); k_pos = np.arange(Tk)   # queries are the last Tq keys
    out = om.attention(q, k, v, q_pos, k_pos)
    tq = torch.from_numpy(q).permute(1, 0, 2)
    tk = torch.from_numpy(k).permute(1, 0, 2).repeat_interleave(Hq // Hkv, dim=0)
    tv = torch.from_numpy(v).permute(1, 0, 2).repeat_interleave(Hq // Hkv, dim=0)
    mask = torch.from_numpy(k_pos[None, :] <= q_pos[:, None])
    ref = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, attn_mask=mask).permute(1, 0, 2).numpy()
    np.testing.assert_allclose(out, ref, atol=1e-12)


def test_attention_causal():
    g = np.random.default_rng(1)
    q = g.standard_normal((10, 2, 8)); k = g.standard_normal((10, 1, 8)); v = g.standard_normal((10, 1, 8))
    pos = np.arange(10)
    o1 = om.attention(q, k, v, pos, pos)
    k2, v2 = k.copy(), v.copy(); k2[6:] += 5.0; v2[6:] -= 3.0
    o2 = om.attention(q, k2, v2, pos, pos)
    np.testing.assert_allclose(o1[:6], o2[:6], atol=0)
    assert np.abs(o1[6:] - o2[6:]).max() > 1e-3
    np.testing.assert_allclose(o1[0], np.repeat(v[0], 2, axis=0), atol=1e-15)   # first row sees one key


# -- RoPE -------------------------------------------------------------------------
def test_rope_identity_at_zero_and_norm():
    x = np.random.default_rng(2).standard_normal((5, 3, 32))
    np.testing.assert_allclose(om.rope(x, np.zeros(5, dtype=np.int64), 1e6), x, atol=0)
    y = om.rope(x, np.arange(5) * 1000, 1e6)
    np.testing.assert_allclose(np.linalg.norm(y, axis=-1), np.linalg.norm(x, axis=-1), rtol=1e-13)


def test_rope_complex_form():
    """Rotate-half equals multiplying complex pairs (x_i + i x_{i+hd/2}) by e^{i pos theta^(-2i/hd)}."""
    hd, theta = 64, 1e6
    x = np.random.default_rng(3).standard_normal((6, 2, hd))
    pos = np.array([0, 1, 5, 77, 1023, 4000])
    y = om.rope(x, pos, theta)
    zc = x[..., : hd // 2] + 1j * x[..., hd // 2:]
    freqs = np.array([theta ** (-(2.0 * i) / hd) for i in range(hd // 2)])
    rot = np.exp(1j * np.outer(pos, freqs))[:, None, :]
    zr = zc * rot
    np.testing.assert_allclose(y[..., : hd // 2], zr.real, atol=1e-12)
    np.testing.assert_allclose(y[..., hd // 2:], zr.imag, atol=1e-12)


def test_rope_relative_position():
    hd = 32
    g = np.random.default_rng(4)
    q = g.standard_normal((1, 1, hd)); k = g.standard_normal((1, 1, hd))
    s = [float(np.sum(om.rope(q, np.array([m + 11]), 1e6) * om.rope(k, np.array([m]), 1e6))) for m in (0, 5, 300)]
    np.testing.assert_allclose(s, s[0], rtol=1e-10)


# -- RMSNorm / MLP / LoRA -------------------------------------------------------------
def test_rmsnorm_vs_torch():
    x = np.random.default_rng(5).standard_normal((9, 48)) * 3
    w = np.random.default_rng(6).standard_normal(48)
    ref = torch.nn.functional.rms_norm(torch.from_numpy(x), (48,), torch.from_numpy(w), eps=1e-6).numpy()
    np.testing.assert_allclose(om.rmsnorm(x, w, 1e-6), ref, rtol=1e-12)
    y = om.rmsnorm(x, np.ones(48), 0.0)
    np.testing.assert_allclose(np.sqrt(np.mean(y * y, -1)), 1.0, rtol=1e-13)


def test_silu_vs_torch():
    x = np.linspace(-20, 20, 401)
    np.testing.assert_allclose(om.silu(x), torch.nn.functional.silu(torch.from_numpy(x)).numpy(), rtol=1e-14, atol=1e-300)


def _small_lora_weights():
    shape = configs.ModelShape(vocab=300, d_model=32, n_layers=4, ffn=48, la_heads=2, la_dk=8, la_dv=8,
                               fa_q_heads=4, fa_kv_heads=2, fa_head_dim=8, lora_rank=4, lora_alpha=8.0,
                               bf16_weights=False)
    return synth.make_weights(configs.Config("t", 9, shape, configs.TINY.work))


def test_lora_unmerged_equals_merged():
    W = _small_lora_weights()
    o = om.Oracle(W, np.float64)
    x = np.random.default_rng(7).standard_normal((5, 32))
    for l in range(4):
        for tgt in synth.LORA_TARGETS:
            full = bool(W.shape.layer_is_full[l])
            idx = synth.lora_target_index(full, tgt)
            j = synth.LORA_TARGETS.index(tgt)
            base = W.layers[l][idx].astype(np.float64)
            Wm = base + 2.0 * W.lora_b[l][j].astype(np.float64) @ W.lora_a[l][j].astype(np.float64)
            xin = x if tgt not in ("o", "down") else np.random.default_rng(8).standard_normal((5, base.shape[1]))
            np.testing.assert_allclose(o.linear(xin, l, tgt), xin @ Wm.T, rtol=1e-12, atol=1e-14)


def test_lora_rank0_identity():
    W = _small_lora_weights()
    x = np.random.default_rng(9).standard_normal((3, 32))
    o = om.Oracle(W, np.float64)
    o.s = configs.ModelShape(**{**W.shape.__dict__, "lora_rank": 0})
    np.testing.assert_allclose(o.linear(x, 0, "q"), x @ W.layers[0][1].astype(np.float64).T, rtol=1e-14)


def test_mlp_structure():
    """down(silu(gate x) * up x): with up = identity-like rows and down = identity, output = silu(gate x)."""
    W = _small_lora_weights()
    o = om.Oracle(W, np.float64)
    o.s = configs.ModelShape(**{**W.shape.__dict__, "lora_rank": 0})
    d, F = 32, 48
    x = np.random.default_rng(10).standard_normal((4, d))
    Wg = np.random.default_rng(11).standard_normal((F, d))
    Wu = np.zeros((F, d)); Wu[:d, :d] = np.eye(d)          # up x = [x, 0]
    Wd = np.zeros((d, F)); Wd[:d, :d] = np.eye(d)          # down h = h[:d]
    layer = list(W.layers[0])
    layer[8], layer[9], layer[10] = Wg, Wu, Wd
    o.W = synth.Weights(W.shape, W.embed, W.final_norm, [layer] + W.layers[1:], W.lora_a, W.lora_b)
    g = x @ Wg.T
    np.testing.assert_allclose(o.mlp(0, x), (g / (1 + np.exp(-g)))[:, :d] * x, rtol=1e-13)


# -- whole model ----------------------------------------------------------------------
def test_upcast_bf16_bits():
    vals = np.array([1.0, -2.5, 0.15625, 3.0e-3, 65504.0], dtype=np.float32)
    bits = synth.f32_to_bf16_bits(vals)
    back = om.upcast(bits, np.float64)
    assert np.all(np.abs(back - vals) <= np.abs(vals) * 2.0 ** -8)
    np.testing.assert_array_equal(om.upcast(np.array([0x3F80, 0xC020], np.uint16), np.float64), [1.0, -2.5])


def test_model_causal(tiny_weights, tiny_requests):
    """Row i's output does not depend on rows after i (both mixers are causal)."""
    o = om.Oracle(tiny_weights, np.float64)
    r = tiny_requests[0]
    x0 = o.embed_rows(r.tokens, None)
    h_full, _ = o.forward(x0, np.arange(len(x0)))
    h_part, _ = o.forward(x0[:40], np.arange(40))
    np.testing.assert_allclose(h_part, h_full[:40], atol=1e-12)


def test_branched_equals_unbranched_f64(tiny_weights, tiny_requests):
    o = om.Oracle(tiny_weights, np.float64)
    r = tiny_requests[0]
    rb = o.decide(r, branched=True)
    ru = o.decide(r, branched=False)
    for a, b in zip(rb, ru):
        np.testing.assert_allclose(a["hidden"], b["hidden"], atol=1e-10)
        np.testing.assert_allclose(a["probs"], b["probs"], atol=1e-12)


def test_branched_equals_unbranched_f32(tiny_weights, tiny_requests):
    o = om.Oracle(tiny_weights, np.float32)
    r = tiny_requests[0]
    for a, b in zip(o.decide(r, True), o.decide(r, False)):
        assert np.abs(a["hidden"] - b["hidden"]).max() <= 1e-5 * max(1.0, np.abs(b["hidden"]).max())


def test_question_isolation(tiny_weights, tiny_requests):
    """A question's result does not change when others are added, removed or reordered."""
    o = om.Oracle(tiny_weights, np.float64)
    r = tiny_requests[0]
    _, caches, P = o.prefill(r.tokens)
    all3 = o.decide_branched(caches, P, r.questions)
    rev = o.decide_branched(caches, P, r.questions[::-1])[::-1]
    one = o.decide_branched(caches, P, r.questions[1:2])
    for a, b in zip(all3, rev):
        np.testing.assert_array_equal(a["probs"], b["probs"])
    np.testing.assert_array_equal(all3[1]["probs"], one[0]["probs"])


# -- readout ---------------------------------------------------------------------------
def test_readout_golden():
    ex = json.load(open(os.path.join(GOLD, "readout_examples.json")))
    for c in ex["cases"]:
        r = om.decision(np.array(c["logits"], dtype=np.float64), c["type"])
        np.testing.assert_allclose(r["probs"], c["probs"], atol=1e-12)
        assert r["argmax"] == c["argmax"]
        for key in ("expected_score", "yes_prob", "answer_confidence", "confidence", "entropy_confidence"):
            assert abs(r[key] - c[key]) < 1e-9, (key, r[key], c[key])


def test_readout_invariants():
    g = np.random.default_rng(12)
    for n in range(1, 12):
        for t in (0, 1, 2):
            z = g.standard_normal(n) * 3
            r = om.decision(z, t)
            assert abs(r["probs"].sum() - 1) < 1e-12
            assert 0 <= r["expected_score"] <= n - 1
            assert 0 <= r["entropy_confidence"] <= 1 + 1e-12
            assert r["answer_confidence"] == r["probs"].max()
    # one-hot (logit gap far beyond exp range) -> confidence 1, expected score = index
    z = np.array([0.0, 0.0, 800.0, 0.0])
    r = om.decision(z, 1)
    assert r["confidence"] == 1.0 and r["expected_score"] == 2.0
    # even split -> 0
    assert abs(om.decision(np.zeros(7), 0)["confidence"]) < 1e-12
    # ties -> lowest index
    assert om.decision(np.array([1.0, 3.0, 3.0]), 0)["argmax"] == 1


# -- full-vocabulary option log-probabilities ------------------------------------------------
def test_lm_logprobs_vs_library_and_candidate_renormalisation(tiny_weights):
    from scipy.special import logsumexp
    o = om.Oracle(tiny_weights, np.float64)
    g = np.random.default_rng(13)
    h = g.standard_normal(256) * 3
    opts = np.array([17, 400, 4095, 1000], dtype=np.int32)
    lp, lse = o.option_lm_logprobs(h, opts)
    E = om.upcast(tiny_weights.embed, np.float64)
    hn = om.rmsnorm(h[None], np.ones(256), 1e-6)[0]
    z = E @ hn
    assert abs(lse - logsumexp(z)) < 1e-10
    np.testing.assert_allclose(lp, z[opts] - logsumexp(z), atol=1e-10)
    assert np.all(lp < 0) and np.exp(lp).sum() < 1
    # renormalising over the candidates gives back the option softmax of the readout
    r = o.readout(h, 0, opts)
    np.testing.assert_allclose(np.exp(lp - logsumexp(lp)), r["probs"], atol=1e-12)


# -- the bf16 backbone policy mode ------------------------------------------------------------
def test_round_bf16_vs_torch():
    g = np.random.default_rng(21)
    x = np.concatenate([g.standard_normal(10000) * 10.0 ** g.integers(-6, 6, 10000),
                        np.array([1.0, 1.00390625, 1.01171875, -2.5, 0.0, 65504.0])]).astype(np.float32)
    ref = torch.from_numpy(x).to(torch.bfloat16).to(torch.float32).numpy()
    np.testing.assert_array_equal(om.round_bf16(x), ref)


def test_bf16_policy_rounds_only_product_inputs(tiny_weights):
    """Exact bf16 inputs and weights: the bf16 mode equals the fp32 mode exactly; otherwise the
    product equals the fp32 product of the rounded operands."""
    o32 = om.Oracle(tiny_weights, np.float32)
    o16 = om.Oracle(tiny_weights, np.float32, precision="bf16")
    g = np.random.default_rng(22)
    xb = om.round_bf16(g.standard_normal((6, 256)))
    W = om.round_bf16(tiny_weights.layers[0][1])
    np.testing.assert_array_equal(o16.linear(xb, 0, 1), xb @ W.T)
    x = g.standard_normal((6, 256)).astype(np.float32)
    np.testing.assert_array_equal(o16.linear(x, 0, 1), om.round_bf16(x) @ W.T)
    assert np.abs(o16.linear(x, 0, 1) - o32.linear(x, 0, 1)).max() > 0


def test_bf16_policy_merges_lora_then_rounds():
    W = _small_lora_weights()
    o16 = om.Oracle(W, np.float64, precision="bf16")
    x = om.round_bf16(np.random.default_rng(23).standard_normal((3, 32)))
    Wm = W.layers[0][1].astype(np.float64) + 2.0 * W.lora_b[0][0].astype(np.float64) @ W.lora_a[0][0].astype(np.float64)
    np.testing.assert_allclose(o16.linear(x, 0, "q"), x @ om.round_bf16(Wm).astype(np.float64).T, rtol=1e-12)


# -- the f16 backbone policy mode (the CUDA path's rounding points) ---------------------------
def test_round_f16_vs_torch():
    g = np.random.default_rng(24)
    x = np.concatenate([g.standard_normal(10000) * 10.0 ** g.integers(-9, 4, 10000),
                        np.array([1.0, 1.0 + 2.0 ** -11, 1.0 + 3 * 2.0 ** -11, -2.5, 0.0, 65504.0, 2.0 ** -24,
                                  3 * 2.0 ** -26, 6.1e-5])]).astype(np.float32)
    ref = torch.from_numpy(x).to(torch.float16).to(torch.float32).numpy()
    np.testing.assert_array_equal(om.round_f16(x), ref)
    # ties go to the even neighbour: 1 + 2^-11 lies halfway between 1 and 1 + 2^-10
    assert om.round_f16(np.float32(1.0 + 2.0 ** -11)) == 1.0
    assert om.round_f16(np.float32(1.0 + 3 * 2.0 ** -11)) == np.float32(1.0 + 2.0 ** -9)


def test_f16_policy_merges_lora_then_rounds_and_rounds_inputs():
    W = _small_lora_weights()
    o = om.Oracle(W, np.float64, precision="f16")
    g = np.random.default_rng(25)
    x = g.standard_normal((3, 32))
    Wm = W.layers[0][1].astype(np.float64) + 2.0 * W.lora_b[0][0].astype(np.float64) @ W.lora_a[0][0].astype(np.float64)
    np.testing.assert_allclose(o.linear(x, 0, "q"),
                               om.round_f16(x).astype(np.float64) @ om.round_f16(Wm).astype(np.float64).T, rtol=1e-12)
    # the f16 rounding of the merged weight is about eight times finer than bf16's
    e16 = np.abs(om.round_f16(Wm) - Wm).max()
    eb = np.abs(om.round_bf16(Wm) - Wm).max()
    assert 0 < e16 < eb / 4


# -- given embedding rows ahead of the tokens ----------------------------------------------
def _bf16_table_weights(tiny_weights):
    """The tiny model with its embedding table rounded to bf16, so that a row of it is exactly
    representable as a given embedding row (bf16 bits)."""
    import dataclasses
    bits = synth.f32_to_bf16_bits(np.asarray(tiny_weights.embed, np.float32))
    return dataclasses.replace(tiny_weights, embed=bits), bits


def test_given_rows_precede_tokens_and_share_positions(tiny_weights, tiny_requests):
    """Given embedding rows that are exactly the table rows of ids t1, followed by tokens t2, must
    act as the prompt t1 + t2: the given rows come first, the tokens' positions continue from
    them (RoPE and causality see one sequence of len(t1) + len(t2) rows), and the rows are used
    as-is (equality with the table rows leaves no room for a scale). Swapping the order or
    restarting the tokens' positions at 0 changes the result, which is checked too, so the
    equality is sensitive to both."""
    W, bits = _bf16_table_weights(tiny_weights)
    o = om.Oracle(W, np.float64)
    r = tiny_requests[0]
    t1, t2 = r.tokens[:40], r.tokens[40:]
    given = bits[t1.astype(np.int64)]
    as_ids = synth.Request(tokens=r.tokens, embeds=None, questions=r.questions)
    as_rows = synth.Request(tokens=t2, embeds=given, questions=r.questions)
    assert as_rows.prefix_rows == len(r.tokens)
    for branched in (True, False):
        for a, b in zip(o.decide(as_ids, branched), o.decide(as_rows, branched)):
            np.testing.assert_array_equal(a["probs"], b["probs"])
            np.testing.assert_array_equal(a["hidden"], b["hidden"])
    # the row order is observable: the same rows with the given block placed after the tokens
    x_first = o.embed_rows(t2, given)
    x_ids = o.embed_rows(r.tokens, None)
    np.testing.assert_array_equal(x_first, x_ids)
    h_ids, _ = o.forward(x_ids, np.arange(len(x_ids)))
    x_last = np.concatenate([x_ids[40:], x_ids[:40]])
    h_last, _ = o.forward(x_last, np.arange(len(x_last)))
    assert np.abs(h_last[-1] - h_ids[-1]).max() > 1e-3
    # so is the numbering: tokens restarting at position 0 after the given rows
    pos_restart = np.concatenate([np.arange(40), np.arange(len(t2))])
    h_restart, _ = o.forward(x_ids, pos_restart)
    assert np.abs(h_restart[-1] - h_ids[-1]).max() > 1e-3
