"""Pins of the oracle's optional short causal convolution in the gated delta-rule layers
(depthwise over the q|k|v projections, SiLU after it, before the L2 norms; its last width-1
input rows continue a prefix like the recurrent state does)."""
import numpy as np
import pytest

from oracle import model as om
from prefill_only_decision_gb300 import configs, synth

D_MODEL, H, DK, HQ, HKV, HD, FFN, WIDTH = 32, 2, 8, 4, 2, 8, 48, 4


def _conv_model(seed=21, width=WIDTH):
    shape = configs.ModelShape(vocab=300, d_model=D_MODEL, n_layers=4, ffn=FFN, la_heads=H, la_dk=DK, la_dv=DK,
                               fa_q_heads=HQ, fa_kv_heads=HKV, fa_head_dim=HD, lora_rank=4, lora_alpha=8.0,
                               bf16_weights=False, conv_width=width)
    cfg = configs.Config("conv", seed, shape, configs.TINY.work)
    return synth.make_weights(cfg), synth.make_requests(cfg)


@pytest.mark.parametrize("T", [1, 2, 3, 7, 20])
def test_causal_conv_matches_numpy_convolve(T):
    """Each channel is a full 1-D convolution with the taps reversed, cut to the first T rows
    (zero history = zero padding before the sequence)."""
    g = np.random.default_rng(T)
    C = 5
    x = g.standard_normal((T, C))
    w = g.standard_normal((C, WIDTH))
    y, hist = om.causal_conv(x, w, np.zeros((WIDTH - 1, C)))
    for c in range(C):
        np.testing.assert_allclose(y[:, c], np.convolve(x[:, c], w[c, ::-1])[:T], rtol=1e-13, atol=1e-14)
    padded = np.concatenate([np.zeros((WIDTH - 1, C)), x])
    np.testing.assert_array_equal(hist, padded[-(WIDTH - 1):])


@pytest.mark.parametrize("split", [0, 1, 2, 3, 5, 11])
def test_causal_conv_continues_across_any_split(split):
    """Convolving rows [0, s) and then [s, T) from the returned history equals one pass over
    [0, T), whether or not the first part is shorter than the width."""
    g = np.random.default_rng(100 + split)
    T, C = 12, 3
    x = g.standard_normal((T, C))
    w = g.standard_normal((C, WIDTH))
    h0 = g.standard_normal((WIDTH - 1, C))
    y, h_end = om.causal_conv(x, w, h0)
    y1, h1 = om.causal_conv(x[:split], w, h0)
    y2, h2 = om.causal_conv(x[split:], w, h1)
    np.testing.assert_allclose(np.concatenate([y1, y2]), y, rtol=1e-14, atol=1e-15)
    np.testing.assert_array_equal(h2, h_end)


def test_width_one_unit_tap_is_identity():
    x = np.random.default_rng(3).standard_normal((6, 4))
    y, hist = om.causal_conv(x, np.ones((4, 1)), np.zeros((0, 4)))
    np.testing.assert_array_equal(y, x)
    assert hist.shape == (0, 4)


def test_conv_then_silu_feed_the_delta_rule():
    """With the taps a unit delta on the current row (the convolution passes its input through)
    and w_q = w_k, the layer's first two outputs follow the delta rule's two-step closed form on
    q = k = SiLU(w_k x), v = SiLU(w_v x): the convolution and SiLU sit before the L2 norms and
    act on v as well."""
    W, _ = _conv_model()
    l = 0
    W.layers[l][2] = W.layers[l][1].copy()                     # w_k = w_q
    delta = np.zeros_like(W.layers[l][11]); delta[:, -1] = 1.0
    W.layers[l][11] = delta
    o = om.Oracle(W, np.float64)
    o.s = configs.ModelShape(**{**W.shape.__dict__, "lora_rank": 0})
    xn = np.random.default_rng(4).standard_normal((2, D_MODEL))
    y, cache = o.gdn_layer(l, xn, None)
    Wl = [np.asarray(t, np.float64) for t in W.layers[l]]
    silu = lambda z: z / (1.0 + np.exp(-z))   # noqa: E731
    k = silu(xn @ Wl[2].T).reshape(2, H, DK)
    k = k / np.sqrt(np.sum(k * k, axis=-1, keepdims=True) + 1e-6)
    v = silu(xn @ Wl[3].T).reshape(2, H, DK)
    a = np.exp(-np.log1p(np.exp(xn @ Wl[4].T)))
    b = 1.0 / (1.0 + np.exp(-(xn @ Wl[5].T)))
    n1, n2 = np.sum(k[0] * k[0], -1), np.sum(k[1] * k[1], -1)
    k12 = np.sum(k[0] * k[1], -1)
    o1 = (b[0] * n1)[:, None] * v[0]
    o2 = (a[1] * b[0] * k12 * (1 - b[1] * n2))[:, None] * v[0] + (b[1] * n2)[:, None] * v[1]
    ref = np.stack([o1.reshape(-1), o2.reshape(-1)]) @ Wl[6].T
    np.testing.assert_allclose(y, ref, rtol=1e-10, atol=1e-14)
    # the history is the last width-1 pre-convolution q|k|v rows (zeros before the first)
    qkv = np.concatenate([xn @ Wl[1].T, xn @ Wl[2].T, xn @ Wl[3].T], axis=1)
    np.testing.assert_allclose(cache.conv[-2:], qkv, rtol=1e-12, atol=1e-15)
    np.testing.assert_array_equal(cache.conv[:-2], 0.0)


def test_conv_model_branched_equals_unbranched_and_is_causal():
    """With the convolution on, questions continuing the prefix snapshot (recurrent state,
    K/V and convolution history) give the plain forward over prefix + suffix."""
    W, reqs = _conv_model()
    o = om.Oracle(W, np.float64)
    r = reqs[0]
    for a, b in zip(o.decide(r, branched=True), o.decide(r, branched=False)):
        np.testing.assert_allclose(a["hidden"], b["hidden"], rtol=1e-10, atol=1e-12)
        np.testing.assert_allclose(a["probs"], b["probs"], atol=1e-12)
    x0 = o.embed_rows(r.tokens, None)
    h_full, _ = o.forward(x0, np.arange(len(x0)))
    h_part, _ = o.forward(x0[:40], np.arange(40))
    np.testing.assert_allclose(h_part, h_full[:40], atol=1e-12)


def test_conv_changes_the_model_and_width_zero_is_the_plain_layer():
    W, reqs = _conv_model()
    r = reqs[0]
    with_conv = om.Oracle(W, np.float64).decide(r, branched=True)
    plain_shape = configs.ModelShape(**{**W.shape.__dict__, "conv_width": 0})
    plain_layers = [t[:11] if len(t) == 12 else t for t in W.layers]
    Wp = synth.Weights(plain_shape, W.embed, W.final_norm, plain_layers, W.lora_a, W.lora_b)
    plain = om.Oracle(Wp, np.float64).decide(r, branched=True)
    assert max(np.abs(a["hidden"] - b["hidden"]).max() for a, b in zip(with_conv, plain)) > 1e-3
    # the plain model's weights are those of a model drawn without a convolution
    Wz = synth.make_weights(configs.Config("conv", 21, plain_shape, configs.TINY.work))
    for lp, lz in zip(plain_layers, Wz.layers):
        for a, b in zip(lp, lz):
            np.testing.assert_array_equal(a, b)
