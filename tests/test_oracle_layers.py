"""Pins of the oracle's layer wiring (CPU): special weights under which a block, a mixer or the
readout reduces to a closed form, so that a dropped residual, a norm in the wrong place, a
swapped projection slice, a wrong GQA group or a wrong readout row fails here.

Each case follows from the layer definition the oracle implements (pre-norm residual blocks;
the gated delta rule S_t = a_t S_{t-1} (I - b_t k_t k_t^T) + b_t v_t k_t^T, o_t = S_t q_t with
L2-normalised q, k; causal GQA attention; SwiGLU; a tied-embedding readout at the last suffix
row) and not from the oracle's code."""
import numpy as np
import pytest

from oracle import model as om
from prefill_only_decision_gb300 import configs, synth

D_MODEL, H, DK, HQ, HKV, HD, FFN = 32, 2, 8, 4, 2, 8, 48


def _weights(seed=5):
    shape = configs.ModelShape(vocab=300, d_model=D_MODEL, n_layers=4, ffn=FFN, la_heads=H, la_dk=DK, la_dv=DK,
                               fa_q_heads=HQ, fa_kv_heads=HKV, fa_head_dim=HD, lora_rank=0,
                               bf16_weights=False)
    W = synth.make_weights(configs.Config("pins", seed, shape, configs.TINY.work))
    # random norm weights (not 1), so that a norm applied in the wrong place shows
    g = np.random.default_rng(seed + 100)
    for l, full in enumerate(shape.layer_is_full):
        for i in ((0, 5) if full else (0, 7)):
            W.layers[l][i] = (1.0 + 0.3 * g.standard_normal(D_MODEL)).astype(np.float32)
    W = synth.Weights(shape, W.embed, (1.0 + 0.3 * g.standard_normal(D_MODEL)).astype(np.float32), W.layers,
                      W.lora_a, W.lora_b)
    return W


# tensor positions in a layer's list: [attn_norm, mixer..., mlp_norm, gate, up, down]
GDN = dict(norm=0, q=1, k=2, v=3, a=4, b=5, o=6, mlp_norm=7, gate=8, up=9, down=10)
FA = dict(norm=0, q=1, k=2, v=3, o=4, mlp_norm=5, gate=6, up=7, down=8)


def _idx(full):
    return FA if full else GDN


def _zero(W, l, name):
    full = bool(W.shape.layer_is_full[l])
    i = _idx(full)[name]
    W.layers[l][i] = np.zeros_like(W.layers[l][i])


def _rms(x, w, eps=1e-6):
    torch = pytest.importorskip("torch")
    t = torch.from_numpy(np.asarray(x, dtype=np.float64))
    return torch.nn.functional.rms_norm(t, (t.shape[-1],), torch.from_numpy(np.asarray(w, np.float64)),
                                        eps).numpy()


def test_blocks_are_identity_when_their_outputs_are_zero():
    """With every out-projection and down-projection zero, both residual branches add nothing:
    each block, and the whole stack, returns its input rows unchanged."""
    W = _weights()
    for l in range(W.shape.n_layers):
        _zero(W, l, "o")
        _zero(W, l, "down")
    o = om.Oracle(W, np.float64)
    x = np.random.default_rng(1).standard_normal((7, D_MODEL))
    h, _ = o.forward(x, np.arange(7))
    np.testing.assert_array_equal(h, x)


@pytest.mark.parametrize("l", [0, 3])   # a gated delta-rule layer and a full-attention layer
@pytest.mark.parametrize("branch", ["mixer", "mlp"])
def test_prenorm_update_ignores_input_scale(l, branch):
    """Pre-norm: a branch sees RMSNorm(x), so with the other branch switched off the update a
    block adds, x' - x, does not change when x is scaled by c > 0 (up to the eps term)."""
    W = _weights()
    _zero(W, l, "down" if branch == "mixer" else "o")
    o = om.Oracle(W, np.float64)
    x = np.random.default_rng(2).standard_normal((6, D_MODEL))
    pos = np.arange(6)
    u1 = o.layer(l, x, pos)[0] - x
    for c in (0.5, 3.0):
        uc = o.layer(l, c * x, pos)[0] - c * x
        np.testing.assert_allclose(uc, u1, rtol=2e-5, atol=1e-9)
    assert np.abs(u1).max() > 1e-3   # the branch is not silent


def test_gdn_layer_first_tokens_closed_form():
    """With w_q = w_k (so q_t = k_t after the L2 norm) and a zero start state, two steps of the
    rule give S_1 = b_1 v_1 k_1^T and, with n_t = k_t . k_t,
      o_1 = b_1 n_1 v_1,   o_2 = a_2 b_1 (k_1 . k_2) (1 - b_2 n_2) v_1 + b_2 n_2 v_2
    per head, a = exp(-softplus(w_a x)), b = sigmoid(w_b x); the mixer output is w_o [o heads].
    (No 1/sqrt(dk) on q; n_t = 1 up to the L2 norm's eps.)"""
    W = _weights()
    l = 0
    W.layers[l][GDN["k"]] = W.layers[l][GDN["q"]].copy()
    o = om.Oracle(W, np.float64)
    xn = np.random.default_rng(3).standard_normal((2, D_MODEL))
    y, cache = o.gdn_layer(l, xn, None)
    Wl = [np.asarray(t, np.float64) for t in W.layers[l]]
    k = (xn @ Wl[GDN["k"]].T).reshape(2, H, DK)
    k = k / np.sqrt(np.sum(k * k, axis=-1, keepdims=True) + 1e-6)
    v = (xn @ Wl[GDN["v"]].T).reshape(2, H, DK)
    a = np.exp(-np.log1p(np.exp(xn @ Wl[GDN["a"]].T)))
    b = 1.0 / (1.0 + np.exp(-(xn @ Wl[GDN["b"]].T)))
    n1, n2 = np.sum(k[0] * k[0], -1), np.sum(k[1] * k[1], -1)
    k12 = np.sum(k[0] * k[1], -1)
    o1 = (b[0] * n1)[:, None] * v[0]
    o2 = (a[1] * b[0] * k12 * (1 - b[1] * n2))[:, None] * v[0] + (b[1] * n2)[:, None] * v[1]
    ref = np.stack([o1.reshape(-1), o2.reshape(-1)]) @ Wl[GDN["o"]].T
    np.testing.assert_allclose(y, ref, rtol=1e-10, atol=1e-14)
    # the state after two tokens maps k_2 to o_2 (o_t = S_t q_t with q_t = k_t)
    np.testing.assert_allclose(np.einsum("hij,hj->hi", cache.S, k[1]), o2, rtol=1e-10, atol=1e-14)


def test_attention_layer_single_row_reads_its_own_value():
    """One row attends only to itself: softmax over one key is 1, so q head h outputs the value
    row of kv head floor(h Hkv / Hq), unrotated whatever the position; the mixer output is
    w_o [those values]."""
    W = _weights()
    l = 3
    o = om.Oracle(W, np.float64)
    xn = np.random.default_rng(4).standard_normal((1, D_MODEL))
    Wl = [np.asarray(t, np.float64) for t in W.layers[l]]
    v = (xn @ Wl[FA["v"]].T).reshape(HKV, HD)
    heads = np.concatenate([v[(h * HKV) // HQ] for h in range(HQ)])
    for p in (0, 5, 1000):
        y, _ = o.attn_layer(l, xn, np.array([p]), None)
        np.testing.assert_allclose(y[0], Wl[FA["o"]] @ heads, rtol=1e-12, atol=1e-14)


def test_readout_row_and_tied_logits_through_identity_layers():
    """Identity blocks (zero out- and down-projections): the last-layer hidden row of a question
    is the embedding row of its last suffix token, and the option logits are
    E[opt] . RMSNorm(E[last]) with the final norm's weight (tied embedding)."""
    W = _weights()
    for l in range(W.shape.n_layers):
        _zero(W, l, "o")
        _zero(W, l, "down")
    o = om.Oracle(W, np.float64)
    req = synth.make_requests(configs.Config("pins", 5, W.shape, configs.TINY.work))[0]
    E = np.asarray(W.embed, np.float64)
    res = o.decide(req, branched=True)
    for q, r in zip(req.questions, res):
        last = E[int(q.suffix[-1])]
        np.testing.assert_array_equal(r["hidden"], last)
        z = E[np.asarray(q.option_ids, np.int64)] @ _rms(last[None, :], W.final_norm)[0]
        p = np.exp(z - z.max())
        p /= p.sum()
        np.testing.assert_allclose(r["probs"], p, rtol=1e-12, atol=1e-15)
