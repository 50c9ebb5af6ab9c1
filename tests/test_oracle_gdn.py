"""Pins for the oracle's gated delta rule (CPU only).

Each test checks the oracle against something other than itself: a hand-worked
example, closed forms of special cases, or the other of its two formulations
(token recurrence vs chunked WY form), which share no arithmetic.
"""
import json
import os

import numpy as np
import pytest
from scipy.special import expit

from oracle import gdn

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def _rand(T, H, Dk, Dv, seed, dt=np.float64):
    g = np.random.default_rng(seed)
    q = gdn.l2norm(g.standard_normal((T, H, Dk)).astype(dt), 1e-6)
    k = gdn.l2norm(g.standard_normal((T, H, Dk)).astype(dt), 1e-6)
    v = g.standard_normal((T, H, Dv)).astype(dt)
    a = g.standard_normal((T, H)).astype(dt)
    b = g.standard_normal((T, H)).astype(dt)
    S0 = (0.3 * g.standard_normal((H, Dv, Dk))).astype(dt)
    al, be = gdn.gates(a, b)
    return q, k, v, al, be, S0


def test_hand_example():
    ex = json.load(open(os.path.join(GOLD, "gdn_hand_example.json")))
    a = np.array(ex["a"]); b = np.array(ex["b"])
    al, be = gdn.gates(a, b)
    assert np.allclose(al, 0.5, atol=0, rtol=1e-15) and np.allclose(be, 0.5, atol=0, rtol=1e-15)
    q, k, v = (np.array(ex[n]) for n in ("q", "k", "v"))
    o, S = gdn.recurrent(q, k, v, al, be, np.zeros((1, 2, 2)))
    np.testing.assert_allclose(o, np.array(ex["o"]), atol=1e-14)
    np.testing.assert_allclose(S, np.array(ex["S_final"]), atol=1e-14)
    o2, S2 = gdn.chunked(q, k, v, al, be, np.zeros((1, 2, 2)), 2)
    np.testing.assert_allclose(o2, np.array(ex["o"]), atol=1e-14)
    np.testing.assert_allclose(S2, np.array(ex["S_final"]), atol=1e-14)


def test_gates_closed_form():
    x = np.linspace(-30, 30, 1001)
    al, be = gdn.gates(x, x)
    # exp(-softplus(a)) = 1 / (1 + e^a) = sigmoid(-a)
    np.testing.assert_allclose(al, expit(-x), rtol=1e-12, atol=1e-300)
    np.testing.assert_allclose(be, expit(x), rtol=1e-12, atol=1e-300)


def test_l2norm_unit():
    x = np.random.default_rng(0).standard_normal((50, 3, 64))
    n = np.linalg.norm(gdn.l2norm(x, 0.0), axis=-1)
    np.testing.assert_allclose(n, 1.0, rtol=1e-14)
    # eps sits inside the root: a zero vector stays zero
    assert np.all(gdn.l2norm(np.zeros((1, 4)), 1e-6) == 0)


def test_identity_state_when_no_write_no_decay():
    q, k, v, _, _, S0 = _rand(20, 2, 8, 6, 1)
    al = np.ones((20, 2)); be = np.zeros((20, 2))
    o, S = gdn.recurrent(q, k, v, al, be, S0)
    np.testing.assert_allclose(S, S0, atol=0)
    np.testing.assert_allclose(o, np.einsum("hij,thj->thi", S0, q), atol=1e-14)


def test_decay_only():
    q, k, v, al, _, S0 = _rand(17, 3, 8, 5, 2)
    be = np.zeros_like(al)
    _, S = gdn.recurrent(q, k, v, al, be, S0)
    np.testing.assert_allclose(S, np.prod(al, axis=0)[:, None, None] * S0, rtol=1e-12)


def test_single_token_from_zero():
    q, k, v, al, be, _ = _rand(1, 4, 8, 8, 3)
    o, S = gdn.recurrent(q, k, v, al, be, np.zeros((4, 8, 8)))
    np.testing.assert_allclose(S, be[0][:, None, None] * v[0][:, :, None] * k[0][:, None, :], atol=1e-15)
    np.testing.assert_allclose(o[0], be[0][:, None] * np.sum(k[0] * q[0], -1)[:, None] * v[0], atol=1e-15)


def test_exact_overwrite_orthonormal_keys():
    """beta = 1, alpha = 1, orthonormal keys: after writing (k, v), S k = v (delta rule)."""
    Dk, Dv, T = 8, 5, 8
    g = np.random.default_rng(4)
    Qm, _ = np.linalg.qr(g.standard_normal((Dk, Dk)))
    k = Qm.T[:, None, :]                         # T orthonormal keys
    v = g.standard_normal((T, 1, Dv))
    q = k.copy()
    S0 = g.standard_normal((1, Dv, Dk))
    o, S = gdn.recurrent(q, k, v, np.ones((T, 1)), np.ones((T, 1)), S0)
    np.testing.assert_allclose(o[:, 0], v[:, 0], atol=1e-12)          # o_t = S_t k_t = v_t
    np.testing.assert_allclose(np.einsum("ij,tj->ti", S[0], k[:, 0]), v[:, 0], atol=1e-12)


def test_exact_overwrite_partial_beta():
    """beta in (0,1), alpha = 1: S k moves a fraction beta from S k toward v."""
    Dk, Dv = 6, 4
    g = np.random.default_rng(5)
    k = gdn.l2norm(g.standard_normal((1, 1, Dk)), 0.0)
    v = g.standard_normal((1, 1, Dv))
    S0 = g.standard_normal((1, Dv, Dk))
    be = np.array([[0.3]])
    _, S = gdn.recurrent(k, k, v, np.ones((1, 1)), be, S0)
    Sk0 = S0[0] @ k[0, 0]
    np.testing.assert_allclose(S[0] @ k[0, 0], 0.7 * Sk0 + 0.3 * v[0, 0], atol=1e-13)


@pytest.mark.parametrize("T", [1, 63, 64, 65, 200])
@pytest.mark.parametrize("C", [16, 64])
def test_chunked_equals_recurrent_f64(T, C):
    q, k, v, al, be, S0 = _rand(T, 2, 16, 12, 10 + T)
    o1, S1 = gdn.recurrent(q, k, v, al, be, S0)
    o2, S2 = gdn.chunked(q, k, v, al, be, S0, C)
    np.testing.assert_allclose(o2, o1, atol=1e-10, rtol=0)
    np.testing.assert_allclose(S2, S1, atol=1e-10, rtol=0)


def test_chunked_equals_recurrent_f32():
    q, k, v, al, be, S0 = _rand(130, 2, 64, 64, 7, dt=np.float32)
    o1, S1 = gdn.recurrent(q, k, v, al, be, S0)
    o2, S2 = gdn.chunked(q, k, v, al, be, S0, 64)
    scale = np.abs(o1).max()
    assert np.abs(o2 - o1).max() <= 1e-4 * scale
    assert np.abs(S2 - S1).max() <= 1e-4 * np.abs(S1).max()


def test_chunked_strong_decay_no_overflow():
    """Very small alpha (large a): no division by cumulative decay products."""
    q, k, v, _, be, S0 = _rand(128, 1, 8, 8, 8)
    a = np.full((128, 1), 12.0)
    al, _ = gdn.gates(a, a)
    o1, S1 = gdn.recurrent(q, k, v, al, be, S0)
    o2, S2 = gdn.chunked(q, k, v, al, be, S0, 64)
    assert np.all(np.isfinite(o2)) and np.all(np.isfinite(S2))
    np.testing.assert_allclose(o2, o1, atol=1e-12)
