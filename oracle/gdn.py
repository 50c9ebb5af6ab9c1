"""Gated delta rule (Gated DeltaNet) for the oracle.

Layer definition (the hybrid decoder's linear-attention layers; the pages
keep a "FP32 Gated DeltaNet recurrent state" per layer, System1-Omni RFC #114,
section 5 "Shared-prefix execution and performance plan"):

    alpha_t = exp(-softplus(a_t)),  beta_t = sigmoid(b_t)
    S_t     = alpha_t S_{t-1} (I - beta_t k_t k_t^T) + beta_t v_t k_t^T
    o_t     = S_t q_t

with q_t, k_t L2-normalised per head. S is [Dv, Dk] per head (it maps key
space to value space). The chunked form is the WY representation of
Yang, Kautz & Hatamizadeh, "Gated Delta Networks" (2024); RFC #114 section 5
notes that chunk boundaries may change rounding but not the result.
"""
from __future__ import annotations

import numpy as np
from scipy.linalg import solve_triangular


def softplus(x):
    """log(1 + e^x), evaluated without overflow."""
    return np.logaddexp(0.0, x).astype(x.dtype)


def sigmoid(x):
    return (1.0 / (1.0 + np.exp(-x))).astype(x.dtype)


def l2norm(x, eps):
    """x / sqrt(sum(x^2) + eps) over the last axis (eps inside the root)."""
    return x / np.sqrt(np.sum(x * x, axis=-1, keepdims=True) + x.dtype.type(eps))


def gates(a, b):
    """alpha = exp(-softplus(a)), beta = sigmoid(b), elementwise."""
    return np.exp(-softplus(a)), sigmoid(b)


def recurrent(q, k, v, alpha, beta, S0):
    """Token-by-token gated delta rule.

    q, k: [T, H, Dk] (already normalised); v: [T, H, Dv]; alpha, beta: [T, H];
    S0: [H, Dv, Dk]. Returns o [T, H, Dv] and the final state [H, Dv, Dk].

    Uses S (I - b k k^T) = S - b (S k) k^T, so each step is O(Dv*Dk):
        S_t = alpha S_{t-1} + beta (v - alpha S_{t-1} k) k^T.
    """
    T = q.shape[0]
    S = S0.copy()
    o = np.empty(v.shape, dtype=v.dtype)
    for t in range(T):
        al = alpha[t][:, None, None]
        Sk = np.einsum("hij,hj->hi", S, k[t])                   # S_{t-1} k_t   [H, Dv]
        u = beta[t][:, None] * (v[t] - alpha[t][:, None] * Sk)  # beta (v - alpha S k)
        S = al * S + u[:, :, None] * k[t][:, None, :]
        o[t] = np.einsum("hij,hj->hi", S, q[t])
    return o, S


def chunked(q, k, v, alpha, beta, S0, C):
    """Chunk-parallel form of `recurrent` with chunk length C.

    Inside a chunk (rows = tokens), with g = cumsum(log alpha),
    Gamma_ts = exp(g_t - g_s) for s <= t and gamma = exp(g):
        A  = strict_lower(diag(beta) (Gamma * K K^T)),  T = (I + A)^-1
        W  = T diag(beta * gamma) K,   Ut = T diag(beta) V,   U = Ut - W S0^T
        O  = diag(gamma) Q S0^T + lower_incl(Gamma * Q K^T) U
        S_C = gamma_C S0 + U^T diag(exp(g_C - g)) K
    U are the delta-rule write vectors beta_t (v_t - alpha_t S_{t-1} k_t); the
    system follows from unrolling S_t = alpha_t S_{t-1} + u_t k_t^T.
    """
    T, H, Dk = k.shape
    Dv = v.shape[2]
    dt = v.dtype
    o = np.empty((T, H, Dv), dtype=dt)
    S = S0.copy()
    for c0 in range(0, T, C):
        c1 = min(T, c0 + C)
        for h in range(H):
            Q, K, Vv = q[c0:c1, h], k[c0:c1, h], v[c0:c1, h]
            al, be = alpha[c0:c1, h], beta[c0:c1, h]
            g = np.cumsum(np.log(al))
            n = c1 - c0
            strict = np.tril(np.ones((n, n), dtype=bool), -1)
            incl = np.tril(np.ones((n, n), dtype=bool), 0)
            Gam = np.exp(np.where(incl, g[:, None] - g[None, :], 0.0))  # used for s <= t only
            A = np.where(strict, be[:, None] * Gam * (K @ K.T), 0).astype(dt)
            IA = np.eye(n, dtype=dt) + A
            gam = np.exp(g)
            W = solve_triangular(IA, (be * gam)[:, None] * K, lower=True, unit_diagonal=True)
            Ut = solve_triangular(IA, be[:, None] * Vv, lower=True, unit_diagonal=True)
            Sh = S[h]
            U = Ut - W @ Sh.T
            P = np.where(incl, Gam * (Q @ K.T), 0).astype(dt)
            o[c0:c1, h] = gam[:, None] * (Q @ Sh.T) + P @ U
            S[h] = gam[-1] * Sh + U.T @ (np.exp(g[-1] - g)[:, None] * K)
    return o, S
