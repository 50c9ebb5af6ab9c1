"""Hybrid decoder forward and decision readout, written plainly for the oracle.

What is computed (sources by page and section):
  * Decision = one prefill pass, then a softmax over the option tokens'
    logits at the last position, no decoding (Cua-S1 4B issue #10, the plan's
    first item; the sys1rust README's answer-type table).
  * The state prefix is encoded once and every question suffix continues
    from the prefix's complete state: full-attention KV and the FP32 gated
    delta-rule state (System1-Omni RFC #114, section 4 "Branching" row and
    section 5). A continuation equals the plain forward over prefix plus row
    up to rounding (RFC #114, the implementer's plan comment). The plain
    definition is therefore `decide_unbranched`; `decide_branched` is the
    faster equivalent the GPU path uses.
  * Logits are rows of the tied embedding (RFC #114, section 3: input/output
    embedding tying); the head is float32 (issue #10, "a float32 head").
  * LoRA rank 32 / alpha 64 on q, k, v, o, gate, up, down (RFC #114, section 1;
    issue #10 plan item 3). The oracle applies it UNMERGED:
    y = x W^T + (alpha/r) (x A^T) B^T.
  * Answer types and confidences: the sys1rust README, "Each question gets one
    of 3 answer types" and the two confidence bullets after it.

Readings where the pages are silent (each is listed in the design notes):
  pre-norm residual blocks; RMSNorm eps 1e-6 with weights as given; L2 norm
  x / sqrt(sum x^2 + 1e-6); a_t and b_t are per-head scalar projections
  w_a x, w_b x; no 1/sqrt(dk) on q in the delta rule; the optional short
  convolution (shape.conv_width > 0; the RFC's "convolution history" of the
  snapshot, section 5, width not given) is depthwise and causal over the
  q|k|v projections, followed by SiLU, before the L2 norms, with the last
  width-1 input rows as the continuation history; rotate-half RoPE over the
  whole head dimension with inv_freq_i = theta^(-2i/hd); plain 1-D positions,
  the suffix continuing at P; readout row = last suffix token; noul option
  ids are [yes, no]; argmax ties go to the lowest index.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field
from typing import List, Optional

import numpy as np

from . import gdn

CHOICE, SCORE, NOUL = 0, 1, 2

# Position of each LoRA target's base tensor in a layer's tensor list
# ([attn_norm, mixer..., mlp_norm, w_gate, w_up, w_down]).
_GDN_IDX = {"q": 1, "k": 2, "v": 3, "o": 6, "gate": 8, "up": 9, "down": 10}
_FA_IDX = {"q": 1, "k": 2, "v": 3, "o": 4, "gate": 6, "up": 7, "down": 8}
_TARGETS = ("q", "k", "v", "o", "gate", "up", "down")


def round_bf16(x):
    """Round to the nearest bf16 value (ties to even) and return it as float32.

    bf16 keeps the top 16 bits of an IEEE float32; rounding adds half of the dropped range
    (0x7FFF, plus one when the kept part is odd) before truncating.
    """
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    u = (u + 0x7FFF + ((u >> 16) & 1)) >> 16 << 16
    return u.astype(np.uint32).view(np.float32)


def round_f16(x):
    """Round to the nearest IEEE half-precision value (ties to even; values below 2^-14 to the
    subnormal grid of 2^-24) and return it as float32."""
    return np.asarray(x, dtype=np.float32).astype(np.float16).astype(np.float32)


def upcast(w, dt):
    """Weights as stored (float32, or bf16 bit patterns in uint16) -> dt."""
    if w is None:
        return None
    if w.dtype == np.uint16:
        return (w.astype(np.uint32) << 16).view(np.float32).astype(dt, copy=False)
    return w.astype(dt, copy=False)


def rmsnorm(x, w, eps):
    """x / sqrt(mean(x^2) + eps) * w over the last axis."""
    return x / np.sqrt(np.mean(x * x, axis=-1, keepdims=True) + x.dtype.type(eps)) * w


def silu(x):
    return x / (1.0 + np.exp(-x))


def rope(x, pos, theta):
    """Rotate-half rotary embedding over the full head dim.

    x: [T, nh, hd]; pos: [T]. Pair (i, i + hd/2) is rotated by pos * theta^(-2i/hd).
    """
    hd = x.shape[-1]
    half = hd // 2
    dt = x.dtype
    inv = np.power(np.float64(theta), -np.arange(half, dtype=np.float64) * 2.0 / hd)
    ang = pos.astype(np.float64)[:, None] * inv[None, :]
    c = np.cos(ang).astype(dt)[:, None, :]
    s = np.sin(ang).astype(dt)[:, None, :]
    x1, x2 = x[..., :half], x[..., half:]
    return np.concatenate([x1 * c - x2 * s, x2 * c + x1 * s], axis=-1)


def causal_conv(x, w, hist):
    """Depthwise causal convolution over rows, continuing from `hist`.

    x: [T, C] input rows; w: [C, W] per-channel taps, tap j weighting the row W-1-j steps
    back (tap W-1 is the current row); hist: [W-1, C] the inputs before x (zeros at the
    start of a sequence). Returns y [T, C] with y_t = sum_j w[:, j] * x_{t-(W-1)+j}, and the
    history after x (its last W-1 input rows, reaching into hist when T < W-1).
    """
    W = w.shape[1]
    xx = np.concatenate([hist, x], axis=0)
    T = x.shape[0]
    y = np.zeros_like(x)
    for j in range(W):
        y += w[:, j][None, :] * xx[j:j + T]
    new_hist = xx[xx.shape[0] - (W - 1):] if W > 1 else xx[:0]
    return y, new_hist.copy()


def attention(q, k, v, q_pos, k_pos):
    """Causal GQA attention by brute force.

    q [Tq, Hq, hd]; k, v [Tk, Hkv, hd]; query i sees key j iff k_pos[j] <= q_pos[i].
    q head h reads kv head floor(h * Hkv / Hq).
    """
    Tq, Hq, hd = q.shape
    Hkv = k.shape[1]
    dt = q.dtype
    out = np.empty((Tq, Hq, v.shape[2]), dtype=dt)
    mask = k_pos[None, :] <= q_pos[:, None]
    scale = dt.type(1.0 / math.sqrt(hd))
    for h in range(Hq):
        g = (h * Hkv) // Hq
        s = (q[:, h] @ k[:, g].T) * scale
        s = np.where(mask, s, -np.inf)
        s = s - s.max(axis=1, keepdims=True)
        p = np.exp(s)
        p /= p.sum(axis=1, keepdims=True)
        out[:, h] = p @ v[:, g]
    return out


@dataclass
class LayerCache:
    """Complete continuation state of one layer after a prefix."""
    S: Optional[np.ndarray] = None        # gated delta rule: [H, Dv, Dk]
    conv: Optional[np.ndarray] = None     # short convolution history: last w-1 input rows [w-1, C]
    K: Optional[np.ndarray] = None        # attention: post-RoPE keys [P, Hkv, hd]
    V: Optional[np.ndarray] = None
    pos: Optional[np.ndarray] = None      # key positions [P]


class Oracle:
    """precision="fp32": every step in dt, LoRA unmerged (the author's-reference semantics).
    precision="bf16" / "f16": a backbone precision policy (System1-Omni issue #10, the fast
    path's half-precision backbone with "a float32 head"; RFC #114 section 3 on merging the
    adapter): the LoRA delta is merged into each weight at load in fp32 and the merged weight
    rounded once to the 16-bit type, and every matrix-product input (normed rows, mixer output,
    SwiGLU output, attention q/k/v) is rounded to it; accumulation, the recurrent state,
    attention softmax, residual stream and the readout stay fp32. These modes measure what a
    16-bit backbone costs against the fp32 definition; "f16" is the CUDA path's policy."""

    def __init__(self, weights, dtype=np.float32, precision="fp32"):
        self.W = weights
        self.s = weights.shape
        self.dt = np.dtype(dtype)
        if precision not in ("fp32", "bf16", "f16"):
            raise ValueError(precision)
        self.policy = precision != "fp32"         # a 16-bit policy mode is active
        self.rnd = round_f16 if precision == "f16" else round_bf16
        self.full = list(self.s.layer_is_full)
        r = self.s.lora_rank
        self.lora_scale = (self.s.lora_alpha / r) if r > 0 else 0.0

    # -- building blocks ----------------------------------------------------
    def _w(self, l, i):
        return upcast(self.W.layers[l][i], self.dt)

    def linear(self, x, l, target_or_idx):
        """x W^T plus the unmerged LoRA term (alpha/r) (x A^T) B^T."""
        full = self.full[l]
        if isinstance(target_or_idx, str):
            idx = (_FA_IDX if full else _GDN_IDX)[target_or_idx]
            j = _TARGETS.index(target_or_idx)
        else:
            idx, j = target_or_idx, None
        has_lora = j is not None and self.s.lora_rank > 0 and self.W.lora_a[l][j] is not None
        if self.policy:
            Wm = self._w(l, idx)
            if has_lora:
                A = upcast(self.W.lora_a[l][j], self.dt)
                B = upcast(self.W.lora_b[l][j], self.dt)
                Wm = Wm + self.dt.type(self.lora_scale) * (B @ A)
            return self.rnd(x).astype(self.dt) @ self.rnd(Wm).astype(self.dt).T
        y = x @ self._w(l, idx).T
        if has_lora:
            A = upcast(self.W.lora_a[l][j], self.dt)
            B = upcast(self.W.lora_b[l][j], self.dt)
            y = y + self.dt.type(self.lora_scale) * ((x @ A.T) @ B.T)
        return y

    def embed_rows(self, tokens, embeds):
        E = self.W.embed
        rows = [upcast(E[np.asarray(tokens, dtype=np.int64)], self.dt)]
        if embeds is not None and len(embeds):
            rows.insert(0, upcast(embeds, self.dt))
        return np.concatenate(rows, axis=0)

    def gdn_layer(self, l, xn, cache: Optional[LayerCache]):
        s = self.s
        T = xn.shape[0]
        H, Dk, Dv = s.la_heads, s.la_dk, s.la_dv
        q = self.linear(xn, l, "q")
        k = self.linear(xn, l, "k")
        v = self.linear(xn, l, "v")
        conv_hist = None
        if s.conv_width > 0:
            # short causal convolution over the q|k|v projections, then SiLU (before the
            # L2 norms); its history continues the prefix like the recurrent state does
            qkv = np.concatenate([q, k, v], axis=1)
            Wc = self._w(l, 11)
            hist = cache.conv if cache is not None and cache.conv is not None else \
                np.zeros((s.conv_width - 1, qkv.shape[1]), dtype=self.dt)
            y, conv_hist = causal_conv(qkv, Wc, hist)
            y = silu(y)
            q, k, v = y[:, :H * Dk], y[:, H * Dk:2 * H * Dk], y[:, 2 * H * Dk:]
        q = q.reshape(T, H, Dk)
        k = k.reshape(T, H, Dk)
        v = v.reshape(T, H, Dv)
        xa = self.rnd(xn).astype(self.dt) if self.policy else xn
        a = xa @ self._w(l, 4).T
        b = xa @ self._w(l, 5).T
        q = gdn.l2norm(q, s.l2_eps)
        k = gdn.l2norm(k, s.l2_eps)
        alpha, beta = gdn.gates(a, b)
        S0 = cache.S if cache is not None else np.zeros((H, Dv, Dk), dtype=self.dt)
        o, S = gdn.recurrent(q, k, v, alpha, beta, S0)
        y = self.linear(o.reshape(T, H * Dv), l, "o")
        return y, LayerCache(S=S, conv=conv_hist)

    def attn_layer(self, l, xn, pos, cache: Optional[LayerCache]):
        s = self.s
        T = xn.shape[0]
        Hq, Hkv, hd = s.fa_q_heads, s.fa_kv_heads, s.fa_head_dim
        q = rope(self.linear(xn, l, "q").reshape(T, Hq, hd), pos, s.rope_theta)
        k = rope(self.linear(xn, l, "k").reshape(T, Hkv, hd), pos, s.rope_theta)
        v = self.linear(xn, l, "v").reshape(T, Hkv, hd)
        if self.policy:   # attention operands and the cached K/V are stored in the 16-bit type by the policy
            q, k, v = (self.rnd(t).astype(self.dt) for t in (q, k, v))
        if cache is not None:
            K = np.concatenate([cache.K, k]); V = np.concatenate([cache.V, v])
            kp = np.concatenate([cache.pos, pos])
        else:
            K, V, kp = k, v, pos
        o = attention(q, K, V, pos, kp)
        y = self.linear(o.reshape(T, Hq * hd), l, "o")
        return y, LayerCache(K=K, V=V, pos=kp)

    def mlp(self, l, xn):
        # (in a policy mode, `linear` rounds the SwiGLU output like every other product input)
        return self.linear(silu(self.linear(xn, l, "gate")) * self.linear(xn, l, "up"), l, "down")

    # -- forward ------------------------------------------------------------
    def forward(self, x, pos, caches: Optional[List[LayerCache]] = None):
        """Pre-norm blocks h = x + Mixer(RMSNorm(x)), x' = h + MLP(RMSNorm(h)).

        x: [T, d] input rows; pos: [T] absolute positions. `caches` continues a
        prefix (None = start from zero state). Returns the last layer's output
        [T, d] (before the final norm) and the per-layer continuation state.
        """
        x = x.astype(self.dt, copy=True)
        out_caches = []
        for l in range(len(self.full)):
            x, nc = self.layer(l, x, pos, caches[l] if caches is not None else None)
            out_caches.append(nc)
        return x, out_caches

    def layer(self, l, x, pos, cache: Optional[LayerCache] = None):
        """One pre-norm block l on rows x [T, d] at positions pos (continuing `cache`, None =
        from zero state): returns x' = h + MLP(RMSNorm(h)), h = x + Mixer(RMSNorm(x)), and the
        layer's continuation state."""
        eps = self.s.rms_eps
        full = self.full[l]
        x = x.astype(self.dt, copy=False)
        xn = rmsnorm(x, self._w(l, 0), eps)
        if full:
            y, nc = self.attn_layer(l, xn, pos, cache)
        else:
            y, nc = self.gdn_layer(l, xn, cache)
        h = x + y
        hn = rmsnorm(h, self._w(l, 5 if full else 7), eps)
        return h + self.mlp(l, hn), nc

    def readout(self, h_last, qtype, option_ids):
        """Decision readout from the last-layer hidden row h_last [d]."""
        hn = rmsnorm(h_last[None, :], upcast(self.W.final_norm, self.dt), self.s.rms_eps)[0]
        Eopt = upcast(self.W.embed[np.asarray(option_ids, dtype=np.int64)], self.dt)
        z = Eopt @ hn
        return decision(z, qtype)

    def option_lm_logprobs(self, h_last, option_ids):
        """Log-probability of each option token under the full vocabulary at the readout row.

        log p(o) = z_o - log sum_v exp(z_v), z = E RMSNorm(h_last), E the tied embedding
        (System1-Omni RFC #114, section 4 "Readout" row and the paragraph after the table: token
        log-probabilities normalised over the full vocabulary; a further normalisation across the
        candidates of a question gives back the option softmax). Returns (logprobs, lse).
        """
        hn = rmsnorm(h_last[None, :], upcast(self.W.final_norm, self.dt), self.s.rms_eps)[0]
        V = self.W.embed.shape[0]
        z = np.empty(V, dtype=np.float64)
        step = 16384
        for v0 in range(0, V, step):          # the full vocabulary, a block of rows at a time
            z[v0:v0 + step] = upcast(self.W.embed[v0:v0 + step], self.dt) @ hn
        m = z.max()
        lse = float(m + np.log(np.sum(np.exp(z - m))))
        return z[np.asarray(option_ids, dtype=np.int64)] - lse, lse

    def prefill(self, tokens, embeds=None):
        x0 = self.embed_rows(tokens, embeds)
        P = x0.shape[0]
        h, caches = self.forward(x0, np.arange(P), None)
        return h, caches, P

    def decide_branched(self, caches, P, questions):
        """Each question continues from the same immutable prefix state."""
        res = []
        for q in questions:
            x0 = self.embed_rows(q.suffix, None)
            pos = P + np.arange(x0.shape[0])
            h, _ = self.forward(x0, pos, caches)
            r = self.readout(h[-1], q.type, q.option_ids)
            r["hidden"] = h[-1]
            res.append(r)
        return res

    def decide_unbranched(self, tokens, embeds, questions):
        """The plain definition: a full forward over prefix + suffix per question."""
        res = []
        for q in questions:
            x0 = np.concatenate([self.embed_rows(tokens, embeds), self.embed_rows(q.suffix, None)])
            h, _ = self.forward(x0, np.arange(x0.shape[0]), None)
            r = self.readout(h[-1], q.type, q.option_ids)
            r["hidden"] = h[-1]
            res.append(r)
        return res

    def decide(self, request, branched=True):
        if branched:
            _, caches, P = self.prefill(request.tokens, request.embeds)
            return self.decide_branched(caches, P, request.questions)
        return self.decide_unbranched(request.tokens, request.embeds, request.questions)


def decision(z, qtype):
    """Probabilities, decision and confidences from one question's option logits.

    sys1rust README, answer-type table and confidence bullets:
      choice: most likely label and all probabilities; score: expected level
      sum_i i p_i (levels 0..n-1 in the given order), may fall between levels;
      noul: probability of yes (= p[0], ids given as [yes, no]).
      answer_confidence = max_i p_i (noul: max(yes, no)).
      confidence = 1 - H(p)/ln(n) for choice and score (0 for an even split,
      1 for one-hot); for noul it equals answer_confidence.
    entropy_confidence = 1 - H(p)/ln(n) for every type (n = 1 gives 1).
    """
    z = np.asarray(z)
    n = z.shape[0]
    m = np.max(z)
    e = np.exp(z - m)
    p = e / np.sum(e)
    am = int(np.argmax(p))  # first maximum on ties
    nz = p > 0
    Hn = float(-np.sum(p[nz] * np.log(p[nz])))
    ent_conf = 1.0 if n == 1 else 1.0 - Hn / math.log(n)
    ans = float(p[am])
    return {
        "probs": p,
        "argmax": am,
        "expected_score": float(np.sum(np.arange(n) * p)),
        "yes_prob": float(p[0]),
        "answer_confidence": ans,
        "confidence": ans if qtype == NOUL else ent_conf,
        "entropy_confidence": ent_conf,
        "logits": z,
    }
