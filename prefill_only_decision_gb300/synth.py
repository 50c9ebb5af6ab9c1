"""Seeded synthetic weights and requests.

The pages publish no weights and their benchmark sets are not available, so
every input is drawn here: random-init weights of the stated architecture and
uniform token streams of the stated lengths. The same arrays are handed to
the CUDA path and to the oracle. This module draws random numbers and rounds
them to bf16 bit patterns; it holds none of the method's arithmetic.

Recipe
  * weight tensor i of a model with seed s: normal(0, 0.02) from
    PCG64(SeedSequence([s, i])); RMSNorm weights are 1; LoRA A and B are both
    normal(0, 0.02).
  * bf16 models: every tensor is rounded to bf16 (round to nearest even) here,
    and both sides receive the rounded bits (numpy uint16).
  * token ids: uniform over [16, vocab) from SeedSequence([s, 1000000]);
    option ids are distinct within a question.
  * given prefix embedding rows (image-patch stand-ins): normal(0, 1), bf16,
    from SeedSequence([s, 2000000 + request]).
  * models with a short convolution (conv_width > 0): its depthwise weights
    [channels, width], normal(0, 0.3) (about the spread of a default
    1-D convolution initialisation at width 4), are the last tensor of each
    gated delta-rule layer.
"""
from __future__ import annotations

import os
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass
from typing import List, Optional

import numpy as np

from .configs import CHOICE, NOUL, SCORE, Config, ModelShape

LORA_TARGETS = ("q", "k", "v", "o", "gate", "up", "down")
TOKEN_STREAM = 1_000_000
EMBED_STREAM = 2_000_000
LORA_BASE = 500_000


def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round float32 to bf16 (nearest even) and return the 16-bit patterns."""
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32)
    r = ((u >> 16) & 1) + np.uint32(0x7FFF)
    return ((u + r) >> 16).astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.ascontiguousarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def layer_tensor_shapes(shape: ModelShape, full: bool):
    """Per-layer tensor list in the boundary's fixed order (name, [out, in])."""
    d, F = shape.d_model, shape.ffn
    out = [("attn_norm", (d,))]
    if full:
        hq, hkv, hd = shape.fa_q_heads, shape.fa_kv_heads, shape.fa_head_dim
        out += [("w_q", (hq * hd, d)), ("w_k", (hkv * hd, d)), ("w_v", (hkv * hd, d)),
                ("w_o", (d, hq * hd))]
    else:
        H, dk, dv = shape.la_heads, shape.la_dk, shape.la_dv
        out += [("w_q", (H * dk, d)), ("w_k", (H * dk, d)), ("w_v", (H * dv, d)),
                ("w_a", (H, d)), ("w_b", (H, d)), ("w_o", (d, H * dv))]
    out += [("mlp_norm", (d,)), ("w_gate", (F, d)), ("w_up", (F, d)), ("w_down", (d, F))]
    if not full and shape.conv_width > 0:
        out += [("conv", (2 * shape.la_heads * shape.la_dk + shape.la_heads * shape.la_dv, shape.conv_width))]
    return out


def lora_target_index(full: bool, target: str) -> int:
    """Position of a LoRA target's base tensor inside the layer's tensor list."""
    if full:
        return {"q": 1, "k": 2, "v": 3, "o": 4, "gate": 6, "up": 7, "down": 8}[target]
    return {"q": 1, "k": 2, "v": 3, "o": 6, "gate": 8, "up": 9, "down": 10}[target]


@dataclass
class Weights:
    shape: ModelShape
    embed: np.ndarray                 # [V, d]  uint16 (bf16 bits) or float32
    final_norm: np.ndarray            # [d]
    layers: List[List[np.ndarray]]    # per layer, fixed order
    lora_a: List[List[Optional[np.ndarray]]]   # [layer][target] -> [r, in]
    lora_b: List[List[Optional[np.ndarray]]]   # [layer][target] -> [out, r]

    @property
    def is_bf16(self) -> bool:
        return self.shape.bf16_weights


def _normal(seed: int, index: int, shp, std: float, bf16: bool) -> np.ndarray:
    g = np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, index])))
    a = g.standard_normal(size=shp, dtype=np.float32)
    a *= np.float32(std)
    return f32_to_bf16_bits(a) if bf16 else a


def _ones(shp, bf16: bool) -> np.ndarray:
    a = np.ones(shp, dtype=np.float32)
    return f32_to_bf16_bits(a) if bf16 else a


def make_weights(cfg: Config, threads: Optional[int] = None) -> Weights:
    """Draw all weights of `cfg`'s model (deterministic in the seed)."""
    shape, seed, bf16 = cfg.shape, cfg.seed, cfg.shape.bf16_weights
    threads = threads or max(1, len(os.sched_getaffinity(0)))
    jobs = []  # (key, fn)
    jobs.append((("embed",), lambda: _normal(seed, 0, (shape.vocab, shape.d_model), 0.02, bf16)))
    jobs.append((("final_norm",), lambda: _ones((shape.d_model,), bf16)))
    for l, full in enumerate(shape.layer_is_full):
        for t, (name, shp) in enumerate(layer_tensor_shapes(shape, bool(full))):
            idx = 2 + l * 64 + t
            if name.endswith("norm"):
                jobs.append((("layer", l, t), (lambda shp=shp: _ones(shp, bf16))))
            elif name == "conv":
                jobs.append((("layer", l, t), (lambda shp=shp, idx=idx: _normal(seed, idx, shp, 0.3, bf16))))
            else:
                jobs.append((("layer", l, t), (lambda shp=shp, idx=idx: _normal(seed, idx, shp, 0.02, bf16))))
        if shape.lora_rank > 0:
            tl = layer_tensor_shapes(shape, bool(full))
            for j, tgt in enumerate(LORA_TARGETS):
                out_f, in_f = tl[lora_target_index(bool(full), tgt)][1]
                r = shape.lora_rank
                ia = LORA_BASE + (l * 8 + j) * 2
                jobs.append((("la", l, j), (lambda ia=ia, r=r, in_f=in_f: _normal(seed, ia, (r, in_f), 0.02, bf16))))
                jobs.append((("lb", l, j), (lambda ia=ia, r=r, out_f=out_f: _normal(seed, ia + 1, (out_f, r), 0.02, bf16))))
    with ThreadPoolExecutor(threads) as ex:
        res = list(ex.map(lambda kv: (kv[0], kv[1]()), jobs))
    L = shape.n_layers
    layers = [[None] * len(layer_tensor_shapes(shape, bool(f))) for f in shape.layer_is_full]
    la = [[None] * len(LORA_TARGETS) for _ in range(L)]
    lb = [[None] * len(LORA_TARGETS) for _ in range(L)]
    embed = final_norm = None
    for key, arr in res:
        if key[0] == "embed":
            embed = arr
        elif key[0] == "final_norm":
            final_norm = arr
        elif key[0] == "layer":
            layers[key[1]][key[2]] = arr
        elif key[0] == "la":
            la[key[1]][key[2]] = arr
        else:
            lb[key[1]][key[2]] = arr
    return Weights(shape, embed, final_norm, layers, la, lb)


@dataclass
class Question:
    type: int
    suffix: np.ndarray       # int32 [S]
    option_ids: np.ndarray   # int32 [n]; noul: [yes, no]


@dataclass
class Request:
    tokens: np.ndarray               # int32 [P_tok]
    embeds: Optional[np.ndarray]     # uint16 bf16 bits [n_embeds, d] or None; precede tokens
    questions: List[Question]

    @property
    def prefix_rows(self) -> int:
        return len(self.tokens) + (0 if self.embeds is None else self.embeds.shape[0])


def make_requests(cfg: Config, n_requests: Optional[int] = None) -> List[Request]:
    """Draw the workload of `cfg` (deterministic in the seed)."""
    w, shape = cfg.work, cfg.shape
    V = shape.vocab
    g = np.random.Generator(np.random.PCG64(np.random.SeedSequence([cfg.seed, TOKEN_STREAM])))
    n_req = w.n_requests if n_requests is None else n_requests
    reqs = []
    for r in range(n_req):
        P = w.prefix_len
        if w.prefix_range:
            P = int(g.integers(w.prefix_range[0], w.prefix_range[1] + 1))
            if r == 0:
                P = w.prefix_len  # the first request sits at the nominal prefix length
        toks = g.integers(16, V, size=P, dtype=np.int64).astype(np.int32)
        emb = None
        if w.n_embeds:
            ge = np.random.Generator(np.random.PCG64(np.random.SeedSequence([cfg.seed, EMBED_STREAM + r])))
            emb = f32_to_bf16_bits(ge.standard_normal((w.n_embeds, shape.d_model), dtype=np.float32))
        qs = []
        for j, t in enumerate(w.types):
            if w.fixed_options:
                n = w.fixed_options[j % len(w.fixed_options)]
            elif t == NOUL:
                n = 2
            elif t == CHOICE:
                n = int(g.integers(w.choice_range[0], w.choice_range[1] + 1))
            else:
                n = int(g.integers(w.score_range[0], w.score_range[1] + 1))
            if t == NOUL:
                n = 2
            suf = g.integers(16, V, size=w.suffix_len, dtype=np.int64).astype(np.int32)
            opts = (16 + g.choice(V - 16, size=n, replace=False)).astype(np.int32)
            qs.append(Question(t, suf, opts))
        reqs.append(Request(toks, emb, qs))
    return reqs


def random_question(g: np.random.Generator, V: int, qtype: int, suffix_len: int, n_opt: int) -> Question:
    """One question with `suffix_len` tokens and `n_opt` distinct option ids."""
    if qtype == NOUL:
        n_opt = 2
    suf = g.integers(16, V, size=suffix_len, dtype=np.int64).astype(np.int32)
    opts = (16 + g.choice(V - 16, size=n_opt, replace=False)).astype(np.int32)
    return Question(qtype, suf, opts)


__all__ = ["CHOICE", "SCORE", "NOUL", "Weights", "Question", "Request", "make_weights",
           "make_requests", "random_question", "f32_to_bf16_bits", "bf16_bits_to_f32",
           "layer_tensor_shapes", "lora_target_index", "LORA_TARGETS"]
