"""Model shapes and request workloads for the five synthetic configurations.

Shapes follow the hybrid-decoder description of the System1-Omni RFC #114
("24 linear-attention and 8 full-attention layers", rank-32 / alpha-64
adapter) and the Cua-S1 4B issue #10; the sizes of the tiny, small and
27B-class models are the synthetic stand-ins used for parity and scaling.
Every fourth layer (index 3, 7, ...) is full attention, the rest are gated
delta-rule layers.

This module holds sizes only: no arithmetic of the method.
"""
from __future__ import annotations

from dataclasses import dataclass, field
from typing import List


@dataclass(frozen=True)
class ModelShape:
    vocab: int
    d_model: int
    n_layers: int
    ffn: int
    la_heads: int
    la_dk: int
    la_dv: int
    fa_q_heads: int
    fa_kv_heads: int
    fa_head_dim: int
    rope_theta: float = 1.0e6
    rms_eps: float = 1.0e-6
    l2_eps: float = 1.0e-6
    lora_rank: int = 0
    lora_alpha: float = 0.0
    bf16_weights: bool = True
    # short causal convolution over each gated delta-rule layer's q|k|v projections (0: none).
    # Oracle only for now: the CUDA path refuses models that set it.
    conv_width: int = 0

    @property
    def layer_is_full(self) -> List[int]:
        return [1 if (l % 4) == 3 else 0 for l in range(self.n_layers)]

    def n_params(self, with_embed: bool = True) -> int:
        d, F = self.d_model, self.ffn
        tot = 0
        for full in self.layer_is_full:
            tot += 2 * d  # norms
            if full:
                hq, hkv, hd = self.fa_q_heads, self.fa_kv_heads, self.fa_head_dim
                tot += (hq + 2 * hkv) * hd * d + d * hq * hd
            else:
                H, dk, dv = self.la_heads, self.la_dk, self.la_dv
                tot += (2 * H * dk + H * dv + 2 * H) * d + d * H * dv
                tot += (2 * H * dk + H * dv) * self.conv_width
            tot += 3 * F * d
        if with_embed:
            tot += self.vocab * d + d
        return tot


CHOICE, SCORE, NOUL = 0, 1, 2
TYPE_NAMES = {CHOICE: "choice", SCORE: "score", NOUL: "noul"}


@dataclass
class Workload:
    """Request mix of one configuration.

    n_requests requests, each with a prefix of `prefix_len` token rows
    (after `n_embeds` given embedding rows) and `types` questions whose
    suffixes have `suffix_len` tokens. Option counts per question are drawn
    from `choice_range` / `score_range` (inclusive) unless `fixed_options`
    gives them; noul questions always have two ids (yes, no).
    """
    n_requests: int
    prefix_len: int
    suffix_len: int
    types: List[int]
    n_embeds: int = 0
    fixed_options: List[int] = field(default_factory=list)
    choice_range: tuple = (2, 8)
    score_range: tuple = (2, 8)
    prefix_range: tuple = ()   # (lo, hi) inclusive: per-request prefix drawn from it


@dataclass
class Config:
    name: str
    seed: int
    shape: ModelShape
    work: Workload


TINY = Config(
    "tiny", 0,
    ModelShape(vocab=4096, d_model=256, n_layers=4, ffn=768, la_heads=4, la_dk=64, la_dv=64,
               fa_q_heads=4, fa_kv_heads=2, fa_head_dim=64, bf16_weights=False),
    Workload(n_requests=1, prefix_len=96, suffix_len=24, types=[CHOICE, SCORE, NOUL],
             fixed_options=[3, 4, 2]),
)

SMALL = Config(
    "small", 1,
    ModelShape(vocab=32000, d_model=1024, n_layers=8, ffn=3072, la_heads=8, la_dk=128, la_dv=128,
               fa_q_heads=8, fa_kv_heads=2, fa_head_dim=128, lora_rank=32, lora_alpha=64.0),
    Workload(n_requests=16, prefix_len=512, suffix_len=32, types=[CHOICE, SCORE, NOUL, CHOICE],
             choice_range=(2, 8), score_range=(2, 8)),
)

QWEN4B = Config(
    "4b", 2,
    ModelShape(vocab=151936, d_model=2560, n_layers=32, ffn=9216, la_heads=16, la_dk=128, la_dv=128,
               fa_q_heads=16, fa_kv_heads=4, fa_head_dim=128, lora_rank=32, lora_alpha=64.0),
    Workload(n_requests=1, prefix_len=1024, suffix_len=48, types=[CHOICE, SCORE, NOUL],
             fixed_options=[3, 4, 2]),
)

QWEN4B_MM = Config(
    "4b_mm", 3,
    QWEN4B.shape,
    Workload(n_requests=8, prefix_len=256, n_embeds=1024, suffix_len=40,
             types=[CHOICE, SCORE, NOUL] * 10 + [CHOICE, SCORE],
             choice_range=(2, 10), score_range=(3, 7)),
)

QWEN27B = Config(
    "27b", 4,
    ModelShape(vocab=151936, d_model=5120, n_layers=64, ffn=17408, la_heads=32, la_dk=128, la_dv=128,
               fa_q_heads=40, fa_kv_heads=8, fa_head_dim=128, lora_rank=32, lora_alpha=64.0),
    Workload(n_requests=74, prefix_len=1536, suffix_len=64, types=[CHOICE], fixed_options=[4],
             prefix_range=(512, 3072)),
)

CONFIGS = {c.name: c for c in (TINY, SMALL, QWEN4B, QWEN4B_MM, QWEN27B)}
