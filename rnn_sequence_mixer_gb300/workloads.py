"""The five named workloads of the mixer (shapes, dtypes, seeds).

Shapes follow the RNN layers of the HypeNet models of arXiv 2601.22156
(Table 6: Qwen3-1.7B-sized HypeNet-2B has 16 heads of dim 128 and RoPE
theta 1e6; HypeNet-5B/9B have 32 heads).  Inputs are synthetic N(0, 1)
draws (``inputs.py``): the paper's efficiency runs use a trained model on real
text, which this library does not need.
"""
from __future__ import annotations

from dataclasses import dataclass

import torch


@dataclass(frozen=True)
class Workload:
    name: str
    kind: str          # "prefill", "decode" or "fwd_bwd"
    B: int
    T: int
    H: int
    d: int
    dtype: torch.dtype
    chunk: int
    rope_base: float
    seed: int
    prefill_T: int = 0  # decode: tokens of the prefill that initialises the state
    steps: int = 0      # decode: single-token steps after it
    eps: float = 1e-6

    @property
    def tokens(self) -> int:
        return self.B * (self.steps if self.kind == "decode" else self.T)


TINY_FP32 = Workload("tiny_fp32_B1_T256_H2_d64", "prefill", 1, 256, 2, 64, torch.float32, 64, 1e4, 1)
PREFILL_16K = Workload("prefill_B1_T16384_H16_d128_bf16", "prefill", 1, 16384, 16, 128,
                       torch.bfloat16, 64, 1e6, 2)
PREFILL_512K = Workload("prefill_B1_T524288_H16_d128_bf16", "prefill", 1, 524288, 16, 128,
                        torch.bfloat16, 128, 1e6, 3)
DECODE_B64 = Workload("decode_B64_H32_d128_bf16_after4096", "decode", 64, 1, 32, 128,
                      torch.bfloat16, 64, 1e6, 4, prefill_T=4096, steps=256)
DECODE_B1 = Workload("decode_B1_H16_d128_bf16_after4096", "decode", 1, 1, 16, 128,
                     torch.bfloat16, 64, 1e6, 7, prefill_T=4096, steps=256)
FWD_BWD_16K = Workload("fwd_bwd_B8_T16384_H32_d128_bf16", "fwd_bwd", 8, 16384, 32, 128,
                       torch.bfloat16, 128, 1e6, 5)

ALL = (TINY_FP32, PREFILL_16K, PREFILL_512K, DECODE_B64, DECODE_B1, FWD_BWD_16K)


@dataclass(frozen=True)
class AttentionWorkload:
    """The hybrid's softmax attention layer (Section 5.1, Eq. 11; Appendix A,
    Eq. 17).  HypeNet-2B is Qwen3-1.7B-sized: 16 query heads over 8 key/value
    heads of dim 128, logit-scale base a = 500 (Table 6)."""
    name: str
    B: int
    T: int
    Hq: int
    Hkv: int
    d: int
    a: float
    seed: int
    eps: float = 1e-6


ATTENTION_16K = AttentionWorkload("attention_B1_T16384_Hq16_Hkv8_d128_bf16_a500", 1, 16384, 16, 8,
                                  128, 500.0, 6)


@dataclass(frozen=True)
class LayerWorkload:
    """One RNN layer with its projections (Appendix A, Eq. 18): x [B, T, D] through
    x W_q,k,v,z (the feature map fused), the mixer from those features and the
    output projection.  HypeNet-2B keeps Qwen3-1.7B's width D = 2048 with 16 RNN
    heads of dim 128."""
    name: str
    B: int
    T: int
    D: int
    H: int
    d: int
    chunk: int
    rope_base: float
    seed: int
    eps: float = 1e-6


LAYER_16K = LayerWorkload("rnn_layer_B1_T16384_D2048_H16_d128_bf16", 1, 16384, 2048, 16, 128, 128,
                          1e6, 8)
