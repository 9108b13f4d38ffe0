"""Seeded synthetic inputs shared by the tests, the smoke check and the bench.

Holds no attention arithmetic: it only draws N(0,1) values (rounded to
bf16) from a seeded CPU generator and lays them out in the requested storage
order, so the CUDA path and the oracle see bit-identical inputs.

The recipe follows the gradient-parity repro of diffusers issue #14265
("Reproduction": torch.manual_seed(777), q/k/v/grad_out ~ randn in bf16);
shapes are those of the workloads the library is measured on (Flux-like
joint sequences, long video-DiT sequences, sequence-first DeepSpeed layout).
"""
from __future__ import annotations

from dataclasses import dataclass

import torch

DEFAULT_SEED = 777


@dataclass(frozen=True)
class AttnShape:
    B: int
    S: int
    Hq: int
    Hkv: int
    D: int
    P: int
    layout: str = "bshd"  # storage order: "bshd" = [B,S,H,D], "sbhd" = [S,B,H,D]


# The workloads, by what they are.
MHA_B2_S512_P2 = AttnShape(B=2, S=512, Hq=8, Hkv=8, D=64, P=2, layout="bshd")
SEQFIRST_S1001_P4 = AttnShape(B=1, S=1001, Hq=16, Hkv=16, D=64, P=4, layout="sbhd")
FLUX_GQA_S4608_P4 = AttnShape(B=1, S=4608, Hq=24, Hkv=8, D=128, P=4, layout="bshd")
VIDEO_S32760_P8 = AttnShape(B=1, S=32760, Hq=24, Hkv=24, D=128, P=8, layout="bshd")
# causal language model of the DeepSpeed Ulysses pull request's end-to-end
# check: 24 query heads, 4 key/value heads, head dimension 256, 1024 tokens,
# sequence parallelism 2 (and 8)
GQA_D256_S1024 = AttnShape(B=1, S=1024, Hq=24, Hkv=4, D=256, P=2, layout="bshd")
# ring 4 x ulysses 2 hybrid: exchange of [1,65536,32,128] (+ k, v with 8 heads),
# then GQA 32/8 attention over 4 ring chunks on the exchanged tensors.
HYBRID_S65536 = AttnShape(B=1, S=65536, Hq=32, Hkv=8, D=128, P=4, layout="bshd")
HYBRID_RING, HYBRID_ULYSSES = 4, 2


def _randn_bf16(shape, gen):
    return torch.randn(*shape, generator=gen, dtype=torch.float32).to(torch.bfloat16)


def _store(t_bshd: torch.Tensor, layout: str) -> torch.Tensor:
    """Return a logical [B,S,H,D] view whose storage is in `layout` order."""
    if layout == "bshd":
        return t_bshd.contiguous()
    if layout == "sbhd":
        return t_bshd.permute(1, 0, 2, 3).contiguous().permute(1, 0, 2, 3)
    raise ValueError(layout)


def attn_inputs(shape: AttnShape, seed: int = DEFAULT_SEED):
    """q, k, v, dout as CPU bf16 logical [B,S,H,D] views stored in shape.layout order.

    The draw order is q, k, v, dout, each ~N(0,1) rounded to bf16."""
    g = torch.Generator().manual_seed(seed)
    B, S, Hq, Hkv, D = shape.B, shape.S, shape.Hq, shape.Hkv, shape.D
    q = _randn_bf16((B, S, Hq, D), g)
    k = _randn_bf16((B, S, Hkv, D), g)
    v = _randn_bf16((B, S, Hkv, D), g)
    do = _randn_bf16((B, S, Hq, D), g)
    return tuple(_store(t, shape.layout) for t in (q, k, v, do))


def exchange_input(B, S, H, D, layout="bshd", seed=DEFAULT_SEED):
    """One bf16 tensor ~N(0,1), logical [B,S,H,D], stored in `layout` order."""
    g = torch.Generator().manual_seed(seed)
    return _store(_randn_bf16((B, S, H, D), g), layout)
