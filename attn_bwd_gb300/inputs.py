"""Seeded synthetic inputs for attention backward workloads.

This module only draws random numbers and names workload shapes.  It holds
none of the attention arithmetic, so that the fp64 oracle (``oracle/``) and
the CUDA path can both consume exactly the same tensors without sharing any
of the method's code.

Distributions follow the workloads the pages time:
  * i.i.d. N(0, 1) for Q, K, V, dO (the MI250x sweep in "[Issue]: Backward
    performance", ROCm/flash-attention #44, and the Llama-3 shaped sweep in
    "[Kernel] Flash attention 2", Liger-Kernel #275, "Benchmarking");
  * i.i.d. Uniform[0, 1) for Q, K, V, dO with softmax scale 1.1 (the repro in
    "Extra transposes cause 8x speedup for sequence-parallel Flash Attention
    backward", triton #1806, "Minimal Repro").
"""
from __future__ import annotations

import dataclasses
import math

import torch

DTYPES = {"f16": torch.float16, "bf16": torch.bfloat16}


@dataclasses.dataclass(frozen=True)
class Shape:
    """One attention problem: Q/O/dO are [B, Hq, Nq, d], K/V are [B, Hkv, Nkv, d]."""

    B: int
    Hq: int
    Hkv: int
    Nq: int
    Nkv: int
    d: int
    causal: int                  # 0 / False: none, 1 / True: top-left, 2: bottom-right
    dtype: str = "bf16"          # "f16" or "bf16"
    dist: str = "normal"         # "normal" -> N(0,1), "uniform" -> U[0,1)
    scale: float | None = None   # None -> 1/sqrt(d)

    @property
    def softmax_scale(self) -> float:
        return self.scale if self.scale is not None else 1.0 / math.sqrt(self.d)

    @property
    def torch_dtype(self) -> torch.dtype:
        return DTYPES[self.dtype]

    def name(self) -> str:
        c = {0: "full", 1: "causal", 2: "causalbr"}[int(self.causal)]
        return (f"B{self.B}_Hq{self.Hq}_Hkv{self.Hkv}_Nq{self.Nq}_Nkv{self.Nkv}"
                f"_d{self.d}_{self.dtype}_{self.dist}_{c}")


def draw(shape: Shape, seed: int, device: str | torch.device = "cpu"):
    """Return (q, k, v, do) in the shape's 16-bit dtype, drawn from one seeded generator.

    The draws happen in fp32 and are rounded once to the storage dtype; both
    the oracle (after widening to fp64) and the CUDA path read these exact
    16-bit values.
    """
    gen = torch.Generator(device=device)
    gen.manual_seed(seed)
    sizes = [
        (shape.B, shape.Hq, shape.Nq, shape.d),
        (shape.B, shape.Hkv, shape.Nkv, shape.d),
        (shape.B, shape.Hkv, shape.Nkv, shape.d),
        (shape.B, shape.Hq, shape.Nq, shape.d),
    ]
    out = []
    for sz in sizes:
        if shape.dist == "normal":
            t = torch.randn(sz, generator=gen, device=device, dtype=torch.float32)
        elif shape.dist == "uniform":
            t = torch.rand(sz, generator=gen, device=device, dtype=torch.float32)
        else:
            raise ValueError(f"unknown distribution {shape.dist!r}")
        out.append(t.to(shape.torch_dtype))
    return tuple(out)


# --- the five workloads (shapes and distributions only) ----------------------

def tiny_mha() -> list[Shape]:
    """B=1, H=2, N=128, d=64, fp16, N(0,1), non-causal."""
    return [Shape(1, 2, 2, 128, 128, 64, False, "f16")]


def ragged() -> list[Shape]:
    """B=2, H=4, d=64, fp16, N in {1,17,31,33,100}, causal and not."""
    return [Shape(2, 4, 4, n, n, 64, c, "f16")
            for n in (1, 17, 31, 33, 100) for c in (False, True)]


def mid_sweep() -> list[Shape]:
    """B=16, H=16, d in {64,128}, N in {256,576,784}, fp16 and bf16, non-causal."""
    return [Shape(16, 16, 16, n, n, d, False, dt)
            for dt in ("f16", "bf16") for d in (64, 128) for n in (256, 576, 784)]


def long_uniform() -> list[Shape]:
    """B=2, H=16, N=2048, d=128, fp16, U[0,1), scale 1.1, non-causal."""
    return [Shape(2, 16, 16, 2048, 2048, 128, False, "f16", "uniform", 1.1)]


def llama_gqa(n: int) -> Shape:
    """B=4, Hq=32, Hkv=8, d=128, bf16, causal, Nq=Nkv=n (n swept 2^5..2^14)."""
    return Shape(4, 32, 8, n, n, 128, True, "bf16")


LLAMA_SWEEP = [2 ** p for p in range(5, 15)]
HEADLINE = llama_gqa(8192)


@dataclasses.dataclass(frozen=True)
class Packed:
    """A packed batch of sequences of different lengths: Q/O/dO are [Hq, total_q, d],
    K/V are [Hkv, total_k, d]; sequence b owns rows cu_q[b]..cu_q[b+1] (and cu_k) of every head."""

    lens_q: tuple
    lens_k: tuple
    Hq: int
    Hkv: int
    d: int
    causal: int
    dtype: str = "bf16"

    @property
    def cu_q(self):
        return [0] + [int(x) for x in torch.tensor(self.lens_q).cumsum(0).tolist()]

    @property
    def cu_k(self):
        return [0] + [int(x) for x in torch.tensor(self.lens_k).cumsum(0).tolist()]

    @property
    def softmax_scale(self) -> float:
        return 1.0 / math.sqrt(self.d)

    @property
    def torch_dtype(self) -> torch.dtype:
        return DTYPES[self.dtype]

    def name(self) -> str:
        c = {0: "full", 1: "causal", 2: "causalbr"}[int(self.causal)]
        return (f"q{'-'.join(map(str, self.lens_q))}_k{'-'.join(map(str, self.lens_k))}"
                f"_Hq{self.Hq}_Hkv{self.Hkv}_d{self.d}_{self.dtype}_{c}")


def draw_packed(pk: Packed, seed: int, device: str | torch.device = "cpu"):
    """(q, k, v, do) of a packed batch, N(0,1) drawn in fp32 from one seeded generator, rounded once."""
    gen = torch.Generator(device=device)
    gen.manual_seed(seed)
    tq, tk = sum(pk.lens_q), sum(pk.lens_k)
    sizes = [(pk.Hq, tq, pk.d), (pk.Hkv, tk, pk.d), (pk.Hkv, tk, pk.d), (pk.Hq, tq, pk.d)]
    return tuple(torch.randn(sz, generator=gen, device=device, dtype=torch.float32).to(pk.torch_dtype)
                 for sz in sizes)


def packed_mix():
    """Length mixes for packed-batch parity: single rows, empty sequences, ragged tails past
    one and two tiles, Nq < Nkv and Nq > Nkv within one batch, both head dims."""
    out = []
    for c in (0, 1, 2):
        out.append(Packed((1, 130, 0, 257, 64), (1, 130, 5, 257, 64), 4, 2, 128, c, "bf16"))
        out.append(Packed((77, 300, 16), (200, 130, 16), 2, 1, 64, c, "f16"))
    out.append(Packed((50, 20, 129), (0, 33, 129), 2, 2, 128, 0, "bf16"))   # a sequence with no keys
    out.append(Packed((33, 190, 1), (65, 140, 7), 4, 1, 80, 2, "bf16"))     # head dim 80
    return out
