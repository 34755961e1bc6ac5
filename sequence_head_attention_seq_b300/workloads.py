"""Seeded synthetic inputs shaped like the pages' workloads.

This module only draws random numbers and names shapes.  It holds none of
the attention or relayout arithmetic, so the CUDA path and the oracle can both
take their inputs from it without sharing any of the method.

Layout of a drawn tensor: the sequence-shard layout the pages start from,
``[N][b][s/N][h][d]`` (shard r = sequence rows [r*s/N, (r+1)*s/N) of every
head, as in the transformers "Support deepspeed sequence parallel" PR's data
collator and the long-context-attention issue "关于数据分割和合并").  Values
are N(0, 1) * scale drawn in fp32 and rounded to bf16.

Seeds: ``1000 * index + tensor_id`` with tensor_id q=0, k=1, v=2, dout=3 and
key lengths from a CPU generator seeded ``1000 * index + 4``.
"""
from __future__ import annotations

import dataclasses

import torch

TENSOR_IDS = {"q": 0, "k": 1, "v": 2, "dout": 3, "key_len": 4}


@dataclasses.dataclass(frozen=True)
class Workload:
    """One synthetic problem: full sequence s, h heads in total, N sequence shards."""
    name: str
    index: int          # 1-based position in the workload list (seed base)
    b: int
    h: int
    d: int
    s: int
    N: int              # sequence-parallel degree (shards in, head groups out)
    causal: bool
    scale: float        # q/k/v standard deviation; dout is always N(0, 1)
    key_len_range: tuple | None = None   # inclusive [lo, hi] of valid keys per batch row
    split_q: int = 1    # >1: the query rows are also evaluated as this many shards

    @property
    def s_local(self) -> int:
        return self.s // self.N

    @property
    def h_local(self) -> int:
        return self.h // self.N

    def shard_shape(self) -> tuple:
        return (self.N, self.b, self.s_local, self.h, self.d)

    def group_shape(self) -> tuple:
        return (self.N, self.b, self.s, self.h_local, self.d)

    def seed(self, tensor: str) -> int:
        return 1000 * self.index + TENSOR_IDS[tensor]


WORKLOADS = {
    w.name: w
    for w in (
        # two 64-row query shards of one 128-token sequence, each against the full K/V
        Workload("tiny", 1, b=1, h=2, d=64, s=128, N=2, causal=True, scale=1.0, split_q=2),
        # LLaMA-7B-shaped layer, 4 sequence shards -> 4 head groups of 8 heads
        Workload("llama7b", 2, b=1, h=32, d=128, s=4096, N=4, causal=True, scale=1.0),
        # LLaMA-70B-shaped long context (hidden 8192), 8 shards -> 8 groups of 8 heads
        Workload("llama70b", 3, b=1, h=64, d=128, s=32768, N=8, causal=True, scale=0.5),
        # padded batch, no sequence split, right-padded keys per batch row
        Workload("padded", 4, b=8, h=16, d=64, s=2048, N=1, causal=False, scale=1.0,
                 key_len_range=(1024, 2048)),
        # 131072 tokens after the Ulysses split: 8 groups of 8 local heads (64 in total)
        Workload("ulysses131k", 5, b=1, h=64, d=128, s=131072, N=8, causal=True, scale=0.5),
    )
}

ORDER = ["tiny", "llama7b", "llama70b", "padded", "ulysses131k"]


def randn_bf16(shape, seed: int, scale: float = 1.0, device="cpu") -> torch.Tensor:
    """N(0, 1) * scale, drawn in fp32 by torch's generator on `device`, rounded to bf16."""
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    x = torch.randn(tuple(shape), generator=g, device=device, dtype=torch.float32)
    if scale != 1.0:
        x.mul_(scale)
    return x.to(torch.bfloat16)


def key_lengths(b: int, lo: int, hi: int, seed: int) -> torch.Tensor:
    """b integers uniform in [lo, hi] (inclusive), int32, from a CPU generator."""
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    return torch.randint(lo, hi + 1, (b,), generator=g, dtype=torch.int32)


def make_inputs(w: Workload, device="cpu", with_dout: bool = True) -> dict:
    """q, k, v (and dout) in the sequence-shard layout; key_len when the workload pads."""
    out = {}
    for name in ("q", "k", "v"):
        out[name] = randn_bf16(w.shard_shape(), w.seed(name), w.scale, device)
    if with_dout:
        out["dout"] = randn_bf16(w.shard_shape(), w.seed("dout"), 1.0, device)
    if w.key_len_range is not None:
        lo, hi = w.key_len_range
        out["key_len"] = key_lengths(w.b, lo, hi, w.seed("key_len"))
    else:
        out["key_len"] = None
    return out
