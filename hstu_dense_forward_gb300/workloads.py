"""Seeded synthetic inputs for the HSTU forward (shared by tests, smoke and bench).

Data generation only: shapes, lengths, value distributions and seeds. Nothing
here computes any part of the operator.

Recipe (one torch.Generator on the CPU, drawn in this fixed order): sequence
lengths -> num_context -> num_targets -> q -> k -> v -> rab. Lengths are
uniform integers in [lo, hi]; values are normal (randn * sigma) or uniform
(2*rand - 1) in float32, then cast to the workload dtype. The same CPU tensors
feed the GPU run (after .cuda()) and the fp64 oracle.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field, replace
from typing import Optional

import torch

DTYPES = {"fp32": torch.float32, "fp16": torch.float16, "bf16": torch.bfloat16}


@dataclass(frozen=True)
class Workload:
    name: str
    dtype: str                    # "fp32" | "fp16" | "bf16"
    batch: int
    num_heads_q: int
    num_heads_kv: int
    head_dim: int
    max_seqlen: int
    len_lo: int = 0               # lengths ~ U[len_lo, len_hi] unless fixed_offsets is set
    len_hi: int = 0
    fixed_offsets: Optional[tuple] = None
    causal: bool = True
    context_range: Optional[tuple] = None   # num_context ~ U[lo, hi]
    target_range: Optional[tuple] = None    # num_targets ~ U[lo, hi]
    target_group_size: int = 0
    dist: str = "normal"          # "normal" (randn*sigma) | "uniform" (U(-1, 1))
    sigma: float = 1.0
    rab: bool = False
    rab_sigma: float = 0.1
    seed: int = 0
    alpha: Optional[float] = None        # default 1/sqrt(head_dim)
    silu_scale: Optional[float] = None   # default 1/max_seqlen
    index_dtype: torch.dtype = torch.int64

    @property
    def torch_dtype(self) -> torch.dtype:
        return DTYPES[self.dtype]

    @property
    def alpha_value(self) -> float:
        return self.alpha if self.alpha is not None else 1.0 / math.sqrt(self.head_dim)

    @property
    def silu_scale_value(self) -> float:
        return self.silu_scale if self.silu_scale is not None else 1.0 / self.max_seqlen


# The five workloads of the benchmark spec, in order: a tiny fp32 case, the bf16 causal jagged
# throughput case, the rab (HBM) case, the fp16 GQA context/target case and the
# long-sequence d=256 case.
WORKLOADS = {
    "fp32_tiny": Workload(
        name="fp32_tiny", dtype="fp32", batch=2, num_heads_q=2, num_heads_kv=2, head_dim=32,
        max_seqlen=24, fixed_offsets=(0, 16, 40), causal=False, sigma=1.0, seed=0),
    "bf16_causal_b32_s2048_h4_d128": Workload(
        name="bf16_causal_b32_s2048_h4_d128", dtype="bf16", batch=32, num_heads_q=4,
        num_heads_kv=4, head_dim=128, max_seqlen=2048, len_lo=256, len_hi=2048, causal=True,
        sigma=0.5, seed=1),
    "bf16_rab_b16_s1024_h8_d64": Workload(
        name="bf16_rab_b16_s1024_h8_d64", dtype="bf16", batch=16, num_heads_q=8, num_heads_kv=8,
        head_dim=64, max_seqlen=1024, len_lo=512, len_hi=1024, causal=True, sigma=0.25,
        rab=True, rab_sigma=0.1, seed=2),
    "fp16_gqa8x2_targets_b8_s4096_d128": Workload(
        name="fp16_gqa8x2_targets_b8_s4096_d128", dtype="fp16", batch=8, num_heads_q=8,
        num_heads_kv=2, head_dim=128, max_seqlen=4096, len_lo=1024, len_hi=4096, causal=True,
        context_range=(0, 32), target_range=(16, 256), target_group_size=16, sigma=0.3, seed=3),
    "bf16_long_b4_s8192_h4_d256": Workload(
        name="bf16_long_b4_s8192_h4_d256", dtype="bf16", batch=4, num_heads_q=4, num_heads_kv=4,
        head_dim=256, max_seqlen=8192, len_lo=8192, len_hi=8192, causal=False,
        dist="uniform", seed=4),
}

BENCH_WORKLOAD = "bf16_causal_b32_s2048_h4_d128"


def scaled(w: Workload, *, batch=None, max_seqlen=None, len_lo=None, len_hi=None, **kw) -> Workload:
    """A smaller (or otherwise modified) copy of a workload with the same structure."""
    ch = dict(kw)
    if batch is not None:
        ch["batch"] = batch
    if max_seqlen is not None:
        ch["max_seqlen"] = max_seqlen
    if len_lo is not None:
        ch["len_lo"] = len_lo
    if len_hi is not None:
        ch["len_hi"] = len_hi
    return replace(w, **ch)


def generate(w: Workload) -> dict:
    """CPU tensors of one workload instance: q, k, v, seq_offsets, num_context,
    num_targets, rab (None where absent) plus the scalar arguments."""
    g = torch.Generator().manual_seed(w.seed)
    if w.fixed_offsets is not None:
        offsets = torch.tensor(w.fixed_offsets, dtype=torch.int64)
        lengths = offsets[1:] - offsets[:-1]
    else:
        lengths = torch.randint(w.len_lo, w.len_hi + 1, (w.batch,), generator=g, dtype=torch.int64)
        offsets = torch.zeros(w.batch + 1, dtype=torch.int64)
        offsets[1:] = torch.cumsum(lengths, 0)
    num_context = None
    if w.context_range is not None:
        num_context = torch.randint(w.context_range[0], w.context_range[1] + 1, (w.batch,),
                                    generator=g, dtype=torch.int64)
    num_targets = None
    if w.target_range is not None:
        num_targets = torch.randint(w.target_range[0], w.target_range[1] + 1, (w.batch,),
                                    generator=g, dtype=torch.int64)
    T = int(offsets[-1])
    dt = w.torch_dtype

    def draw(*shape):
        if w.dist == "uniform":
            x = torch.rand(*shape, generator=g, dtype=torch.float32) * 2.0 - 1.0
        else:
            x = torch.randn(*shape, generator=g, dtype=torch.float32) * w.sigma
        return x.to(dt)

    q = draw(T, w.num_heads_q, w.head_dim)
    k = draw(T, w.num_heads_kv, w.head_dim)
    v = draw(T, w.num_heads_kv, w.head_dim)
    rab = None
    if w.rab:
        S = w.max_seqlen
        rab = (torch.randn(w.batch, w.num_heads_q, S, S, generator=g, dtype=torch.float32)
               * w.rab_sigma).to(dt)
    idx = w.index_dtype
    return dict(q=q, k=k, v=v, seq_offsets=offsets.to(idx),
                num_context=None if num_context is None else num_context.to(idx),
                num_targets=None if num_targets is None else num_targets.to(idx), rab=rab,
                max_seqlen=w.max_seqlen, causal=w.causal, target_group_size=w.target_group_size,
                alpha=w.alpha_value, silu_scale=w.silu_scale_value)


def to_device(inputs: dict, device) -> dict:
    """Copy the tensor entries of generate()'s result to a device."""
    return {k: (v.to(device) if isinstance(v, torch.Tensor) else v) for k, v in inputs.items()}
