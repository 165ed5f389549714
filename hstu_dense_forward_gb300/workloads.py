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

DTYPES = {"fp32": torch.float32, "fp16": torch.float16, "bf16": torch.bfloat16,
          "fp8": torch.float8_e4m3fn}


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


# The five configurations, in order: a tiny fp32 case, the bf16 causal jagged
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
    # the causal workload with FP8 E4M3 inputs (feature table, "FP8 quantization: cast")
    "fp8_causal_b32_s2048_h4_d128": Workload(
        name="fp8_causal_b32_s2048_h4_d128", dtype="fp8", batch=32, num_heads_q=4,
        num_heads_kv=4, head_dim=128, max_seqlen=2048, len_lo=256, len_hi=2048, causal=True,
        sigma=0.5, seed=1),
    # head dim 512 (Inputs and Outputs table: v's D up to 512), causal jagged
    "bf16_causal_b8_s2048_h4_d512": Workload(
        name="bf16_causal_b8_s2048_h4_d512", dtype="bf16", batch=8, num_heads_q=4,
        num_heads_kv=4, head_dim=512, max_seqlen=2048, len_lo=512, len_hi=2048, causal=True,
        sigma=0.5, seed=6),
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


# --------------------------------------------------------------------------- key side
@dataclass(frozen=True)
class KVWorkload:
    """Queries that are the newest tokens of longer sequences whose history sits in a paged
    KV cache (Inputs and Outputs table: seq_offsets_q / seq_offsets_k, kv_cache,
    page_offsets, page_ids, last_page_len; feature table, "Page")."""
    name: str
    dtype: str
    batch: int
    num_heads_q: int
    num_heads_kv: int
    head_dim: int
    hist_range: tuple             # cached history rows ~ U[lo, hi]
    new_range: tuple              # new k/v rows ~ U[lo, hi]
    page_size: int = 128          # 0: no cache (the history rows are passed as new rows)
    query_range: Optional[tuple] = None  # None: the queries are the new rows; else
                                         # Lq ~ U[lo, hi], clipped to the keys
    spare_pages: int = 8          # cache pages no sequence uses
    causal: bool = True
    context_range: Optional[tuple] = None
    targets_are_queries: bool = False    # num_targets = Lq (the new tokens are the targets)
    target_group_size: int = 0
    sigma: float = 1.0
    rab: bool = False
    rab_sigma: float = 0.1
    seed: int = 0
    alpha: Optional[float] = None        # default 1/sqrt(head_dim)
    index_dtype: torch.dtype = torch.int64

    @property
    def max_seqlen(self) -> int:    # bound on query rows
        hi = self.query_range[1] if self.query_range else self.new_range[1]
        return max(8, -(-hi // 8) * 8)

    @property
    def max_seqlen_k(self) -> int:  # bound on keys (a multiple of 8: the rab row stride)
        return -(-(self.hist_range[1] + self.new_range[1]) // 8) * 8

    @property
    def alpha_value(self) -> float:
        return self.alpha if self.alpha is not None else 1.0 / math.sqrt(self.head_dim)

    @property
    def silu_scale_value(self) -> float:
        return 1.0 / self.max_seqlen_k


KV_WORKLOADS = {
    # ranking with a cached user history: the new tokens are the candidates (targets of
    # group size 1: each sees the history and itself)
    "bf16_paged_b128_hist1k_4k_h4_d128": KVWorkload(
        name="bf16_paged_b128_hist1k_4k_h4_d128", dtype="bf16", batch=128, num_heads_q=4,
        num_heads_kv=4, head_dim=128, hist_range=(1024, 4096), new_range=(32, 256),
        page_size=128, targets_are_queries=True, target_group_size=1, sigma=0.5, seed=5),
    # the same with an FP8 E4M3 cache and inputs (half the bytes per key)
    "fp8_paged_b128_hist1k_4k_h4_d128": KVWorkload(
        name="fp8_paged_b128_hist1k_4k_h4_d128", dtype="fp8", batch=128, num_heads_q=4,
        num_heads_kv=4, head_dim=128, hist_range=(1024, 4096), new_range=(32, 256),
        page_size=128, targets_are_queries=True, target_group_size=1, sigma=0.5, seed=5),
}


def generate_kv(w: KVWorkload) -> dict:
    """CPU tensors of one key-side workload: q [Tq, Nq, D], k / v [Tk, Nk, D] (new rows),
    seq_offsets (queries), seq_offsets_k, kv_cache [num_pages, 2, page_size, Nk, D] with
    page_offsets, page_ids (a random permutation of the pages), last_page_len, plus
    num_context / num_targets / rab and the scalars. Every cache row, used or not, holds
    finite values. With page_size 0 the history rows are prepended to the new rows instead
    (the same keys passed contiguously)."""
    g = torch.Generator().manual_seed(w.seed)
    B = w.batch
    hist = torch.randint(w.hist_range[0], w.hist_range[1] + 1, (B,), generator=g)
    lnew = torch.randint(w.new_range[0], w.new_range[1] + 1, (B,), generator=g)
    lk = hist + lnew
    if w.query_range is None:
        lq = lnew.clone()
    else:
        lq = torch.minimum(torch.randint(w.query_range[0], w.query_range[1] + 1, (B,),
                                         generator=g), lk)
    num_context = None
    if w.context_range is not None:
        num_context = torch.randint(w.context_range[0], w.context_range[1] + 1, (B,),
                                    generator=g)
    num_targets = lq.clone() if w.targets_are_queries else None
    dt = DTYPES[w.dtype]

    def draw(*shape):
        return (torch.randn(*shape, generator=g, dtype=torch.float32) * w.sigma).to(dt)

    def offsets(lengths):
        o = torch.zeros(B + 1, dtype=torch.int64)
        o[1:] = torch.cumsum(lengths, 0)
        return o

    Nq, Nk, D = w.num_heads_q, w.num_heads_kv, w.head_dim
    q = draw(int(lq.sum()), Nq, D)
    out = dict(q=q, seq_offsets=offsets(lq), num_context=num_context, num_targets=num_targets,
               causal=w.causal, target_group_size=w.target_group_size, alpha=w.alpha_value,
               silu_scale=w.silu_scale_value, max_seqlen=w.max_seqlen,
               max_seqlen_k=w.max_seqlen_k)
    if w.page_size:
        ps = w.page_size
        npages = (hist + ps - 1) // ps
        num_pages = int(npages.sum()) + w.spare_pages
        cache = draw(num_pages, 2, ps, Nk, D)
        ids = torch.randperm(num_pages, generator=g)[:int(npages.sum())]
        last = torch.where(npages > 0, hist - (npages - 1) * ps, torch.ones_like(hist))
        out.update(k=draw(int(lnew.sum()), Nk, D), v=draw(int(lnew.sum()), Nk, D),
                   seq_offsets_k=offsets(lnew), kv_cache=cache, page_offsets=offsets(npages),
                   page_ids=ids, last_page_len=last)
    else:
        out.update(k=draw(int(lk.sum()), Nk, D), v=draw(int(lk.sum()), Nk, D),
                   seq_offsets_k=offsets(lk), kv_cache=None, page_offsets=None, page_ids=None,
                   last_page_len=None)
    rab = None
    if w.rab:
        S = w.max_seqlen_k
        rab = (torch.randn(B, Nq, S, S, generator=g, dtype=torch.float32) * w.rab_sigma).to(dt)
    out["rab"] = rab
    idx = w.index_dtype
    for key in ("seq_offsets", "seq_offsets_k", "page_offsets", "page_ids", "last_page_len",
                "num_context", "num_targets"):
        if out.get(key) is not None:
            out[key] = out[key].to(idx)
    out["history"] = hist  # cached rows per sequence (for checks; not an operator input)
    return out
