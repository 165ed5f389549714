"""The allocation-free entry point (hstu_fwd_run_noalloc) against the plan-based one.

Some callers cannot call cudaMalloc at all (a plugin that is only handed its input
and output buffers, a runtime whose pool already holds all device memory, a latency
path that must not take cudaMalloc's implicit synchronisation); for them the library
keeps its work list in a fixed device array. This file is collected last so that a
failure here never hides the other GPU tests."""
import ctypes

import numpy as np
import pytest
import torch

from hstu_dense_forward_gb300 import _abi, hstu_fwd, hstu_fwd_noalloc
from hstu_dense_forward_gb300 import workloads as W

pytestmark = pytest.mark.gpu

TOL = {"bf16": 2e-2, "fp16": 1e-2, "fp32": 1e-5}


def _run_both(w, dev, layout="jagged", rab_bcast=False):
    """The plan-based call and the allocation-free call on the same inputs; returns the
    largest difference relative to max |plan output|."""
    inp = W.to_device(W.generate(w), dev)
    q, k, v, so, rab = inp["q"], inp["k"], inp["v"], inp["seq_offsets"], inp["rab"]
    if rab_bcast:
        rab = rab[:, :1].contiguous()  # [B, 1, S, S]: one bias plane for every head
    if layout == "normal":  # every sequence has max_seqlen tokens: [B, S, N, D]
        B, S = w.batch, w.max_seqlen
        q, k, v = (t.view(B, S, *t.shape[1:]) for t in (q, k, v))
        so = None
    kw = dict(max_seqlen=w.max_seqlen, rab=rab, num_context=inp["num_context"],
              num_targets=inp["num_targets"], causal=w.causal,
              target_group_size=w.target_group_size, alpha=w.alpha_value,
              silu_scale=w.silu_scale_value, layout=layout)
    ref = hstu_fwd(q, k, v, so, **kw)
    out = torch.full_like(q, float("nan"))
    hstu_fwd_noalloc(q, k, v, so, out, **kw)
    torch.cuda.synchronize()
    T = int(inp["seq_offsets"][-1])
    r = ref.reshape(-1, *ref.shape[-2:])[:T].double().cpu().numpy()
    g = out.reshape(-1, *out.shape[-2:])[:T].double().cpu().numpy()
    return float(np.max(np.abs(g - r)) / np.max(np.abs(r)))


def test_noalloc_matches_plan_entry_point_on_two_calls_in_a_row(cuda_device):
    """Calls in a row (different workloads, so each one overwrites the previous one's work
    list in the shared array) all match the plan-based entry point: bf16 with context and
    targets, fp16 with rab, the fp32 CUDA-core path, the normal layout with a rab plane
    broadcast to every head, and head dim 512."""
    first = W.Workload(name="na1", dtype="bf16", batch=4, num_heads_q=4, num_heads_kv=2,
                       head_dim=128, max_seqlen=512, len_lo=100, len_hi=512, causal=True,
                       context_range=(0, 10), target_range=(0, 40), target_group_size=4,
                       sigma=0.5, seed=81)
    second = W.Workload(name="na2", dtype="fp16", batch=3, num_heads_q=2, num_heads_kv=2,
                        head_dim=64, max_seqlen=264, len_lo=60, len_hi=264, causal=True,
                        rab=True, rab_sigma=0.3, seed=82)
    third = W.WORKLOADS["fp32_tiny"]
    fourth = W.Workload(name="na4", dtype="bf16", batch=3, num_heads_q=4, num_heads_kv=4,
                        head_dim=64, max_seqlen=200, len_lo=200, len_hi=200, causal=True,
                        rab=True, rab_sigma=0.3, sigma=0.5, seed=84)
    fifth = W.Workload(name="na5", dtype="bf16", batch=2, num_heads_q=2, num_heads_kv=1,
                       head_dim=512, max_seqlen=300, len_lo=100, len_hi=300, causal=True,
                       seed=85)
    for w, layout, bcast in ((first, "jagged", False), (second, "jagged", False),
                             (third, "jagged", False), (fourth, "normal", True),
                             (fifth, "jagged", False)):
        err = _run_both(w, cuda_device, layout=layout, rab_bcast=bcast)
        assert np.isfinite(err) and err <= TOL[w.dtype], f"{w.name} ({layout}): {err:.3e}"


def test_noalloc_rejects_work_lists_beyond_the_static_array(cuda_device):
    d = _abi.Desc()
    for name, val in dict(dtype=_abi.HSTU_BF16, batch=1024, num_heads_q=1, num_heads_kv=1,
                          head_dim=64, max_seqlen=4096, index_is_int64=1,
                          mask_type=_abi.HSTU_MASK_CAUSAL).items():
        setattr(d, name, val)
    buf = torch.zeros(16, dtype=torch.int64, device=cuda_device)
    rc = _abi.lib().hstu_fwd_run_noalloc(ctypes.byref(d), buf.data_ptr(), buf.data_ptr(),
                                         buf.data_ptr(), buf.data_ptr(), None, None, None, 8,
                                         1.0, 1.0, buf.data_ptr(), None)
    assert rc == _abi.HSTU_ERR_UNSUPPORTED  # 1024 * 32 entries > 16384
