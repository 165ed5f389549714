"""The largest inputs the Inputs and Outputs table allows (q: B in [1, 2048], S in [1, 20480],
N_q in [1, 16]), through the C ABI, on sampled rows against the fp64 oracle: one sequence of
20480 tokens with 16 query heads, and 2048 short sequences."""
import numpy as np
import pytest
import torch

import oracle
from hstu_dense_forward_gb300 import hstu_fwd
from hstu_dense_forward_gb300 import workloads as W

pytestmark = pytest.mark.gpu

TOL = {"fp32": 1e-5, "bf16": 2e-2, "fp16": 1e-2}


def _sampled(inp, got, w, rows, causal=True):
    so = inp["seq_offsets"]
    ref = oracle.hstu_fwd_rows(inp["q"], inp["k"], inp["v"], so, np.array(rows),
                               num_context=inp["num_context"], num_targets=inp["num_targets"],
                               mask_type=oracle.MASK_CAUSAL if causal else oracle.MASK_NONE,
                               target_group_size=w.target_group_size, alpha=w.alpha_value,
                               silu_scale=w.silu_scale_value, max_seqlen=w.max_seqlen,
                               nthreads=16)
    sel = torch.stack([got[int(so[b]) + i, h] for b, h, i in rows]).double().cpu().numpy()
    return float(np.abs(sel - ref).max() / np.abs(ref).max())


@pytest.mark.parametrize("dtype,heads", [("bf16", (16, 16)), ("fp16", (16, 2)), ("fp32", (16, 4))])
def test_longest_sequence_all_heads(cuda_device, dtype, heads):
    w = W.Workload(name="max_s", dtype=dtype, batch=1, num_heads_q=heads[0],
                   num_heads_kv=heads[1], head_dim=128, max_seqlen=20480,
                   fixed_offsets=(0, 20480), causal=True, context_range=(0, 256),
                   target_range=(0, 512), target_group_size=3, sigma=0.5, seed=91)
    inp = W.generate(w)
    d = W.to_device(inp, cuda_device)
    got = hstu_fwd(d["q"], d["k"], d["v"], d["seq_offsets"], max_seqlen=w.max_seqlen,
                   num_context=d["num_context"], num_targets=d["num_targets"],
                   target_group_size=3, alpha=w.alpha_value, silu_scale=w.silu_scale_value)
    torch.cuda.synchronize()
    g = np.random.default_rng(1)
    rows = [(0, int(g.integers(0, heads[0])), int(i))
            for i in np.concatenate([[0, 1, 127, 128, 20479], g.integers(0, 20480, 27)])]
    assert _sampled(inp, got, w, rows) <= TOL[dtype]
    assert torch.isfinite(got.float()).all()


@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
def test_largest_batch_of_short_sequences(cuda_device, dtype):
    w = W.Workload(name="max_b", dtype=dtype, batch=2048, num_heads_q=4, num_heads_kv=4,
                   head_dim=64, max_seqlen=16, len_lo=0, len_hi=16, causal=True, sigma=0.5,
                   seed=92)
    inp = W.generate(w)
    d = W.to_device(inp, cuda_device)
    got = hstu_fwd(d["q"], d["k"], d["v"], d["seq_offsets"], max_seqlen=16,
                   alpha=w.alpha_value, silu_scale=w.silu_scale_value)
    torch.cuda.synchronize()
    so = inp["seq_offsets"]
    g = np.random.default_rng(2)
    rows = []
    for b in list(g.integers(0, 2048, 60)) + [0, 2047]:
        L = int(so[b + 1] - so[b])
        if L:
            rows.append((int(b), int(g.integers(0, 4)), int(g.integers(0, L))))
    assert _sampled(inp, got, w, rows) <= TOL[dtype]


@pytest.mark.parametrize("head_dim,heads", [(512, (16, 4)), (48, (16, 16))])
def test_longest_sequence_other_head_dims(cuda_device, head_dim, heads):
    """The longest sequence with 16 query heads at head dim 512 (two O halves per tile) and
    at a padded head dim (48 on the 64 kernel), context and targets at their limits."""
    w = W.Workload(name="max_d", dtype="bf16", batch=1, num_heads_q=heads[0],
                   num_heads_kv=heads[1], head_dim=head_dim, max_seqlen=20480,
                   fixed_offsets=(0, 20480), causal=True, context_range=(256, 256),
                   target_range=(512, 512), target_group_size=3, sigma=0.5, seed=93)
    inp = W.generate(w)
    d = W.to_device(inp, cuda_device)
    got = hstu_fwd(d["q"], d["k"], d["v"], d["seq_offsets"], max_seqlen=w.max_seqlen,
                   num_context=d["num_context"], num_targets=d["num_targets"],
                   target_group_size=3, alpha=w.alpha_value, silu_scale=w.silu_scale_value)
    torch.cuda.synchronize()
    g = np.random.default_rng(3)
    rows = [(0, int(g.integers(0, heads[0])), int(i))
            for i in np.concatenate([[0, 255, 256, 19967, 19968, 20479], g.integers(0, 20480, 20)])]
    assert _sampled(inp, got, w, rows) <= TOL["bf16"]
    assert torch.isfinite(got.float()).all()
