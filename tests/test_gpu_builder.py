"""The work-list builder against offsets written on the stream just before a call.

The builder may start before the kernel ahead of it in the stream has finished (programmatic
dependent launch), and that kernel's writes are visible to it only after its grid-dependency
wait. Here a torch kernel writes seq_offsets immediately before every call, alternating two
layouts of the same rows with different query-tile counts, and every output is compared
with the fp64 oracle on the offsets that the stream order gives that call.
"""
import numpy as np
import pytest
import torch

import oracle
from hstu_dense_forward_gb300 import HstuFwdPlan, _abi, hstu_fwd

pytestmark = pytest.mark.gpu

# Two layouts of 1200 rows in six sequences: 6 + 1 + 2 + 1 + 1 + 1 and 1 + 2 + 3 + 5 + 0 + 1
# query tiles of 128 rows.
LAYOUTS = [[0, 700, 701, 900, 1000, 1100, 1200], [0, 64, 300, 600, 1199, 1199, 1200]]
T, H, D, MAX_SEQLEN = 1200, 2, 64, 700
ALPHA, SILU_SCALE = 0.125, 1.0 / MAX_SEQLEN


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16])
def test_offsets_rewritten_before_each_call(cuda_device, dtype):
    g = torch.Generator().manual_seed(11)
    q, k, v = [torch.randn(T, H, D, generator=g).to(dtype) for _ in range(3)]
    refs = [oracle.hstu_fwd(q.double(), k.double(), v.double(), torch.tensor(o, dtype=torch.int64),
                            mask_type=oracle.MASK_CAUSAL, alpha=ALPHA, silu_scale=SILU_SCALE,
                            max_seqlen=MAX_SEQLEN)
            for o in LAYOUTS]
    qd, kd, vd = q.to(cuda_device), k.to(cuda_device), v.to(cuda_device)
    staged = [torch.tensor(o, dtype=torch.int64, device=cuda_device) for o in LAYOUTS]
    so = staged[0].clone()
    outs = []
    for it in range(8):
        torch.add(staged[(it + 1) % 2], 0, out=so)  # a kernel writes the offsets
        outs.append(hstu_fwd(qd, kd, vd, so, max_seqlen=MAX_SEQLEN, causal=True, alpha=ALPHA,
                             silu_scale=SILU_SCALE))
    torch.cuda.synchronize()
    tol = 2e-2 if dtype == torch.bfloat16 else 1e-2
    for it, o in enumerate(outs):
        ref = refs[(it + 1) % 2]
        err = np.max(np.abs(o.double().cpu().numpy() - ref)) / np.max(np.abs(ref))
        assert err <= tol, f"call {it}: rel err {err:.3e}"


def test_offsets_turning_invalid_and_valid_before_calls(cuda_device):
    """A kernel writes offsets that run past the rows just before a call: that call reports
    HSTU_DEVERR_OFFSETS and writes nothing. Valid offsets written just before the next call
    give a correct output and no error."""
    plan = HstuFwdPlan(dtype=torch.bfloat16, batch=6, num_heads_q=H, num_heads_kv=H,
                       head_dim=D, max_seqlen=MAX_SEQLEN, index_is_int64=True, causal=True,
                       target_group_size=0, has_rab=False, has_num_context=False,
                       has_num_targets=False)
    g = torch.Generator().manual_seed(12)
    q = torch.randn(T, H, D, generator=g).to(torch.bfloat16)
    qd = q.to(cuda_device)
    good = torch.tensor(LAYOUTS[1], dtype=torch.int64, device=cuda_device)
    bad = torch.tensor([0, 64, 300, 600, 1199, 1199, 1300], dtype=torch.int64,
                       device=cuda_device)  # 1300 > T
    so = good.clone()
    out = torch.empty_like(qd)
    plan.run(qd, qd, qd, so, out, alpha=ALPHA, silu_scale=SILU_SCALE)
    assert plan.get_error() == _abi.HSTU_DEVERR_NONE
    out.fill_(7.0)
    torch.add(bad, 0, out=so)
    plan.run(qd, qd, qd, so, out, alpha=ALPHA, silu_scale=SILU_SCALE)
    assert plan.get_error() == _abi.HSTU_DEVERR_OFFSETS
    assert bool(torch.all(out == 7.0))
    torch.add(good, 0, out=so)
    plan.run(qd, qd, qd, so, out, alpha=ALPHA, silu_scale=SILU_SCALE)
    assert plan.get_error() == _abi.HSTU_DEVERR_NONE
    ref = oracle.hstu_fwd(q.double(), q.double(), q.double(),
                          torch.tensor(LAYOUTS[1], dtype=torch.int64),
                          mask_type=oracle.MASK_CAUSAL, alpha=ALPHA, silu_scale=SILU_SCALE,
                          max_seqlen=MAX_SEQLEN)
    err = np.max(np.abs(out.double().cpu().numpy() - ref)) / np.max(np.abs(ref))
    assert err <= 2e-2
    plan.close()
