"""Back-to-back calls on one plan overlap on the GPU: the work-list build of a call runs
while the previous call's forward kernel finishes (programmatic dependent launch, two work
lists per plan). Calls with different sequence layouts that alternate between two output
buffers, issued without synchronisation, must leave exactly the results of the same calls
run one at a time: a late write of an earlier call, or a work list overwritten while in
use, would show up as a mismatch."""
from dataclasses import replace

import pytest
import torch

from hstu_dense_forward_gb300 import hstu_fwd
from hstu_dense_forward_gb300 import workloads as W

pytestmark = pytest.mark.gpu

# two layouts of the same 3000 tokens over 6 sequences (max_seqlen 1024)
LENS_A = (1000, 200, 700, 100, 600, 400)
LENS_B = (100, 900, 300, 1000, 250, 450)


def _offsets(lens):
    o = [0]
    for n in lens:
        o.append(o[-1] + n)
    return tuple(o)


def _call(d, out):
    hstu_fwd(d["q"], d["k"], d["v"], d["seq_offsets"], max_seqlen=d["max_seqlen"],
             rab=d["rab"], num_context=d["num_context"], num_targets=d["num_targets"],
             causal=d["causal"], target_group_size=d["target_group_size"], alpha=d["alpha"],
             silu_scale=d["silu_scale"], out=out)


@pytest.mark.parametrize("dtype,d,heads", [("bf16", 128, (4, 4)), ("fp16", 64, (8, 2)),
                                           ("bf16", 256, (2, 2)), ("fp32", 64, (2, 2))])
def test_back_to_back_calls_match_serial(cuda_device, dtype, d, heads):
    base = W.scaled(W.WORKLOADS["bf16_causal_b32_s2048_h4_d128"], batch=len(LENS_A),
                    max_seqlen=1024, dtype=dtype, head_dim=d, num_heads_q=heads[0],
                    num_heads_kv=heads[1])
    da = W.to_device(W.generate(replace(base, fixed_offsets=_offsets(LENS_A), seed=11)),
                     cuda_device)
    db = W.to_device(W.generate(replace(base, fixed_offsets=_offsets(LENS_B), seed=12)),
                     cuda_device)
    assert da["q"].shape == db["q"].shape
    out1 = torch.empty_like(da["q"])
    out2 = torch.empty_like(da["q"])
    _call(da, out1)
    torch.cuda.synchronize()
    ref_a = out1.clone()
    _call(db, out1)
    torch.cuda.synchronize()
    ref_b = out1.clone()
    assert not torch.equal(ref_a, ref_b)
    for _ in range(12):
        _call(da, out1)
        _call(db, out2)
        _call(da, out2)
        _call(db, out1)
    torch.cuda.synchronize()
    assert torch.equal(out1, ref_b)
    assert torch.equal(out2, ref_a)
