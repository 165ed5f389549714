"""Guard bands: out is a view of a larger buffer whose rows after the last token (and a
band before the first) hold a canary; no kernel may write outside [0, T) of out, whatever
the head dim, dtype or output path (TMA block stores, row stores, the fp32 kernel)."""
import pytest
import torch

from hstu_dense_forward_gb300 import hstu_fwd
from hstu_dense_forward_gb300 import workloads as W

pytestmark = pytest.mark.gpu

BAND = 160  # rows of canary on each side (more than one 128-row tile)


@pytest.mark.parametrize("dtype,d", [("bf16", 128), ("fp16", 64), ("bf16", 256), ("bf16", 32),
                                     ("fp32", 64)])
def test_no_write_outside_out(cuda_device, dtype, d):
    w = W.scaled(W.WORKLOADS["bf16_causal_b32_s2048_h4_d128"], batch=3, max_seqlen=300,
                 len_lo=1, len_hi=300, dtype=dtype, head_dim=d, num_heads_q=2, num_heads_kv=2,
                 seed=97)
    inp = W.generate(w)
    dv = W.to_device(inp, cuda_device)
    T = dv["q"].shape[0]
    big = torch.full((T + 2 * BAND, 2, d), 1234.0, dtype=dv["q"].dtype, device=cuda_device)
    out = big[BAND:BAND + T]
    hstu_fwd(dv["q"], dv["k"], dv["v"], dv["seq_offsets"], max_seqlen=300, alpha=w.alpha_value,
             silu_scale=w.silu_scale_value, out=out)
    torch.cuda.synchronize()
    assert bool((big[:BAND] == 1234.0).all())
    assert bool((big[BAND + T:] == 1234.0).all())
    assert bool(torch.isfinite(out.float()).all())


@pytest.mark.parametrize("dtype,d", [("bf16", 64), ("fp16", 32), ("bf16", 128)])
def test_no_write_outside_out_with_rab(cuda_device, dtype, d):
    """The rab kernels write O by row stores from registers (no staging), with ragged last
    tiles: still nothing outside [0, T) of out."""
    w = W.scaled(W.WORKLOADS["bf16_rab_b16_s1024_h8_d64"], batch=3, max_seqlen=304, len_lo=1,
                 len_hi=300, dtype=dtype, head_dim=d, num_heads_q=2, num_heads_kv=2, seed=98)
    inp = W.generate(w)
    dv = W.to_device(inp, cuda_device)
    T = dv["q"].shape[0]
    big = torch.full((T + 2 * BAND, 2, d), 1234.0, dtype=dv["q"].dtype, device=cuda_device)
    out = big[BAND:BAND + T]
    hstu_fwd(dv["q"], dv["k"], dv["v"], dv["seq_offsets"], max_seqlen=304, rab=dv["rab"],
             causal=True, alpha=w.alpha_value, silu_scale=w.silu_scale_value, out=out)
    torch.cuda.synchronize()
    assert bool((big[:BAND] == 1234.0).all())
    assert bool((big[BAND + T:] == 1234.0).all())
    assert bool(torch.isfinite(out.float()).all())
