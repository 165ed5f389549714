"""The forward kernel's bounded waits (failure detection without a GPU fault): a plan
created in the watchdog test mode (HSTU_TEST_STALL=k) has a K producer that signals
nothing, so the first score product's wait runs out after watchdog_ms. The kernel must
then leave every loop, drain, free its tensor memory and return; the host reads
HSTU_DEVERR_TIMEOUT from the error word, and the context stays usable."""
import time

import numpy as np
import pytest
import torch

import oracle
from hstu_dense_forward_gb300 import HstuFwdPlan, hstu_fwd
from hstu_dense_forward_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def test_wait_that_runs_out_reports_timeout(cuda_device, monkeypatch):
    w = W.scaled(W.WORKLOADS["bf16_causal_b32_s2048_h4_d128"], batch=3, max_seqlen=400,
                 len_lo=100, len_hi=400, seed=95)
    inp = W.generate(w)
    d = W.to_device(inp, cuda_device)
    monkeypatch.setenv("HSTU_TEST_STALL", "k")
    plan = HstuFwdPlan(dtype=torch.bfloat16, batch=3, num_heads_q=4, num_heads_kv=4,
                       head_dim=128, max_seqlen=400, index_is_int64=True, causal=True,
                       target_group_size=0, has_rab=False, has_num_context=False,
                       has_num_targets=False, watchdog_ms=20)
    monkeypatch.delenv("HSTU_TEST_STALL")
    out = torch.full_like(d["q"], 7.0)
    t0 = time.perf_counter()
    plan.run(d["q"], d["k"], d["v"], d["seq_offsets"], out, alpha=w.alpha_value,
             silu_scale=w.silu_scale_value)
    err = plan.get_error()  # synchronises
    elapsed = time.perf_counter() - t0
    assert err == 2  # HSTU_DEVERR_TIMEOUT
    assert elapsed < 5.0
    plan.close()
    # the context is intact: an ordinary call afterwards is correct
    got = hstu_fwd(d["q"], d["k"], d["v"], d["seq_offsets"], max_seqlen=400,
                   alpha=w.alpha_value, silu_scale=w.silu_scale_value)
    torch.cuda.synchronize()
    ref = oracle.hstu_fwd(inp["q"], inp["k"], inp["v"], inp["seq_offsets"],
                          mask_type=oracle.MASK_CAUSAL, alpha=w.alpha_value,
                          silu_scale=w.silu_scale_value, max_seqlen=400, nthreads=8)
    g = got.double().cpu().numpy()
    T = int(inp["seq_offsets"][-1])
    assert np.abs(g[:T] - ref[:T]).max() / np.abs(ref[:T]).max() <= 2e-2
