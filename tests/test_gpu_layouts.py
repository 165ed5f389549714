"""The normal layout (Inputs and Outputs table, layout: q [B, S, N, D]), the rab
broadcast form [B, 1, S, S] (feature table, "Support for rab broadcasting") and the custom
mask (mask_type 3), through the C ABI: against the fp64 oracle, and against the equivalent
jagged call / the rab replicated to every head / the built-in causal mask."""
from dataclasses import replace

import numpy as np
import pytest
import torch

import oracle
from hstu_dense_forward_gb300 import hstu_fwd, hstu_fwd_noalloc
from hstu_dense_forward_gb300 import workloads as W

pytestmark = pytest.mark.gpu

TOL = {"fp32": 1e-5, "bf16": 2e-2, "fp16": 1e-2}
BASE = W.WORKLOADS["bf16_causal_b32_s2048_h4_d128"]


def _uniform(dtype, d, B, S, heads, **kw):
    w = W.scaled(BASE, batch=B, max_seqlen=S, dtype=dtype, head_dim=d, num_heads_q=heads[0],
                 num_heads_kv=heads[1], **kw)
    return replace(w, fixed_offsets=tuple(b * S for b in range(B + 1)))


def _jagged_call(d, **kw):
    return hstu_fwd(d["q"], d["k"], d["v"], d["seq_offsets"], max_seqlen=d["max_seqlen"],
                    num_context=d["num_context"], num_targets=d["num_targets"],
                    causal=d["causal"], target_group_size=d["target_group_size"],
                    alpha=d["alpha"], silu_scale=d["silu_scale"], **kw)


def _rel_err(got, ref):
    g = got.double().cpu().numpy().reshape(ref.shape)
    return float(np.max(np.abs(g - ref)) / np.max(np.abs(ref)))


@pytest.mark.parametrize("dtype,d,heads,extra", [
    ("bf16", 128, (4, 4), {}),
    ("fp16", 64, (4, 2), dict(context_range=(0, 20), target_range=(10, 60),
                              target_group_size=3)),
    ("fp32", 64, (2, 2), {}),
])
def test_normal_layout_matches_jagged(cuda_device, dtype, d, heads, extra):
    B, S = 3, 320
    w = _uniform(dtype, d, B, S, heads, **extra)
    dv = W.to_device(W.generate(w), cuda_device)
    ref = _jagged_call(dv)
    q4 = dv["q"].view(B, S, *dv["q"].shape[1:])
    k4 = dv["k"].view(B, S, *dv["k"].shape[1:])
    v4 = dv["v"].view(B, S, *dv["v"].shape[1:])
    got = hstu_fwd(q4, k4, v4, None, num_context=dv["num_context"],
                   num_targets=dv["num_targets"], causal=dv["causal"],
                   target_group_size=dv["target_group_size"], alpha=dv["alpha"],
                   silu_scale=dv["silu_scale"], layout="normal")
    torch.cuda.synchronize()
    assert got.shape == q4.shape
    assert torch.equal(got.view_as(ref), ref)


def test_normal_layout_against_oracle(cuda_device):
    B, S = 2, 200
    w = _uniform("bf16", 64, B, S, (2, 2), target_range=(20, 50), target_group_size=2)
    inp = W.generate(w)
    dv = W.to_device(inp, cuda_device)
    q4 = dv["q"].view(B, S, *dv["q"].shape[1:])
    got = hstu_fwd(q4, dv["k"].view(B, S, *dv["k"].shape[1:]), dv["v"].view(B, S, *dv["v"].shape[1:]),
                   num_targets=dv["num_targets"], target_group_size=2, alpha=inp["alpha"],
                   silu_scale=inp["silu_scale"], layout="normal")
    torch.cuda.synchronize()
    ref = oracle.hstu_fwd(inp["q"], inp["k"], inp["v"], inp["seq_offsets"],
                          num_targets=inp["num_targets"], mask_type=oracle.MASK_CAUSAL,
                          target_group_size=2, alpha=inp["alpha"], silu_scale=inp["silu_scale"],
                          max_seqlen=S, nthreads=8)
    assert _rel_err(got, ref) <= TOL["bf16"]


def _bcast_case(dtype, d, heads, causal=True):
    w = W.scaled(BASE, batch=3, max_seqlen=264, len_lo=1, len_hi=264, dtype=dtype, head_dim=d,
                 num_heads_q=heads[0], num_heads_kv=heads[1], causal=causal)
    inp = W.generate(w)
    g = torch.Generator().manual_seed(21)
    rab = (torch.randn(3, 1, 264, 264, generator=g) * 0.5).to(W.DTYPES[dtype])
    return w, inp, rab


@pytest.mark.parametrize("dtype,d,heads,causal", [("bf16", 128, (4, 4), True),
                                                  ("fp16", 64, (8, 2), False),
                                                  ("bf16", 256, (2, 1), True),
                                                  ("fp32", 32, (4, 4), True)])
def test_rab_broadcast_against_oracle_and_replicated(cuda_device, dtype, d, heads, causal):
    w, inp, rab = _bcast_case(dtype, d, heads, causal)
    dv = W.to_device(inp, cuda_device)
    rab_d = rab.to(cuda_device)
    got = _jagged_call(dv, rab=rab_d)
    rep = _jagged_call(dv, rab=rab_d.expand(-1, heads[0], -1, -1).contiguous())
    torch.cuda.synchronize()
    assert torch.equal(got, rep)
    ref = oracle.hstu_fwd(inp["q"], inp["k"], inp["v"], inp["seq_offsets"], rab=rab,
                          mask_type=oracle.MASK_CAUSAL if causal else oracle.MASK_NONE,
                          alpha=inp["alpha"], silu_scale=inp["silu_scale"], max_seqlen=264,
                          nthreads=8)
    T = int(inp["seq_offsets"][-1])
    assert _rel_err(got[:T], ref[:T]) <= TOL[dtype]


def test_rab_broadcast_allocation_free_entry(cuda_device):
    w, inp, rab = _bcast_case("bf16", 64, (4, 4))
    dv = W.to_device(inp, cuda_device)
    rab_d = rab.to(cuda_device)
    ref = _jagged_call(dv, rab=rab_d)
    out = torch.empty_like(dv["q"])
    hstu_fwd_noalloc(dv["q"], dv["k"], dv["v"], dv["seq_offsets"], out, max_seqlen=264,
                     rab=rab_d, causal=True, alpha=dv["alpha"], silu_scale=dv["silu_scale"])
    torch.cuda.synchronize()
    T = int(inp["seq_offsets"][-1])
    assert torch.equal(out[:T], ref[:T])


def _mask_case(dtype, d, heads, S=264, binary=False, seed=31):
    w = W.scaled(BASE, batch=3, max_seqlen=S, len_lo=1, len_hi=S, dtype=dtype, head_dim=d,
                 num_heads_q=heads[0], num_heads_kv=heads[1], causal=False)
    inp = W.generate(w)
    g = torch.Generator().manual_seed(seed)
    if binary:
        m = (torch.rand(3, heads[0], S, S, generator=g) < 0.6).float()
    else:
        m = torch.rand(3, heads[0], S, S, generator=g) * 3.0 - 1.0  # weights in [-1, 2)
    return inp, m.to(W.DTYPES[dtype])


@pytest.mark.parametrize("dtype,d,heads,binary", [("bf16", 128, (4, 4), False),
                                                  ("fp16", 64, (8, 2), True),
                                                  ("bf16", 256, (2, 2), False),
                                                  ("fp32", 64, (2, 1), False)])
def test_custom_mask_against_oracle(cuda_device, dtype, d, heads, binary):
    """mask_type 3: P multiplied by mask[b, h, i, j] after the SiLU and the scaling."""
    inp, m = _mask_case(dtype, d, heads, binary=binary)
    dv = W.to_device(inp, cuda_device)
    got = hstu_fwd(dv["q"], dv["k"], dv["v"], dv["seq_offsets"], max_seqlen=264,
                   alpha=inp["alpha"], silu_scale=inp["silu_scale"], mask=m.to(cuda_device))
    torch.cuda.synchronize()
    ref = oracle.hstu_fwd(inp["q"], inp["k"], inp["v"], inp["seq_offsets"], mask=m,
                          mask_type=oracle.MASK_CUSTOM, alpha=inp["alpha"],
                          silu_scale=inp["silu_scale"], max_seqlen=264, nthreads=8)
    T = int(inp["seq_offsets"][-1])
    assert _rel_err(got[:T], ref[:T]) <= TOL[dtype]


@pytest.mark.parametrize("dtype,d,heads,binary,bcast", [("bf16", 128, (4, 2), False, False),
                                                        ("fp16", 64, (4, 4), True, True),
                                                        ("bf16", 32, (2, 1), False, False),
                                                        ("fp16", 96, (2, 2), False, False),
                                                        ("fp32", 64, (2, 1), False, True)])
def test_custom_mask_with_rab_against_oracle(cuda_device, dtype, d, heads, binary, bcast):
    """A custom mask together with rab (general entry point): x = alpha q.k + rab before the
    SiLU, P times mask[b, h, i, j] after it; rab per head or one plane for every head."""
    inp, m = _mask_case(dtype, d, heads, binary=binary, seed=33 + d)
    g = torch.Generator().manual_seed(44 + d)
    rab = (torch.randn(3, 1 if bcast else heads[0], 264, 264, generator=g) * 0.5).to(
        W.DTYPES[dtype])
    dv = W.to_device(inp, cuda_device)
    got = hstu_fwd(dv["q"], dv["k"], dv["v"], dv["seq_offsets"], max_seqlen=264,
                   alpha=inp["alpha"], silu_scale=inp["silu_scale"], mask=m.to(cuda_device),
                   rab=rab.to(cuda_device))
    torch.cuda.synchronize()
    ref = oracle.hstu_fwd(inp["q"], inp["k"], inp["v"], inp["seq_offsets"], mask=m, rab=rab,
                          mask_type=oracle.MASK_CUSTOM, alpha=inp["alpha"],
                          silu_scale=inp["silu_scale"], max_seqlen=264, nthreads=8)
    T = int(inp["seq_offsets"][-1])
    assert _rel_err(got[:T], ref[:T]) <= TOL[dtype]


def test_custom_mask_with_zero_rab_equals_mask_alone(cuda_device):
    """rab = 0 beside a custom mask gives the mask-only kernel's output bit for bit (the
    same SiLU arithmetic, with rab / 2 = 0 added)."""
    inp, m = _mask_case("bf16", 128, (4, 4), seed=35)
    dv = W.to_device(inp, cuda_device)
    md = m.to(cuda_device)
    zero = torch.zeros(3, 4, 264, 264, dtype=torch.bfloat16, device=cuda_device)
    kw = dict(max_seqlen=264, alpha=inp["alpha"], silu_scale=inp["silu_scale"], mask=md)
    a = hstu_fwd(dv["q"], dv["k"], dv["v"], dv["seq_offsets"], **kw)
    b = hstu_fwd(dv["q"], dv["k"], dv["v"], dv["seq_offsets"], rab=zero, **kw)
    torch.cuda.synchronize()
    T = int(inp["seq_offsets"][-1])
    assert torch.equal(a[:T], b[:T])


def test_custom_causal_mask_matches_builtin(cuda_device):
    """The built-in causal mask written out as a 0/1 custom mask gives the same output
    (the custom path computes the tiles above the diagonal and multiplies them by 0)."""
    inp, _ = _mask_case("bf16", 128, (4, 4))
    dv = W.to_device(inp, cuda_device)
    S = 264
    causal = torch.tril(torch.ones(S, S)).to(torch.bfloat16)
    m = causal[None, None].expand(3, 4, S, S).contiguous().to(cuda_device)
    got = hstu_fwd(dv["q"], dv["k"], dv["v"], dv["seq_offsets"], max_seqlen=S,
                   alpha=inp["alpha"], silu_scale=inp["silu_scale"], mask=m)
    ref = hstu_fwd(dv["q"], dv["k"], dv["v"], dv["seq_offsets"], max_seqlen=S,
                   alpha=inp["alpha"], silu_scale=inp["silu_scale"], causal=True)
    torch.cuda.synchronize()
    T = int(inp["seq_offsets"][-1])
    g, r = got[:T].float(), ref[:T].float()
    assert float((g - r).abs().max()) <= 1e-3 * float(r.abs().max())


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
def test_d256_rab_runs_are_identical_and_match_oracle(cuda_device, dtype):
    """D = 256 with rab: two epilogue groups share a one-tile rab ring; every run must
    read each tile's own rab (a stale tile would change some rows from run to run)."""
    w = W.scaled(BASE, batch=3, max_seqlen=640, len_lo=300, len_hi=640, dtype=dtype,
                 head_dim=256, num_heads_q=2, num_heads_kv=2, rab=True, rab_sigma=1.0, seed=81)
    inp = W.generate(w)
    dv = W.to_device(inp, cuda_device)
    outs = [_jagged_call(dv, rab=dv["rab"]).clone() for _ in range(6)]
    torch.cuda.synchronize()
    for o in outs[1:]:
        assert torch.equal(o, outs[0])
    ref = oracle.hstu_fwd(inp["q"], inp["k"], inp["v"], inp["seq_offsets"], rab=inp["rab"],
                          mask_type=oracle.MASK_CAUSAL, alpha=inp["alpha"],
                          silu_scale=inp["silu_scale"], max_seqlen=640, nthreads=8)
    T = int(inp["seq_offsets"][-1])
    assert _rel_err(outs[0][:T], ref[:T]) <= TOL[dtype]


def test_general_entry_point_matches_the_specific_ones(cuda_device):
    """hstu_fwd_run_args with a plain plan (rab, context and targets) gives hstu_fwd_run's
    output bit for bit, and rejects inputs the plan does not take (a mask, descales)."""
    import ctypes

    from hstu_dense_forward_gb300 import HstuFwdPlan, _abi
    w = W.Workload(name="args", dtype="bf16", batch=3, num_heads_q=4, num_heads_kv=2,
                   head_dim=64, max_seqlen=264, len_lo=60, len_hi=264, causal=True,
                   context_range=(0, 10), target_range=(0, 30), target_group_size=2, rab=True,
                   rab_sigma=0.3, seed=61)
    d = W.to_device(W.generate(w), cuda_device)
    plan = HstuFwdPlan(dtype=torch.bfloat16, batch=3, num_heads_q=4, num_heads_kv=2, head_dim=64,
                       max_seqlen=264, index_is_int64=True, causal=True, target_group_size=2,
                       has_rab=True, has_num_context=True, has_num_targets=True)
    a_out = torch.full_like(d["q"], float("nan"))
    b_out = torch.full_like(d["q"], float("nan"))
    plan.run(d["q"], d["k"], d["v"], d["seq_offsets"], a_out, rab=d["rab"],
             num_context=d["num_context"], num_targets=d["num_targets"], alpha=d["alpha"],
             silu_scale=d["silu_scale"])
    args = _abi.Args()
    args.q, args.k, args.v, args.out = (d["q"].data_ptr(), d["k"].data_ptr(), d["v"].data_ptr(),
                                        b_out.data_ptr())
    args.seq_offsets, args.rab = d["seq_offsets"].data_ptr(), d["rab"].data_ptr()
    args.num_context, args.num_targets = d["num_context"].data_ptr(), d["num_targets"].data_ptr()
    args.total_tokens, args.alpha, args.silu_scale = d["q"].shape[0], d["alpha"], d["silu_scale"]
    stream = torch.cuda.current_stream(cuda_device).cuda_stream or None
    lib = _abi.lib()
    assert lib.hstu_fwd_run_args(plan._h, ctypes.byref(args), stream) == _abi.HSTU_OK
    torch.cuda.synchronize()
    T = int(d["seq_offsets"][-1])
    assert torch.equal(a_out[:T], b_out[:T])
    args.mask = d["rab"].data_ptr()  # a plain plan takes no mask
    assert lib.hstu_fwd_run_args(plan._h, ctypes.byref(args), stream) == _abi.HSTU_ERR_INVALID_ARG
    args.mask = None
    ds = _abi.Descale()
    args.descale = ctypes.pointer(ds)  # nor descale factors
    assert lib.hstu_fwd_run_args(plan._h, ctypes.byref(args), stream) == _abi.HSTU_ERR_INVALID_ARG
    plan.close()
