"""GPU parity: the CUDA library (through its C ABI) against the fp64 CPU oracle on
the same seeded inputs, element by element.

Bar: max |O_gpu - O_oracle| / max |O_oracle| <= 1e-5 (fp32), 2e-2 (bf16), 1e-2 (fp16),
over every row that belongs to a sequence. Small cases run the whole oracle; the
full-size workloads are compared whole (every output row) where the oracle finishes in
seconds on the host cores, else on sampled rows (oracle row by row), in the launch
configuration the benchmark times.
"""
import os

import numpy as np
import pytest
import torch

import oracle
from hstu_dense_forward_gb300 import HstuFwdPlan, _abi, hstu_fwd
from hstu_dense_forward_gb300 import workloads as W

pytestmark = pytest.mark.gpu

TOL = {"fp32": 1e-5, "bf16": 2e-2, "fp16": 1e-2,
       # FP8 E4M3: P is rounded to E4M3 (relative 2^-4) for the second product; the per-row
       # bound derived from that is checked in test_gpu_fp8.py
       "fp8": 2.0 ** -4}


def _oracle_full(inp, nthreads=8):
    return oracle.hstu_fwd(inp["q"], inp["k"], inp["v"], inp["seq_offsets"], rab=inp["rab"],
                           num_context=inp["num_context"], num_targets=inp["num_targets"],
                           mask_type=oracle.MASK_CAUSAL if inp["causal"] else oracle.MASK_NONE,
                           target_group_size=inp["target_group_size"], alpha=inp["alpha"],
                           silu_scale=inp["silu_scale"], max_seqlen=inp["max_seqlen"],
                           nthreads=nthreads)


def _gpu(inp, dev, out=None):
    d = W.to_device(inp, dev)
    o = hstu_fwd(d["q"], d["k"], d["v"], d["seq_offsets"], max_seqlen=d["max_seqlen"],
                 rab=d["rab"], num_context=d["num_context"], num_targets=d["num_targets"],
                 causal=d["causal"], target_group_size=d["target_group_size"], alpha=d["alpha"],
                 silu_scale=d["silu_scale"], out=out)
    torch.cuda.synchronize()
    return o


def _rel_err(got, ref, so):
    T = int(so[-1])
    g = got[:T].double().cpu().numpy()
    r = ref[:T]
    scale = np.max(np.abs(r))
    assert scale > 0
    return float(np.max(np.abs(g - r)) / scale)


def _check(w, dev):
    inp = W.generate(w)
    got = _gpu(inp, dev)
    ref = _oracle_full(inp)
    err = _rel_err(got, ref, inp["seq_offsets"].numpy())
    assert np.isfinite(err) and err <= TOL[w.dtype], f"{w.name}: rel err {err:.3e}"
    return err


# ----------------------------------------------------------------- small whole-output cases
SMALL = [
    W.WORKLOADS["fp32_tiny"],
    W.scaled(W.WORKLOADS["bf16_causal_b32_s2048_h4_d128"], name="bf16_causal_small", batch=4,
             max_seqlen=400, len_lo=100, len_hi=400),
    W.scaled(W.WORKLOADS["bf16_rab_b16_s1024_h8_d64"], name="bf16_rab_small", batch=3,
             num_heads_q=2, num_heads_kv=2, max_seqlen=264, len_lo=130, len_hi=264),
    W.scaled(W.WORKLOADS["fp16_gqa8x2_targets_b8_s4096_d128"], name="fp16_gqa_targets_small",
             batch=3, num_heads_q=4, num_heads_kv=2, max_seqlen=512, len_lo=200, len_hi=512,
             target_range=(16, 100)),
    W.scaled(W.WORKLOADS["bf16_long_b4_s8192_h4_d256"], name="bf16_d256_small", batch=2,
             num_heads_q=2, num_heads_kv=2, max_seqlen=300, len_lo=300, len_hi=300),
]


@pytest.mark.parametrize("w", SMALL, ids=lambda w: w.name)
def test_small_workloads(cuda_device, w):
    _check(w, cuda_device)


HEAD_DIMS = [16, 32, 48, 64, 80, 96, 112, 128, 144, 160, 176, 192, 208, 224, 240, 256]


@pytest.mark.parametrize("dtype", ["bf16", "fp16", "fp32"])
@pytest.mark.parametrize("d", HEAD_DIMS)
@pytest.mark.parametrize("causal", [True, False])
def test_head_dims(cuda_device, dtype, d, causal):
    """Every multiple of 16 up to 256: the tensor-core kernels built for 32, 64, 128 and 256
    run the others with zero-filled extra columns, whose output columns are never stored
    (the output buffer is filled with NaN first, so a stray store would show)."""
    w = W.Workload(name=f"{dtype}_d{d}", dtype=dtype, batch=3, num_heads_q=2, num_heads_kv=1,
                   head_dim=d, max_seqlen=300, len_lo=1, len_hi=300, causal=causal, seed=7 + d)
    _check(w, cuda_device)


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
@pytest.mark.parametrize("d", [272, 320, 384, 448, 512])
@pytest.mark.parametrize("causal", [True, False])
def test_wide_head_dims(cuda_device, dtype, d, causal):
    """Head dims above 256 (v's D up to 512): S over all D columns, O in two halves of
    256 columns computed by separate work items, with context and target counts."""
    w = W.Workload(name=f"{dtype}_d{d}", dtype=dtype, batch=3, num_heads_q=4, num_heads_kv=2,
                   head_dim=d, max_seqlen=400, len_lo=1, len_hi=400, causal=causal,
                   context_range=(0, 12) if causal else None,
                   target_range=(0, 60) if causal else None, target_group_size=3 if causal else 0,
                   seed=11 + d)
    _check(w, cuda_device)


@pytest.mark.parametrize("d", [16, 48, 80, 208, 400])
def test_padded_head_dims_store_nothing_past_the_output(cuda_device, d):
    """A padded head dim writes exactly its D columns per row: the output is the front of a
    larger buffer whose tail must keep its sentinel (the last rows' extra columns would
    land there)."""
    w = W.Workload(name=f"pad{d}", dtype="bf16", batch=2, num_heads_q=2, num_heads_kv=2,
                   head_dim=d, max_seqlen=260, len_lo=100, len_hi=260, causal=True, seed=90 + d)
    inp = W.generate(w)
    T = int(inp["seq_offsets"][-1])
    n = T * 2 * d
    flat = torch.full((n + 4096,), 7.0, dtype=torch.bfloat16, device=cuda_device)
    got = _gpu(inp, cuda_device, out=flat[:n].view(T, 2, d))
    assert torch.all(flat[n:] == 7.0)
    err = _rel_err(got, _oracle_full(inp), inp["seq_offsets"].numpy())
    assert err <= TOL["bf16"], f"d={d}: rel err {err:.3e}"


@pytest.mark.parametrize("lengths", [(1,), (5, 1, 15), (128,), (129, 127), (256, 255, 257),
                                     (0, 70, 0)])
@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
@pytest.mark.parametrize("causal", [True, False])
def test_ragged_edges(cuda_device, lengths, dtype, causal):
    so = tuple(int(x) for x in np.concatenate([[0], np.cumsum(lengths)]))
    w = W.Workload(name="edges", dtype=dtype, batch=len(lengths), num_heads_q=2, num_heads_kv=2,
                   head_dim=64, max_seqlen=max(max(lengths), 8), fixed_offsets=so, causal=causal,
                   seed=11)
    _check(w, cuda_device)


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
def test_bidirectional_many_sequences(cuda_device, dtype):
    """Without a mask the work list keeps each sequence's query tiles together (one run of
    positions per sequence, binned by its key-tile count): many sequences of lengths from 1
    to 700 fill most bins with runs of different lengths, next to empty sequences."""
    g = np.random.default_rng(41)
    lengths = g.integers(1, 701, size=46)
    lengths[[3, 17, 30]] = 0
    so = tuple(int(x) for x in np.concatenate([[0], np.cumsum(lengths)]))
    w = W.Workload(name="bidir_many", dtype=dtype, batch=len(lengths), num_heads_q=4,
                   num_heads_kv=2, head_dim=64, max_seqlen=704, fixed_offsets=so, causal=False,
                   seed=42)
    _check(w, cuda_device)


@pytest.mark.parametrize("G", [1, 2, 4, 8])
def test_gqa_group_sizes(cuda_device, G):
    w = W.Workload(name=f"gqa{G}", dtype="bf16", batch=2, num_heads_q=8, num_heads_kv=8 // G,
                   head_dim=64, max_seqlen=260, len_lo=130, len_hi=260, causal=True, seed=20 + G)
    _check(w, cuda_device)


@pytest.mark.parametrize("nc,nt,g", [(0, 0, 0), (3, 0, 0), (0, 40, 1), (5, 30, 3), (10, 7, 16),
                                     (0, 300, 4), (200, 20, 2), (7, 150, 64)])
@pytest.mark.parametrize("dtype", ["fp16", "fp32"])
def test_context_target_masks(cuda_device, nc, nt, g, dtype):
    """Context / history / target-group masks, including nt >= L (no history),
    nc beyond the history and groups larger than the target count."""
    w = W.Workload(name="mask", dtype=dtype, batch=3, num_heads_q=2, num_heads_kv=2,
                   head_dim=128, max_seqlen=300, len_lo=150, len_hi=300, causal=True,
                   context_range=(nc, nc), target_range=(nt, nt), target_group_size=g, seed=31)
    _check(w, cuda_device)


@pytest.mark.parametrize("dtype", ["bf16", "fp16", "fp32"])
def test_rab_variants(cuda_device, dtype):
    w = W.Workload(name="rab", dtype=dtype, batch=3, num_heads_q=4, num_heads_kv=2, head_dim=64,
                   max_seqlen=392, len_lo=1, len_hi=392, causal=True, context_range=(0, 20),
                   target_range=(0, 60), target_group_size=5, rab=True, rab_sigma=0.5, seed=41)
    _check(w, cuda_device)


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
@pytest.mark.parametrize("d", [32, 64])
@pytest.mark.parametrize("alpha", [0.3, 0.125, 0.0, 1e-6])
def test_rab_paths_small_head_dims(cuda_device, dtype, d, alpha):
    """Head dims up to 64 add rab with the tensor core when 1/alpha is a finite normal
    value of the input type (0.3: 1/alpha rounded once; 0.125: exact), else in the
    epilogue (alpha = 0; 1e-6, whose reciprocal overflows fp16); both match the oracle."""
    w = W.Workload(name="rabpath", dtype=dtype, batch=3, num_heads_q=4, num_heads_kv=4,
                   head_dim=d, max_seqlen=264, len_lo=40, len_hi=264, causal=True,
                   context_range=(0, 12), target_range=(0, 30), target_group_size=3, rab=True,
                   rab_sigma=0.5, sigma=0.7, alpha=alpha, seed=43)
    _check(w, cuda_device)


def test_int32_offsets(cuda_device):
    w = W.Workload(name="i32", dtype="bf16", batch=3, num_heads_q=2, num_heads_kv=2, head_dim=128,
                   max_seqlen=300, len_lo=50, len_hi=300, causal=True, context_range=(0, 9),
                   target_range=(0, 40), target_group_size=2, index_dtype=torch.int32, seed=51)
    _check(w, cuda_device)


def test_rows_outside_sequences_untouched_and_deterministic(cuda_device):
    w = W.Workload(name="tail", dtype="bf16", batch=2, num_heads_q=2, num_heads_kv=2,
                   head_dim=64, max_seqlen=200, fixed_offsets=(0, 150, 190), causal=True, seed=61)
    inp = W.generate(w)
    # 10 extra rows after the last sequence
    for key in ("q", "k", "v"):
        inp[key] = torch.cat([inp[key], torch.ones(10, *inp[key].shape[1:], dtype=inp[key].dtype)])
    out = torch.full((200, 2, 64), 7.0, dtype=torch.bfloat16, device=cuda_device)
    a = _gpu(inp, cuda_device, out=out).clone()
    assert torch.all(a[190:] == 7.0)
    b = _gpu(inp, cuda_device, out=out)
    assert torch.equal(a, b)


def test_empty_inputs_return_without_launch(cuda_device):
    q = torch.empty(0, 2, 64, dtype=torch.bfloat16, device=cuda_device)
    so = torch.zeros(3, dtype=torch.int64, device=cuda_device)
    out = hstu_fwd(q, q[:, :1], q[:, :1], so, max_seqlen=16)
    assert out.shape == (0, 2, 64)


def test_invalid_offsets_are_reported_not_written(cuda_device):
    """seq_offsets past the tensor end: the work-list builder refuses them, records
    HSTU_DEVERR_OFFSETS and no output row is written."""
    plan = HstuFwdPlan(dtype=torch.bfloat16, batch=2, num_heads_q=2, num_heads_kv=2, head_dim=64,
                       max_seqlen=128, index_is_int64=True, causal=True, target_group_size=0,
                       has_rab=False, has_num_context=False, has_num_targets=False)
    q = torch.randn(100, 2, 64, device=cuda_device).to(torch.bfloat16)
    so = torch.tensor([0, 60, 160], dtype=torch.int64, device=cuda_device)  # 160 > T = 100
    out = torch.full_like(q, 3.0)
    plan.run(q, q, q, so, out)
    assert plan.get_error() == _abi.HSTU_DEVERR_OFFSETS
    assert torch.all(out == 3.0)
    assert plan.get_error() == _abi.HSTU_DEVERR_NONE  # cleared
    plan.close()


# ----------------------------------------------------------------- full-size workloads
def _sample_rows(so, nq, n, rng):
    B = len(so) - 1
    rows = []
    for _ in range(n):
        b = int(rng.integers(0, B))
        L = int(so[b + 1] - so[b])
        if L == 0:
            continue
        i = int(rng.choice([0, L - 1, int(rng.integers(0, L))]))
        rows.append((b, int(rng.integers(0, nq)), i))
    return np.array(rows, dtype=np.int64)


# full-size configurations whose whole output the oracle computes in seconds on the host
# cores; the D = 256 one (about 1.1e12 fp64 multiply-adds) is checked on sampled rows
WHOLE = ("bf16_causal_b32_s2048_h4_d128", "bf16_rab_b16_s1024_h8_d64",
         "fp16_gqa8x2_targets_b8_s4096_d128")


@pytest.mark.parametrize("name", WHOLE)
def test_full_size_whole_output(cuda_device, name):
    """Every output row of the full-size configuration against the oracle."""
    w = W.WORKLOADS[name]
    inp = W.generate(w)
    got = _gpu(inp, cuda_device)
    ref = _oracle_full(inp, nthreads=os.cpu_count() or 8)
    err = _rel_err(got, ref, inp["seq_offsets"].numpy())
    assert np.isfinite(err) and err <= TOL[w.dtype], f"{name}: rel err {err:.3e}"


@pytest.mark.parametrize("name", [n for n in W.WORKLOADS if n != "fp32_tiny"])
def test_full_size_sampled_rows(cuda_device, name):
    w = W.WORKLOADS[name]
    inp = W.generate(w)
    got = _gpu(inp, cuda_device)
    so = inp["seq_offsets"].numpy()
    rows = _sample_rows(so, w.num_heads_q, 192, np.random.default_rng(5))
    ref = oracle.hstu_fwd_rows(inp["q"], inp["k"], inp["v"], so, rows, rab=inp["rab"],
                               num_context=inp["num_context"], num_targets=inp["num_targets"],
                               mask_type=oracle.MASK_CAUSAL if w.causal else oracle.MASK_NONE,
                               target_group_size=w.target_group_size, alpha=w.alpha_value,
                               silu_scale=w.silu_scale_value, max_seqlen=w.max_seqlen,
                               nthreads=16)
    g = torch.stack([got[int(so[b]) + i, h] for b, h, i in rows]).double().cpu().numpy()
    err = float(np.max(np.abs(g - ref)) / np.max(np.abs(ref)))
    assert np.isfinite(err) and err <= TOL[w.dtype], f"{name}: rel err {err:.3e}"
    assert torch.isfinite(got[: int(so[-1])].float()).all()


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
def test_wide_score_range(cuda_device, dtype):
    """alpha = 1 with unit-variance inputs puts x = q.k over roughly [-40, 40], so
    SiLU is exercised deep in both tails (the packed 16-bit tanh near -1 and +1)."""
    w = W.Workload(name="wide", dtype=dtype, batch=2, num_heads_q=2, num_heads_kv=2, head_dim=64,
                   max_seqlen=300, len_lo=200, len_hi=300, causal=True, sigma=1.0, alpha=1.0,
                   seed=71)
    _check(w, cuda_device)
