"""Queries that are the newest tokens of longer key sequences, and keys whose history sits
in a paged KV cache (Inputs and Outputs table: seq_offsets_q / seq_offsets_k /
max_seq_len_k / is_delta_qk, kv_cache / page_offsets / page_ids / last_page_len; feature
table "Page"), through hstu_fwd_run_kv: against the fp64 oracle, against the call with all
queries (the last rows must agree), against the same keys passed contiguously, and the
device checks of the page table."""
from dataclasses import replace

import numpy as np
import pytest
import torch

import oracle
from hstu_dense_forward_gb300 import HstuError, HstuFwdPlan, hstu_fwd
from hstu_dense_forward_gb300 import workloads as W

pytestmark = pytest.mark.gpu

TOL = {"fp32": 1e-5, "bf16": 2e-2, "fp16": 1e-2,
       "fp8": 2.0 ** -4}  # E4M3 rounding of P (derivation in test_gpu_fp8.py)
BASE = W.KV_WORKLOADS["bf16_paged_b128_hist1k_4k_h4_d128"]
KEYS = ("q", "k", "v", "seq_offsets", "seq_offsets_k", "kv_cache", "page_offsets", "page_ids",
        "last_page_len", "num_context", "num_targets", "rab")


def _case(dtype="bf16", d=128, heads=(4, 4), **kw):
    w = replace(BASE, dtype=dtype, head_dim=d, num_heads_q=heads[0], num_heads_kv=heads[1],
                **kw)
    return w, W.generate_kv(w)


def _gpu(inp, dev, **extra):
    dv = {k: (inp[k].to(dev) if inp.get(k) is not None else None) for k in KEYS}
    kw = dict(max_seqlen=inp["max_seqlen"], max_seqlen_k=inp["max_seqlen_k"],
              num_context=dv["num_context"], num_targets=dv["num_targets"], rab=dv["rab"],
              causal=inp["causal"], target_group_size=inp["target_group_size"],
              alpha=inp["alpha"], silu_scale=inp["silu_scale"], seq_offsets_k=dv["seq_offsets_k"],
              kv_cache=dv["kv_cache"], page_offsets=dv["page_offsets"],
              page_ids=dv["page_ids"], last_page_len=dv["last_page_len"])
    kw.update(extra)
    return hstu_fwd(dv["q"], dv["k"], dv["v"], dv["seq_offsets"], **kw)


def _oracle(inp, mask=None, rows=None):
    kw = dict(seq_offsets_k=inp["seq_offsets_k"], kv_cache=inp["kv_cache"],
              page_offsets=inp["page_offsets"], page_ids=inp["page_ids"],
              last_page_len=inp["last_page_len"], num_context=inp["num_context"],
              num_targets=inp["num_targets"], rab=inp["rab"],
              mask_type=(oracle.MASK_CUSTOM if mask is not None else
                         oracle.MASK_CAUSAL if inp["causal"] else oracle.MASK_NONE),
              target_group_size=inp["target_group_size"], alpha=inp["alpha"],
              silu_scale=inp["silu_scale"], max_seqlen=inp["max_seqlen_k"], nthreads=16,
              mask=mask)
    if rows is not None:
        return oracle.hstu_fwd_rows(inp["q"], inp["k"], inp["v"], inp["seq_offsets"], rows, **kw)
    return oracle.hstu_fwd(inp["q"], inp["k"], inp["v"], inp["seq_offsets"], **kw)


def _rel_err(got, ref):
    g = got.double().cpu().numpy().reshape(ref.shape)
    return float(np.max(np.abs(g - ref)) / max(np.max(np.abs(ref)), 1e-30))


# histories that end inside a 128-key tile, on a tile boundary, sequences without history
# and with every key cached, queries reaching into the history
CASES = [
    ("bf16", 128, (4, 4), 128, dict()),
    ("bf16", 128, (4, 4), 32, dict(target_group_size=2, context_range=(0, 40))),
    ("fp16", 64, (8, 2), 256, dict(query_range=(1, 400))),
    ("bf16", 256, (2, 1), 128, dict(causal=False)),
    ("fp16", 32, (4, 4), 32, dict(rab=True, targets_are_queries=False)),
    ("bf16", 64, (4, 4), 128, dict(rab=True, query_range=(0, 300), targets_are_queries=False)),
    ("fp32", 64, (2, 1), 32, dict(target_group_size=3)),
    ("fp32", 32, (2, 2), 128, dict(rab=True, query_range=(1, 200))),
]


@pytest.mark.parametrize("dtype,d,heads,ps,extra", CASES)
def test_paged_matches_oracle(cuda_device, dtype, d, heads, ps, extra):
    w, inp = _case(dtype, d, heads, batch=5, hist_range=(0, 420), new_range=(0, 300),
                   page_size=ps, seed=61, **extra)
    got = _gpu(inp, cuda_device)
    torch.cuda.synchronize()
    ref = _oracle(inp)
    assert _rel_err(got, ref) <= TOL[dtype]


@pytest.mark.parametrize("dtype,d,heads,ps", [("bf16", 128, (4, 4), 128), ("fp16", 64, (4, 2), 32),
                                              ("bf16", 256, (2, 2), 256), ("fp32", 64, (2, 2), 32)])
def test_edge_histories(cuda_device, dtype, d, heads, ps):
    """History lengths 0, 128 (a tile boundary), 1, 300 with no new rows (all keys cached)
    and 257 with one query; lengths set through explicit page tables."""
    g = torch.Generator().manual_seed(7)
    dt = W.DTYPES[dtype]
    hist = [0, 128, 1, 300, 257]
    lnew = [200, 130, 70, 0, 5]
    lq = [150, 130, 71, 300, 1]
    B, Nq, Nk = 5, heads[0], heads[1]
    npages = [-(-h // ps) for h in hist]
    num_pages = sum(npages) + 2
    cache = (torch.randn(num_pages, 2, ps, Nk, d, generator=g) * 0.5).to(dt)
    ids = torch.randperm(num_pages, generator=g)[:sum(npages)]
    po = torch.tensor([0] + list(np.cumsum(npages)))
    last = torch.tensor([h - (n - 1) * ps if n else 1 for h, n in zip(hist, npages)])
    so_k = torch.tensor([0] + list(np.cumsum(lnew)))
    so_q = torch.tensor([0] + list(np.cumsum(lq)))
    inp = dict(q=(torch.randn(sum(lq), Nq, d, generator=g) * 0.5).to(dt),
               k=(torch.randn(max(sum(lnew), 1), Nk, d, generator=g) * 0.5).to(dt),
               v=(torch.randn(max(sum(lnew), 1), Nk, d, generator=g) * 0.5).to(dt),
               seq_offsets=so_q, seq_offsets_k=so_k, kv_cache=cache, page_offsets=po,
               page_ids=ids, last_page_len=last, num_context=None,
               num_targets=torch.tensor(lq), rab=None, causal=True, target_group_size=1,
               alpha=0.3, silu_scale=1.0 / 512, max_seqlen=304, max_seqlen_k=512)
    got = _gpu(inp, cuda_device)
    torch.cuda.synchronize()
    assert _rel_err(got, _oracle(inp)) <= TOL[dtype]


@pytest.mark.parametrize("dtype,d,heads", [("bf16", 128, (4, 4)), ("fp16", 64, (8, 2)),
                                           ("fp32", 64, (2, 2))])
def test_fewer_queries_equal_last_rows_of_full_call(cuda_device, dtype, d, heads):
    """Without a cache, the rows of a call with the last Lq queries equal the same rows
    of the call with all Lk queries, bit for bit (same key tiles in the same order)."""
    w, inp = _case(dtype, d, heads, batch=6, hist_range=(0, 500), new_range=(1, 300),
                   page_size=0, query_range=(0, 400), targets_are_queries=False,
                   context_range=(0, 30), target_group_size=2, seed=62)
    lk = (inp["seq_offsets_k"][1:] - inp["seq_offsets_k"][:-1])
    lq = (inp["seq_offsets"][1:] - inp["seq_offsets"][:-1])
    g = torch.Generator().manual_seed(9)
    q_full = (torch.randn(int(lk.sum()), heads[0], d, generator=g) * 0.5).to(W.DTYPES[dtype])
    rows = torch.cat([torch.arange(int(inp["seq_offsets_k"][b + 1] - lq[b]),
                                   int(inp["seq_offsets_k"][b + 1])) for b in range(6)])
    inp["q"] = q_full[rows]
    nt = torch.randint(0, 50, (6,), generator=g)
    inp["num_targets"] = nt
    delta = _gpu(inp, cuda_device)
    dev = cuda_device
    full = hstu_fwd(q_full.to(dev), inp["k"].to(dev), inp["v"].to(dev),
                    inp["seq_offsets_k"].to(dev), max_seqlen=inp["max_seqlen_k"],
                    num_context=inp["num_context"].to(dev), num_targets=nt.to(dev),
                    target_group_size=2, alpha=inp["alpha"], silu_scale=inp["silu_scale"])
    torch.cuda.synchronize()
    assert torch.equal(delta, full[rows.to(dev)])
    assert _rel_err(delta, _oracle(inp)) <= TOL[dtype]


@pytest.mark.parametrize("dtype,ps", [("bf16", 128), ("fp16", 256), ("fp32", 32)])
def test_paged_equals_contiguous_keys(cuda_device, dtype, ps):
    """The same keys, paged or passed contiguously: bit for bit when every history ends on
    a 128-key tile boundary (same tiles), within the tolerance otherwise (the tile where
    the history ends is split into two products)."""
    for aligned in (True, False):
        hr = (256, 256) if aligned else (100, 700)
        w, inp = _case(dtype, 64, (4, 2), batch=6, hist_range=hr, new_range=(0, 300),
                       page_size=ps, query_range=(1, 500), targets_are_queries=False, seed=63)
        contig = W.generate_kv(replace(w, page_size=0))
        # same values: rebuild the contiguous keys from the paged ones
        ks, vs = [], []
        for b in range(w.batch):
            pages = inp["page_ids"][inp["page_offsets"][b]:inp["page_offsets"][b + 1]]
            h = int(inp["history"][b])
            hk = inp["kv_cache"][pages, 0].reshape(-1, *inp["kv_cache"].shape[3:])[:h]
            hv = inp["kv_cache"][pages, 1].reshape(-1, *inp["kv_cache"].shape[3:])[:h]
            a, e = int(inp["seq_offsets_k"][b]), int(inp["seq_offsets_k"][b + 1])
            ks.append(torch.cat([hk, inp["k"][a:e]]))
            vs.append(torch.cat([hv, inp["v"][a:e]]))
        lk = torch.tensor([x.shape[0] for x in ks])
        so_k = torch.zeros(w.batch + 1, dtype=torch.int64)
        so_k[1:] = torch.cumsum(lk, 0)
        contig.update(q=inp["q"], seq_offsets=inp["seq_offsets"], k=torch.cat(ks),
                      v=torch.cat(vs), seq_offsets_k=so_k)
        a = _gpu(inp, cuda_device)
        b = _gpu(contig, cuda_device)
        torch.cuda.synchronize()
        if aligned:
            assert torch.equal(a, b)
        else:
            assert _rel_err(a, b.double().cpu().numpy()) <= TOL[dtype]


def test_paged_custom_mask_matches_oracle(cuda_device):
    """A custom mask [B, Nq, Sk, Sk] read at the query positions, with a paged history."""
    w, inp = _case("bf16", 128, (2, 2), batch=3, hist_range=(50, 300), new_range=(10, 200),
                   page_size=32, causal=False, targets_are_queries=False, seed=64)
    inp["num_targets"] = None
    Sk = inp["max_seqlen_k"]
    g = torch.Generator().manual_seed(3)
    m = (torch.rand(3, 2, Sk, Sk, generator=g) * 3.0 - 1.0).to(torch.bfloat16)
    got = _gpu(inp, cuda_device, mask=m.to(cuda_device), causal=True)
    torch.cuda.synchronize()
    assert _rel_err(got, _oracle(inp, mask=m)) <= TOL["bf16"]


@pytest.mark.parametrize("dtype,d,ps", [("bf16", 64, 32), ("fp16", 128, 128), ("bf16", 96, 0),
                                         ("fp32", 64, 32)])
def test_key_side_custom_mask_with_rab(cuda_device, dtype, d, ps):
    """A custom mask together with rab on the key side (a paged history, or own k/v offsets
    without a cache): both read at the query positions, rab added before the SiLU and the
    mask multiplied after it."""
    w, inp = _case(dtype, d, (2, 2), batch=3, hist_range=(50, 300), new_range=(10, 200),
                   page_size=ps, causal=False, targets_are_queries=False, rab=True,
                   rab_sigma=0.4, seed=66 + d)
    inp["num_targets"] = None
    Sk = inp["max_seqlen_k"]
    g = torch.Generator().manual_seed(4)
    m = (torch.rand(3, 2, Sk, Sk, generator=g) * 3.0 - 1.0).to(inp["q"].dtype)
    got = _gpu(inp, cuda_device, mask=m.to(cuda_device), causal=True)
    torch.cuda.synchronize()
    assert _rel_err(got, _oracle(inp, mask=m)) <= TOL[dtype]


def _plan_and_inputs(dev, ps=32, max_seqlen=None, max_seqlen_k=None):
    w, inp = _case("bf16", 64, (2, 2), batch=3, hist_range=(40, 200), new_range=(5, 60),
                   page_size=ps, seed=65)
    plan = HstuFwdPlan(dtype=torch.bfloat16, batch=3, num_heads_q=2, num_heads_kv=2, head_dim=64,
                       max_seqlen=max_seqlen or inp["max_seqlen"], index_is_int64=True,
                       causal=True, target_group_size=1, has_rab=False, has_num_context=False,
                       has_num_targets=True, is_delta_qk=True,
                       max_seqlen_k=max_seqlen_k or inp["max_seqlen_k"], page_size=ps)
    dv = {k: (inp[k].to(dev) if inp.get(k) is not None else None) for k in KEYS}
    return plan, inp, dv


def _run(plan, dv, out, **over):
    args = dict(seq_offsets_k=dv["seq_offsets_k"], kv_cache=dv["kv_cache"],
                page_offsets=dv["page_offsets"], page_ids=dv["page_ids"],
                last_page_len=dv["last_page_len"], num_targets=dv["num_targets"], alpha=0.2)
    args.update(over)
    plan.run(dv["q"], dv["k"], dv["v"], dv["seq_offsets"], out, **args)


@pytest.mark.parametrize("what", ["page_id_out_of_range", "page_id_negative", "last_page_len_0",
                                  "last_page_len_too_big", "more_queries_than_keys",
                                  "keys_above_bound"])
def test_bad_page_tables_are_reported(cuda_device, what):
    """Unusable key-side inputs are rejected on the device before any key is read: the
    error word says HSTU_DEVERR_OFFSETS and out keeps its contents."""
    plan, inp, dv = _plan_and_inputs(cuda_device, max_seqlen=512 if what ==
                                     "more_queries_than_keys" else None,
                                     max_seqlen_k=64 if what == "keys_above_bound" else None)
    over = {}
    if what == "page_id_out_of_range":
        ids = dv["page_ids"].clone()
        ids[1] = inp["kv_cache"].shape[0]
        over["page_ids"] = ids
    elif what == "page_id_negative":
        ids = dv["page_ids"].clone()
        ids[0] = -1
        over["page_ids"] = ids
    elif what in ("last_page_len_0", "last_page_len_too_big"):
        last = dv["last_page_len"].clone()
        last[1] = 0 if what == "last_page_len_0" else 33
        over["last_page_len"] = last
    elif what == "more_queries_than_keys":
        # sequence 0 gets one query more than it has keys (within the query bound)
        so, so_k = dv["seq_offsets"].clone(), dv["seq_offsets_k"]
        lk0 = int(inp["history"][0]) + int(so_k[1] - so_k[0])
        so[1:] += lk0 + 1 - int(so[1] - so[0])
        dv = dict(dv, seq_offsets=so,
                  q=torch.zeros(int(so[-1]), 2, 64, dtype=torch.bfloat16, device=cuda_device))
    out = torch.full((dv["q"].shape[0], 2, 64), 7.0, dtype=torch.bfloat16, device=cuda_device)
    _run(plan, dv, out, **over)
    assert plan.get_error() == 1  # HSTU_DEVERR_OFFSETS
    assert bool((out == 7.0).all())
    # the plan stays usable: a valid call afterwards raises no error
    plan2, inp2, dv2 = _plan_and_inputs(cuda_device)
    out2 = torch.empty_like(dv2["q"])
    _run(plan2, dv2, out2)
    assert plan2.get_error() == 0


def test_key_side_arguments_checked(cuda_device):
    """A key-side plan refuses a call without its page table, hstu_fwd_run refuses it, and
    a plain plan refuses a page table."""
    plan, inp, dv = _plan_and_inputs(cuda_device)
    out = torch.empty_like(dv["q"])
    with pytest.raises(HstuError):
        _run(plan, dv, out, page_ids=None)
    with pytest.raises(HstuError):
        _run(plan, dv, out, seq_offsets_k=None)
    with pytest.raises(HstuError):
        plan.run_ptr(dv["q"].data_ptr(), dv["k"].data_ptr(), dv["v"].data_ptr(),
                     dv["seq_offsets"].data_ptr(), 0, 0, dv["num_targets"].data_ptr(),
                     dv["q"].shape[0], 1.0, 1.0, out.data_ptr(), 0)


@pytest.mark.parametrize("name", list(W.KV_WORKLOADS))
def test_full_size_paged_workload_sampled_rows(cuda_device, name):
    """The paged ranking workloads at their full size (128 sequences, cached histories of
    1k-4k keys in 128-row pages, 32-256 new tokens as targets of group size 1; bf16 and
    FP8 E4M3): sampled output rows against the oracle, in the launch configuration the
    benchmark times."""
    w = W.KV_WORKLOADS[name]
    inp = W.generate_kv(w)
    got = _gpu(inp, cuda_device)
    torch.cuda.synchronize()
    so = inp["seq_offsets"]
    g = torch.Generator().manual_seed(11)
    rows = []
    for _ in range(96):
        b = int(torch.randint(0, w.batch, (1,), generator=g))
        lq = int(so[b + 1] - so[b])
        i = int(torch.randint(0, lq, (1,), generator=g)) if lq else 0
        if lq:
            rows.append((b, int(torch.randint(0, w.num_heads_q, (1,), generator=g)), i))
    rows += [(0, 0, 0), (w.batch - 1, w.num_heads_q - 1, int(so[-1] - so[-2]) - 1)]
    ref = _oracle(inp, rows=np.array(rows))
    sel = torch.stack([got[int(so[b]) + i, h] for b, h, i in rows]).double().cpu().numpy()
    err = np.max(np.abs(sel - ref)) / np.max(np.abs(ref))
    assert err <= TOL[w.dtype]
