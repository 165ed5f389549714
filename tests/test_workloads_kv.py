"""The seeded key-side workload generator (CPU): the page table it writes describes
exactly the histories it drew, every cache row is finite, and the generator is
deterministic. The oracle and the kernels both read these tables, so they are checked
here against their definition (Inputs and Outputs table: kv_cache [num_pages, 2,
page_size, N, D], page_offsets [B+1], page_ids, last_page_len [B])."""
from dataclasses import replace

import pytest
import torch

from hstu_dense_forward_gb300 import workloads as W


@pytest.mark.parametrize("ps", [32, 128, 256])
def test_page_table_matches_histories(ps):
    w = replace(W.KV_WORKLOADS["bf16_paged_b128_hist1k_4k_h4_d128"], batch=9,
                hist_range=(0, 700), new_range=(0, 90), page_size=ps, seed=3)
    d = W.generate_kv(w)
    po, ids, last, hist = d["page_offsets"], d["page_ids"], d["last_page_len"], d["history"]
    pages = po[1:] - po[:-1]
    assert int(po[0]) == 0 and bool((pages >= 0).all())
    assert ids.numel() == int(po[-1]) == len(set(ids.tolist()))  # each page used once
    assert bool((ids >= 0).all()) and bool((ids < d["kv_cache"].shape[0]).all())
    used = pages > 0
    assert bool(((last >= 1) & (last <= ps))[used].all())
    h = torch.where(used, (pages - 1) * ps + last, torch.zeros_like(pages))
    assert torch.equal(h, hist)
    assert torch.isfinite(d["kv_cache"].float()).all()
    lq = d["seq_offsets"][1:] - d["seq_offsets"][:-1]
    lnew = d["seq_offsets_k"][1:] - d["seq_offsets_k"][:-1]
    assert torch.equal(lq, lnew)  # the new tokens are the queries
    assert d["k"].shape[0] == int(d["seq_offsets_k"][-1]) and d["q"].shape[0] == int(lq.sum())
    assert torch.equal(d["num_targets"], lq)


def test_contiguous_form_and_determinism():
    w = replace(W.KV_WORKLOADS["bf16_paged_b128_hist1k_4k_h4_d128"], batch=4,
                hist_range=(10, 300), new_range=(1, 50), page_size=0, query_range=(1, 80))
    a, b = W.generate_kv(w), W.generate_kv(w)
    assert a["kv_cache"] is None and a["page_offsets"] is None
    lk = a["seq_offsets_k"][1:] - a["seq_offsets_k"][:-1]
    lq = a["seq_offsets"][1:] - a["seq_offsets"][:-1]
    assert bool((lq <= lk).all())
    for key in ("q", "k", "v", "seq_offsets", "seq_offsets_k"):
        assert torch.equal(a[key].float() if a[key].is_floating_point() else a[key],
                           b[key].float() if b[key].is_floating_point() else b[key])


def test_fp8_workloads_cast_to_e4m3():
    w = replace(W.KV_WORKLOADS["fp8_paged_b128_hist1k_4k_h4_d128"], batch=2,
                hist_range=(100, 200), new_range=(5, 20))
    d = W.generate_kv(w)
    for key in ("q", "k", "v", "kv_cache"):
        assert d[key].dtype == torch.float8_e4m3fn
        assert torch.isfinite(d[key].float()).all()
