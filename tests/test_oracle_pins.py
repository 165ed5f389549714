"""Pins for the fp64 CPU oracle: closed forms, library special cases, hand-written
mask matrices and invariants of the definition. CPU only.

Source for every pin: "RecOps Running Case Documentation"
(gitcode.com/Ascend/RecSDK, docs/en/rec_ops/hstu_v1_forward.md), feature table
(attention mechanism S = Q*K^T, P = silu(S), O = P*V; MHA/GQA; jagged layout;
rab; causal mask from num_context / num_targets / target_group_size) and the
Inputs and Outputs table (mask_type codes, silu_scale default, alpha).
"""
import json
import math
import os

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rng(seed):
    return np.random.default_rng(seed)


def _jagged(rng, lengths, nq, nk, d, scale=1.0):
    so = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int64)
    t = int(so[-1])
    q = rng.standard_normal((t, nq, d)) * scale
    k = rng.standard_normal((t, nk, d)) * scale
    v = rng.standard_normal((t, nk, d))
    return q, k, v, so


# --------------------------------------------------------------------------- closed forms
def test_single_token_closed_forms():
    """L = 1: out = silu_scale * silu(alpha * q.k + rab) * v, at x = +-ln 3 and 0."""
    with open(os.path.join(GOLDEN, "closed_forms.json")) as f:
        cases = json.load(f)["cases"]
    for c in cases:
        d = len(c["q"])
        q = np.array(c["q"]).reshape(1, 1, d)
        k = np.array(c["k"]).reshape(1, 1, d)
        v = np.array(c["v"]).reshape(1, 1, d)
        so = np.array([0, 1])
        rab = None if c["rab"] is None else np.full((1, 1, 1, 1), c["rab"])
        out = oracle.hstu_fwd(q, k, v, so, rab=rab, mask_type=oracle.MASK_CAUSAL,
                              alpha=c["alpha"], silu_scale=c["silu_scale"], max_seqlen=1)
        np.testing.assert_allclose(out.reshape(-1), c["expected"], rtol=0, atol=1e-12,
                                   err_msg=c["name"])


def test_silu_odd_part_identity():
    """silu(x) - silu(-x) = x for every x: with Q = 0 and a random rab, the outputs
    for +rab and -rab differ by silu_scale * sum_j valid * rab_ij * v_j."""
    rng = _rng(11)
    lengths = [5, 3]
    q, k, v, so = _jagged(rng, lengths, 2, 1, 3)
    q[:] = 0.0
    S = max(lengths)
    rab = rng.standard_normal((2, 2, S, S)) * 3.0
    kw = dict(mask_type=oracle.MASK_CAUSAL, num_context=[1, 0], num_targets=[2, 1],
              target_group_size=1, alpha=0.7, silu_scale=0.25, max_seqlen=S)
    a = oracle.hstu_fwd(q, k, v, so, rab=rab, **kw)
    b = oracle.hstu_fwd(q, k, v, so, rab=-rab, **kw)
    expect = np.zeros_like(a)
    for bi, L in enumerate(lengths):
        t0 = so[bi]
        m = oracle.mask_matrix(L, oracle.MASK_CAUSAL, [1, 0][bi], [2, 1][bi], 1)
        for h in range(2):
            expect[t0:t0 + L, h] = 0.25 * (m * rab[bi, h, :L, :L]) @ v[t0:t0 + L, 0]
    np.testing.assert_allclose(a - b, expect, rtol=0, atol=1e-12)


def test_q_zero_with_rab_closed_form():
    """Q = 0: x_ij = rab_ij, so out_i = silu_scale * sum_j valid * silu(rab_ij) * v_j,
    with silu from torch (library)."""
    rng = _rng(12)
    lengths = [4, 6]
    q, k, v, so = _jagged(rng, lengths, 1, 1, 2)
    q[:] = 0.0
    S = 6
    rab = rng.standard_normal((2, 1, S, S))
    out = oracle.hstu_fwd(q, k, v, so, rab=rab, mask_type=oracle.MASK_NONE, alpha=3.0,
                          silu_scale=0.5, max_seqlen=S)
    for bi, L in enumerate(lengths):
        t0 = so[bi]
        p = F.silu(torch.from_numpy(rab[bi, 0, :L, :L])).numpy()
        np.testing.assert_allclose(out[t0:t0 + L, 0], 0.5 * p @ v[t0:t0 + L, 0], rtol=0,
                                   atol=1e-12)


@pytest.mark.parametrize("rab_heads", [1, 3])
def test_q_zero_rab_per_head_and_broadcast_closed_form(rab_heads):
    """Q = 0 with three query heads: out[t0+i, h] = silu_scale * sum_j silu(rab[b, r, i, j])
    * v[t0+j, h] with r = h for rab [B, Nq, S, S] and r = 0 for the broadcast form
    [B, 1, S, S] (feature table, "Support for rab broadcasting"); silu from torch."""
    rng = _rng(13)
    lengths = [3, 5]
    q, k, v, so = _jagged(rng, lengths, 3, 3, 2)
    q[:] = 0.0
    S = 5
    rab = rng.standard_normal((2, rab_heads, S, S))
    out = oracle.hstu_fwd(q, k, v, so, rab=rab, mask_type=oracle.MASK_NONE, alpha=2.0,
                          silu_scale=0.25, max_seqlen=S)
    for bi, L in enumerate(lengths):
        t0 = so[bi]
        for h in range(3):
            r = 0 if rab_heads == 1 else h
            p = F.silu(torch.from_numpy(rab[bi, r, :L, :L])).numpy()
            np.testing.assert_allclose(out[t0:t0 + L, h], 0.25 * p @ v[t0:t0 + L, h], rtol=0,
                                       atol=1e-12)


def test_custom_mask_closed_forms():
    """Custom mask (mask_type 3, Inputs and Outputs table): an all-ones mask gives the
    unmasked forward; the built-in causal 0/1 matrix as a custom mask gives the causal
    forward; Q = 0 with a general mask M gives out_i = silu_scale * sum_j silu(0) ... = 0,
    so a rab R is used instead: out_i = silu_scale * sum_j silu(R_ij) * M_ij * v_j
    (mask applied after SiLU and scaling; silu from torch)."""
    rng = _rng(14)
    lengths = [5, 7]
    q, k, v, so = _jagged(rng, lengths, 2, 1, 3)
    S = 7
    ones = np.ones((2, 2, S, S))
    a = oracle.hstu_fwd(q, k, v, so, mask=ones, mask_type=oracle.MASK_CUSTOM, max_seqlen=S,
                        alpha=0.7, silu_scale=0.3)
    b = oracle.hstu_fwd(q, k, v, so, mask_type=oracle.MASK_NONE, max_seqlen=S, alpha=0.7,
                        silu_scale=0.3)
    np.testing.assert_array_equal(a, b)
    causal = np.tril(np.ones((S, S)))[None, None].repeat(2, 0).repeat(2, 1)
    a = oracle.hstu_fwd(q, k, v, so, mask=causal, mask_type=oracle.MASK_CUSTOM, max_seqlen=S,
                        alpha=0.7, silu_scale=0.3)
    b = oracle.hstu_fwd(q, k, v, so, mask_type=oracle.MASK_CAUSAL, max_seqlen=S, alpha=0.7,
                        silu_scale=0.3)
    np.testing.assert_array_equal(a, b)
    q[:] = 0.0
    R = rng.standard_normal((2, 2, S, S))
    M = rng.uniform(-1.0, 2.0, (2, 2, S, S))
    out = oracle.hstu_fwd(q, k, v, so, rab=R, mask=M, mask_type=oracle.MASK_CUSTOM,
                          max_seqlen=S, alpha=1.5, silu_scale=0.25)
    for bi, L in enumerate(lengths):
        t0 = so[bi]
        for h in range(2):
            p = F.silu(torch.from_numpy(R[bi, h, :L, :L])).numpy() * M[bi, h, :L, :L]
            np.testing.assert_allclose(out[t0:t0 + L, h], 0.25 * p @ v[t0:t0 + L, 0], rtol=0,
                                       atol=1e-12)


# ------------------------------------------------------ fewer queries than keys; KV cache
# Inputs and Outputs table: seq_offsets_q / seq_offsets_k / max_seq_len_k / is_delta_qk
# (query and key lengths may differ) and kv_cache [num_pages, 2, page_size, N, D] with
# page_offsets, page_ids, last_page_len (feature table "Page": the KV cache of the history).
# Reading: the queries are the last Lq tokens of the Lk keys (row i at position Lk - Lq + i).
def _delta_case(rng, lk, lq, nq, nk, d):
    """Full sequences of lk keys; the queries of the delta call are the last lq rows."""
    so_k = np.concatenate([[0], np.cumsum(lk)]).astype(np.int64)
    so_q = np.concatenate([[0], np.cumsum(lq)]).astype(np.int64)
    tk = int(so_k[-1])
    q_full = rng.standard_normal((tk, nq, d))
    k = rng.standard_normal((tk, nk, d))
    v = rng.standard_normal((tk, nk, d))
    rows = np.concatenate([np.arange(so_k[b + 1] - lq[b], so_k[b + 1]) for b in range(len(lk))])
    return q_full, k, v, so_k, so_q, rows.astype(np.int64)


def test_delta_queries_are_the_last_rows_of_the_full_forward():
    """With Lq < Lk queries (the last ones), every output row equals the row of the call
    with all Lk queries, bit for bit: mask, rab and targets are taken at the position."""
    rng = _rng(41)
    lk = [9, 6, 12, 1, 7]
    lq = [4, 6, 1, 1, 0]
    q_full, k, v, so_k, so_q, rows = _delta_case(rng, lk, lq, 4, 2, 3)
    S = 13
    rab = rng.standard_normal((5, 4, S, S))
    for kw in (dict(mask_type=oracle.MASK_CAUSAL, num_context=[2, 0, 3, 0, 1],
                    num_targets=[3, 2, 4, 0, 2], target_group_size=2, rab=rab),
               dict(mask_type=oracle.MASK_CAUSAL),
               dict(mask_type=oracle.MASK_NONE, rab=rab[:, :1].copy())):
        full = oracle.hstu_fwd(q_full, k, v, so_k, alpha=0.8, silu_scale=0.2, max_seqlen=S, **kw)
        delta = oracle.hstu_fwd(q_full[rows], k, v, so_q, seq_offsets_k=so_k, alpha=0.8,
                                silu_scale=0.2, max_seqlen=S, **kw)
        np.testing.assert_array_equal(delta, full[rows])
    with pytest.raises(ValueError):  # more queries than keys
        oracle.hstu_fwd(q_full[:3], k[:2], v[:2], [0, 3], seq_offsets_k=[0, 2], max_seqlen=S)


def test_delta_custom_mask_rows_follow_positions():
    """A custom mask is read at the query's position too: the delta rows equal the full
    call's last rows."""
    rng = _rng(42)
    lk, lq = [8, 5], [3, 5]
    q_full, k, v, so_k, so_q, rows = _delta_case(rng, lk, lq, 2, 2, 2)
    S = 8
    m = rng.uniform(-1.0, 2.0, (2, 2, S, S))
    kw = dict(mask=m, mask_type=oracle.MASK_CUSTOM, alpha=1.1, silu_scale=0.3, max_seqlen=S)
    full = oracle.hstu_fwd(q_full, k, v, so_k, **kw)
    delta = oracle.hstu_fwd(q_full[rows], k, v, so_q, seq_offsets_k=so_k, **kw)
    np.testing.assert_array_equal(delta, full[rows])


def _paged(rng, k_full, v_full, so_k, hist, page_size, spare=3):
    """Move the first hist[b] keys of every sequence into randomly placed pages of a cache
    whose unused rows hold large finite values; return the new rows and the page table."""
    B = len(hist)
    npages = [0 if h == 0 else -(-h // page_size) for h in hist]
    num_pages = sum(npages) + spare
    nk, d = k_full.shape[1:]
    cache = rng.uniform(1e5, 2e5, (num_pages, 2, page_size, nk, d))
    ids = rng.permutation(num_pages)[:sum(npages)].astype(np.int64)
    po = np.concatenate([[0], np.cumsum(npages)]).astype(np.int64)
    last = np.zeros(B, dtype=np.int64)
    new_k, new_v, lnew = [], [], []
    for b in range(B):
        t0 = so_k[b]
        for x in range(npages[b]):
            n = min(page_size, hist[b] - x * page_size)
            pg = ids[po[b] + x]
            cache[pg, 0, :n] = k_full[t0 + x * page_size:t0 + x * page_size + n]
            cache[pg, 1, :n] = v_full[t0 + x * page_size:t0 + x * page_size + n]
            last[b] = n
        new_k.append(k_full[t0 + hist[b]:so_k[b + 1]])
        new_v.append(v_full[t0 + hist[b]:so_k[b + 1]])
        lnew.append(int(so_k[b + 1] - t0 - hist[b]))
    so_new = np.concatenate([[0], np.cumsum(lnew)]).astype(np.int64)
    return np.concatenate(new_k), np.concatenate(new_v), so_new, cache, po, ids, last


@pytest.mark.parametrize("page_size", [4, 8])
def test_paged_history_equals_contiguous_keys(page_size):
    """Keys split into cache pages (shuffled page ids, partly filled last pages, sequences
    without history and without new rows) give the same output as the same keys passed
    contiguously, bit for bit."""
    rng = _rng(43 + page_size)
    lk = [11, 6, 9, 16, 5]
    lq = [3, 6, 9, 2, 1]
    hist = [7, 0, 9, 8, 5]  # partial last page, no history, all keys cached, full pages
    q_full, k, v, so_k, so_q, rows = _delta_case(rng, lk, lq, 2, 1, 3)
    nk_, nv_, so_new, cache, po, ids, last = _paged(rng, k, v, so_k, hist, page_size)
    np.testing.assert_array_equal(oracle.history_lengths(po, last, page_size), hist)
    S = 16 + page_size
    rab = rng.standard_normal((5, 2, S, S))
    kw = dict(mask_type=oracle.MASK_CAUSAL, num_context=[1, 2, 0, 3, 0],
              num_targets=[2, 1, 3, 4, 0], target_group_size=1, rab=rab, alpha=0.6,
              silu_scale=0.4, max_seqlen=S)
    ref = oracle.hstu_fwd(q_full[rows], k, v, so_q, seq_offsets_k=so_k, **kw)
    got = oracle.hstu_fwd(q_full[rows], nk_, nv_, so_q, seq_offsets_k=so_new, kv_cache=cache,
                          page_offsets=po, page_ids=ids, last_page_len=last, **kw)
    np.testing.assert_array_equal(got, ref)


def test_delta_paged_q_zero_closed_form():
    """Q = 0 with a rab R, plain causal mask, keys from a cache plus new rows: query i of a
    sequence with Lk keys sits at p = Lk - Lq + i and
    out_i = silu_scale * sum_{j <= p} silu(R[p, j]) * v_j (silu from torch)."""
    rng = _rng(45)
    lk, lq, hist, ps = [10, 7], [4, 7], [6, 4], 4
    q_full, k, v, so_k, so_q, rows = _delta_case(rng, lk, lq, 1, 1, 2)
    nk_, nv_, so_new, cache, po, ids, last = _paged(rng, k, v, so_k, hist, ps)
    S = 10 + ps
    R = rng.standard_normal((2, 1, S, S))
    out = oracle.hstu_fwd(np.zeros((sum(lq), 1, 2)), nk_, nv_, so_q, seq_offsets_k=so_new,
                          kv_cache=cache, page_offsets=po, page_ids=ids, last_page_len=last,
                          rab=R, mask_type=oracle.MASK_CAUSAL, alpha=3.0, silu_scale=0.5,
                          max_seqlen=S)
    for b in range(2):
        vb = v[so_k[b]:so_k[b + 1], 0]
        for i in range(lq[b]):
            p = lk[b] - lq[b] + i
            w = F.silu(torch.from_numpy(R[b, 0, p, :p + 1])).numpy()
            np.testing.assert_allclose(out[so_q[b] + i, 0], 0.5 * w @ vb[:p + 1], rtol=0,
                                       atol=1e-12)


def test_count_valid_kv_closed_forms():
    """Pairs with the queries at the end of the keys: no mask Lq * Lk; plain causal
    sum_i (Lk - Lq + i + 1) = Lq * (Lk - Lq) + Lq * (Lq + 1) / 2; Lq = Lk is the
    ordinary count."""
    lq, lk = [3, 5, 0, 4], [7, 5, 2, 9]
    assert oracle.count_valid_kv(lq, lk, 2, mask_type=oracle.MASK_NONE) == \
        2 * sum(a * b for a, b in zip(lq, lk))
    assert oracle.count_valid_kv(lq, lk, 3, mask_type=oracle.MASK_CAUSAL) == \
        3 * sum(a * (b - a) + a * (a + 1) // 2 for a, b in zip(lq, lk))
    so = np.concatenate([[0], np.cumsum(lk)])
    kw = dict(num_context=[1, 2, 0, 3], num_targets=[2, 1, 0, 5], target_group_size=2)
    assert oracle.count_valid_kv(lk, lk, 2, **kw) == oracle.count_valid(so, 2, **kw)


# --------------------------------------------------------------------------- library cases
def _torch_dense(q, k, v, rab, alpha, scale, causal):
    """Equal-length, no-context/no-target case with torch fp64 library ops.
    q [B, L, Nq, D]; k, v [B, L, Nk, D]; rab [B, Nq, L, L] or None."""
    G = q.shape[2] // k.shape[2]
    qt = torch.from_numpy(q).permute(0, 2, 1, 3)
    kt = torch.from_numpy(k).repeat_interleave(G, dim=2).permute(0, 2, 1, 3)
    vt = torch.from_numpy(v).repeat_interleave(G, dim=2).permute(0, 2, 1, 3)
    x = alpha * torch.matmul(qt, kt.transpose(-1, -2))
    if rab is not None:
        x = x + torch.from_numpy(rab)
    p = F.silu(x) * scale
    if causal:
        p = p * torch.tril(torch.ones(x.shape[-2:], dtype=torch.float64))
    return torch.matmul(p, vt).permute(0, 2, 1, 3).numpy()


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("nq,nk", [(4, 4), (4, 2), (6, 1)])
def test_equal_lengths_match_torch_matmul(causal, nq, nk):
    rng = _rng(13 + nq + nk + int(causal))
    B, L, D = 3, 7, 5
    q = rng.standard_normal((B, L, nq, D))
    k = rng.standard_normal((B, L, nk, D))
    v = rng.standard_normal((B, L, nk, D))
    rab = rng.standard_normal((B, nq, L, L))
    so = np.arange(B + 1) * L
    out = oracle.hstu_fwd(q.reshape(B * L, nq, D), k.reshape(B * L, nk, D),
                          v.reshape(B * L, nk, D), so, rab=rab,
                          mask_type=oracle.MASK_CAUSAL if causal else oracle.MASK_NONE,
                          alpha=0.37, silu_scale=1.0 / L, max_seqlen=L)
    ref = _torch_dense(q, k, v, rab, 0.37, 1.0 / L, causal)
    np.testing.assert_allclose(out.reshape(B, L, nq, D), ref, rtol=1e-12, atol=1e-12)


def test_jagged_lengths_match_torch_per_sequence():
    """Ragged lengths, rab with max_seqlen > L: each sequence reads the top-left
    [L, L] block of its rab slice."""
    rng = _rng(14)
    lengths = [3, 9, 1, 6]
    S = 10
    q, k, v, so = _jagged(rng, lengths, 2, 2, 4)
    rab = rng.standard_normal((4, 2, S, S))
    out = oracle.hstu_fwd(q, k, v, so, rab=rab, mask_type=oracle.MASK_CAUSAL, alpha=0.5,
                          silu_scale=1.0 / S, max_seqlen=S)
    for bi, L in enumerate(lengths):
        t0 = so[bi]
        ref = _torch_dense(q[None, t0:t0 + L], k[None, t0:t0 + L], v[None, t0:t0 + L],
                           rab[bi:bi + 1, :, :L, :L], 0.5, 1.0 / S, True)
        np.testing.assert_allclose(out[t0:t0 + L], ref[0], rtol=1e-12, atol=1e-12)


def test_silu_scale_default_is_one_over_max_seqlen():
    rng = _rng(15)
    q, k, v, so = _jagged(rng, [4, 2], 1, 1, 3)
    a = oracle.hstu_fwd(q, k, v, so, max_seqlen=8)
    b = oracle.hstu_fwd(q, k, v, so, max_seqlen=8, silu_scale=0.125)
    np.testing.assert_array_equal(a, b)


# --------------------------------------------------------------------------- mask matrices
def _cases():
    with open(os.path.join(GOLDEN, "mask_cases.json")) as f:
        return json.load(f)["cases"]


@pytest.mark.parametrize("case", _cases(), ids=lambda c: c["name"])
def test_mask_matrices_through_forward(case):
    """Q = 0, rab = ln 3, V = identity (D = L): out[i, j] = scale * 0.75 ln3 * valid(i, j),
    so the forward itself must reproduce the hand-written 0/1 matrix."""
    L = case["L"]
    want = np.array([[int(ch) for ch in row] for row in case["matrix"]])
    q = np.zeros((L, 1, L))
    k = _rng(16).standard_normal((L, 1, L))
    v = np.eye(L).reshape(L, 1, L)
    rab = np.full((1, 1, L, L), math.log(3.0))
    out = oracle.hstu_fwd(q, k, v, [0, L], rab=rab, num_context=[case["nc"]],
                          num_targets=[case["nt"]], mask_type=case["mask_type"],
                          target_group_size=case["g"], alpha=1.0, silu_scale=0.5, max_seqlen=L)
    got = out[:, 0, :] / (0.5 * 0.75 * math.log(3.0))
    np.testing.assert_allclose(got, want, rtol=0, atol=1e-12)
    m = oracle.mask_matrix(L, case["mask_type"], case["nc"], case["nt"], case["g"])
    np.testing.assert_array_equal(m, want)


def test_count_valid_closed_forms():
    so = [0, 5, 12, 13]
    assert oracle.count_valid(so, 3, mask_type=oracle.MASK_NONE) == 3 * (25 + 49 + 1)
    assert oracle.count_valid(so, 3) == 3 * (15 + 28 + 1)
    nc, nt = [1, 2, 0], [2, 3, 1]
    want = sum(3 * int(oracle.mask_matrix(L, 0, c, t, 2).sum())
               for L, c, t in zip([5, 7, 1], nc, nt))
    assert oracle.count_valid(so, 3, num_context=nc, num_targets=nt, target_group_size=2) == want


# --------------------------------------------------------------------------- invariants
def test_q_zero_without_rab_gives_zero():
    """silu(0) = 0, so Q = 0 and no rab give O = 0 for every mask."""
    rng = _rng(17)
    q, k, v, so = _jagged(rng, [6, 3], 4, 2, 8)
    q[:] = 0.0
    for mt in (oracle.MASK_CAUSAL, oracle.MASK_NONE):
        out = oracle.hstu_fwd(q, k, v, so, mask_type=mt, num_context=[2, 1],
                              num_targets=[2, 1], target_group_size=1, alpha=1.0,
                              silu_scale=1.0)
        assert np.all(out == 0.0)


def test_causal_rows_ignore_later_keys():
    """For rows i >= num_context, perturbing K/V rows j > i leaves row i unchanged."""
    rng = _rng(18)
    lengths = [9, 7]
    q, k, v, so = _jagged(rng, lengths, 2, 1, 4)
    kw = dict(mask_type=oracle.MASK_CAUSAL, num_context=[2, 1], num_targets=[3, 2],
              target_group_size=2, alpha=0.6, silu_scale=0.2)
    base = oracle.hstu_fwd(q, k, v, so, **kw)
    for bi, L in enumerate(lengths):
        nc = kw["num_context"][bi]
        for i in range(nc, L):
            k2, v2 = k.copy(), v.copy()
            t0 = so[bi]
            k2[t0 + i + 1:t0 + L] += 5.0
            v2[t0 + i + 1:t0 + L] -= 3.0
            pert = oracle.hstu_fwd(q, k2, v2, so, **kw)
            np.testing.assert_array_equal(pert[t0 + i], base[t0 + i])


def test_gqa_equals_replicated_mha():
    rng = _rng(19)
    q, k, v, so = _jagged(rng, [5, 8], 6, 2, 4)
    kw = dict(mask_type=oracle.MASK_CAUSAL, num_context=[1, 3], num_targets=[2, 2],
              target_group_size=1, alpha=0.3, silu_scale=0.1)
    gqa = oracle.hstu_fwd(q, k, v, so, **kw)
    mha = oracle.hstu_fwd(q, np.repeat(k, 3, axis=1), np.repeat(v, 3, axis=1), so, **kw)
    np.testing.assert_array_equal(gqa, mha)


def test_batch_permutation_permutes_outputs():
    rng = _rng(20)
    lengths = [4, 7, 2]
    q, k, v, so = _jagged(rng, lengths, 2, 2, 3)
    S = 8
    rab = rng.standard_normal((3, 2, S, S))
    nc, nt = np.array([1, 2, 0]), np.array([1, 3, 1])
    kw = dict(mask_type=oracle.MASK_CAUSAL, target_group_size=2, alpha=0.4, silu_scale=0.3,
              max_seqlen=S)
    out = oracle.hstu_fwd(q, k, v, so, rab=rab, num_context=nc, num_targets=nt, **kw)
    perm = [2, 0, 1]
    seg = lambda a, b: a[so[b]:so[b + 1]]
    q2 = np.concatenate([seg(q, b) for b in perm])
    k2 = np.concatenate([seg(k, b) for b in perm])
    v2 = np.concatenate([seg(v, b) for b in perm])
    so2 = np.concatenate([[0], np.cumsum([lengths[b] for b in perm])])
    out2 = oracle.hstu_fwd(q2, k2, v2, so2, rab=rab[perm], num_context=nc[perm],
                           num_targets=nt[perm], **kw)
    np.testing.assert_array_equal(out2, np.concatenate([seg(out, b) for b in perm]))


def test_v_ones_gives_equal_columns():
    """V = ones: every output column equals the masked row sum of scale*silu(x)."""
    rng = _rng(21)
    q, k, v, so = _jagged(rng, [6, 5], 2, 1, 4)
    kw = dict(mask_type=oracle.MASK_CAUSAL, num_context=[1, 0], num_targets=[2, 2],
              target_group_size=1, alpha=0.9, silu_scale=0.5)
    out = oracle.hstu_fwd(q, k, np.ones_like(v), so, **kw)
    np.testing.assert_array_equal(out, np.repeat(out[:, :, :1], 4, axis=2))
    # V = e_0 (first column ones, others zero) gives that row sum in column 0 only
    e0 = np.zeros_like(v)
    e0[:, :, 0] = 1.0
    one = oracle.hstu_fwd(q, k, e0, so, **kw)
    np.testing.assert_array_equal(one[:, :, 0], out[:, :, 0])
    assert np.all(one[:, :, 1:] == 0.0)


def test_linear_in_silu_scale_and_v():
    rng = _rng(22)
    q, k, v, so = _jagged(rng, [7], 1, 1, 3)
    a = oracle.hstu_fwd(q, k, v, so, alpha=0.5, silu_scale=0.25)
    b = oracle.hstu_fwd(q, k, v, so, alpha=0.5, silu_scale=0.5)
    np.testing.assert_array_equal(2.0 * a, b)
    c = oracle.hstu_fwd(q, k, 4.0 * v, so, alpha=0.5, silu_scale=0.25)
    np.testing.assert_array_equal(4.0 * a, c)


def test_rows_api_matches_full_forward():
    rng = _rng(23)
    lengths = [5, 9]
    q, k, v, so = _jagged(rng, lengths, 4, 2, 6)
    kw = dict(mask_type=oracle.MASK_CAUSAL, num_context=[2, 0], num_targets=[1, 4],
              target_group_size=2, alpha=0.2, silu_scale=0.1, max_seqlen=9)
    full = oracle.hstu_fwd(q, k, v, so, **kw)
    rows = [(0, 0, 0), (0, 3, 4), (1, 1, 8), (1, 2, 3)]
    got = oracle.hstu_fwd_rows(q, k, v, so, rows, nthreads=2, **kw)
    for r, (b, h, i) in enumerate(rows):
        np.testing.assert_array_equal(got[r], full[so[b] + i, h])


def test_threads_do_not_change_results():
    rng = _rng(24)
    q, k, v, so = _jagged(rng, [9, 4, 6], 4, 4, 5)
    a = oracle.hstu_fwd(q, k, v, so, alpha=0.3, silu_scale=0.2, nthreads=1)
    b = oracle.hstu_fwd(q, k, v, so, alpha=0.3, silu_scale=0.2, nthreads=4)
    np.testing.assert_array_equal(a, b)


def test_rejects_bad_head_ratio():
    rng = _rng(25)
    q, k, v, so = _jagged(rng, [3], 3, 2, 2)
    with pytest.raises(ValueError):
        oracle.hstu_fwd(q, k, v, so)


@pytest.mark.parametrize("seed", range(6))
def test_key_side_identities_random_geometries(seed):
    """Random key-side geometries (page sizes, histories on and off page boundaries, empty
    histories and new rows, queries reaching into the history, GQA, targets and context):
    the paged call equals the contiguous-key call and the last rows of the all-queries call,
    bit for bit."""
    rng = _rng(100 + seed)
    B = int(rng.integers(1, 5))
    nk = int(rng.choice([1, 2]))
    nq = nk * int(rng.choice([1, 2, 3]))
    d = int(rng.integers(1, 5))
    ps = int(rng.choice([1, 2, 3, 4, 8]))
    lk = rng.integers(1, 14, B)
    hist = np.array([int(rng.integers(0, L + 1)) for L in lk])
    lq = np.array([int(rng.integers(0, L + 1)) for L in lk])
    q_full, k, v, so_k, so_q, rows = _delta_case(rng, list(lk), list(lq), nq, nk, d)
    nk_, nv_, so_new, cache, po, ids, last = _paged(rng, k, v, so_k, list(hist), ps)
    S = int(lk.max()) + ps
    kw = dict(mask_type=oracle.MASK_CAUSAL, num_context=rng.integers(0, 4, B),
              num_targets=rng.integers(0, 5, B), target_group_size=int(rng.integers(0, 3)),
              rab=rng.standard_normal((B, nq, S, S)), alpha=0.9, silu_scale=0.3, max_seqlen=S)
    full = oracle.hstu_fwd(q_full, k, v, so_k, **kw)
    delta = oracle.hstu_fwd(q_full[rows], k, v, so_q, seq_offsets_k=so_k, **kw)
    paged = oracle.hstu_fwd(q_full[rows], nk_, nv_, so_q, seq_offsets_k=so_new, kv_cache=cache,
                            page_offsets=po, page_ids=ids, last_page_len=last, **kw)
    np.testing.assert_array_equal(delta, full[rows])
    np.testing.assert_array_equal(paged, delta)


# ------------------------------------------------------------ FP8 descale granularities
def test_dequantize_granularities_by_hand():
    """The factor each element gets, written out for a tiny jagged tensor: sequences of
    3 and 5 rows, 2 heads, blocks of 2 rows (so the second sequence spans 3 blocks)."""
    so = np.array([0, 3, 8])
    x = np.arange(8 * 2 * 1, dtype=np.float64).reshape(8, 2, 1) + 1.0
    # per tensor: one factor
    assert np.array_equal(oracle.dequantize(x, [0.5], "tensor", so), 0.5 * x)
    # per batch: rows 0-2 by 2, rows 3-7 by 3
    want = x.copy()
    want[:3] *= 2.0
    want[3:] *= 3.0
    assert np.array_equal(oracle.dequantize(x, [2.0, 3.0], "batch", so), want)
    # per head: [B, N]
    f = np.array([[1.0, 10.0], [100.0, 1000.0]])
    got = oracle.dequantize(x, f, "head", so)
    assert got[1, 0, 0] == 1.0 * x[1, 0, 0] and got[1, 1, 0] == 10.0 * x[1, 1, 0]
    assert got[7, 0, 0] == 100.0 * x[7, 0, 0] and got[4, 1, 0] == 1000.0 * x[4, 1, 0]
    # per block: [B, nblocks, N], block = position in the sequence // 2
    fb = np.arange(2 * 3 * 2, dtype=np.float64).reshape(2, 3, 2) + 1.0
    got = oracle.dequantize(x, fb, "block", so, block=2)
    for t, b, i in [(0, 0, 0), (1, 0, 1), (2, 0, 2), (3, 1, 0), (4, 1, 1), (5, 1, 2),
                    (6, 1, 3), (7, 1, 4)]:
        for n in range(2):
            assert got[t, n, 0] == fb[b, i // 2, n] * x[t, n, 0], (t, n)


def test_dequantize_reduces_to_per_tensor():
    """Every granularity with all factors equal is the per-tensor case, and rows outside
    every sequence are zero."""
    rng = np.random.default_rng(3)
    so = np.array([0, 100, 100, 300])
    x = rng.normal(size=(310, 3, 4))
    ref = oracle.dequantize(x, [0.25], "tensor", so)
    assert np.all(ref[300:] == 0)
    assert np.array_equal(oracle.dequantize(x, np.full(3, 0.25), "batch", so), ref)
    assert np.array_equal(oracle.dequantize(x, np.full((3, 3), 0.25), "head", so), ref)
    assert np.array_equal(oracle.dequantize(x, np.full((3, 2, 3), 0.25), "block", so), ref)


def test_dequantize_kv_positions_by_hand():
    """Key positions on the key side: sequence 0 has cached pages [3, 1] (page_size 2, last
    page 1 row) then two new rows; sequence 1 no pages and one new row. With per-block
    factors of block 2 the positions 0..4 of sequence 0 fall in blocks 0, 0, 1, 1, 2."""
    cache = np.arange(4 * 2 * 2 * 1 * 1, dtype=np.float64).reshape(4, 2, 2, 1, 1) + 1.0
    k = np.array([[[10.0]], [[20.0]], [[30.0]]])
    v = -k
    so_k = np.array([0, 2, 3])
    po = np.array([0, 2, 2])
    ids = np.array([3, 1])
    last = np.array([1, 1])
    fk = np.array([[[2.0], [3.0], [5.0]], [[7.0], [11.0], [13.0]]])  # [B, 3 blocks, 1 head]
    fv = fk * 10
    ko, vo, co = oracle.dequantize_kv(k, v, cache, fk, fv, "block", so_k, po, ids, last,
                                      block=2)
    # cached: page 3 rows 0, 1 = positions 0, 1 (block 0); page 1 row 0 = position 2 (block 1)
    assert co[3, 0, 0, 0, 0] == 2.0 * cache[3, 0, 0, 0, 0]
    assert co[3, 0, 1, 0, 0] == 2.0 * cache[3, 0, 1, 0, 0]
    assert co[1, 0, 0, 0, 0] == 3.0 * cache[1, 0, 0, 0, 0]
    assert co[1, 1, 0, 0, 0] == 30.0 * cache[1, 1, 0, 0, 0]
    assert co[1, 0, 1, 0, 0] == cache[1, 0, 1, 0, 0]  # past the last page's rows: untouched
    assert co[0, 0, 0, 0, 0] == cache[0, 0, 0, 0, 0]  # a page of no sequence
    # new rows of sequence 0: positions 3 (block 1) and 4 (block 2); sequence 1: position 0
    assert ko[0, 0, 0] == 3.0 * 10.0 and ko[1, 0, 0] == 5.0 * 20.0
    assert ko[2, 0, 0] == 7.0 * 30.0 and vo[2, 0, 0] == 70.0 * -30.0
    # per head: one factor per (sequence, kv head) everywhere
    fh = np.array([[0.5], [4.0]])
    ko, vo, co = oracle.dequantize_kv(k, v, cache, fh, fh, "head", so_k, po, ids, last)
    assert co[1, 1, 0, 0, 0] == 0.5 * cache[1, 1, 0, 0, 0] and ko[2, 0, 0] == 4.0 * 30.0
