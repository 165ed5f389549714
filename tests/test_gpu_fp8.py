"""FP8 E4M3 inputs (feature table, "FP8 quantization types": cast, per-tensor, per-batch,
per-head, per-block): q, k, v as E4M3 with descale factors of each granularity, optional
bf16 rab, both products on the 8-bit tensor cores, P rounded to E4M3 (after scaling by 16)
for the second one, out bf16. Checked against the fp64 oracle run on the dequantized
inputs (the exact values the kernel receives: oracle.dequantize).

Tolerance, derived from the arithmetic: per output row i the kernel's error is at most
  silu_scale * sum_j valid 2^-4 |P_ij| |V_j|     (E4M3 rounding of 16 P: relative 2^-4)
  + silu_scale * sum_j valid 2^-14 c_j |v_j|     (E4M3 subnormals: absolute 2^-10 / 16 in
                                                  units of c_j, the v factor of key j, or
                                                  with block factors the sequence's largest)
  + 2^-8 silu_scale * sum_j |P_ij| |V_j|         (fp32 SiLU with tanh.approx, fp32 sums)
  + 2^-8 |O_i|                                    (bf16 output)
with V_j = c_j v_j the dequantized values, which the tests compute in fp64."""
import numpy as np
import pytest
import torch

import oracle
from hstu_dense_forward_gb300 import hstu_fwd
from hstu_dense_forward_gb300 import workloads as W

pytestmark = pytest.mark.gpu

E4M3 = torch.float8_e4m3fn
BASE = W.WORKLOADS["bf16_causal_b32_s2048_h4_d128"]


def _quant(x, amax_to=224.0):
    """Per-tensor cast: x ~ descale * e4m3(x / descale), descale = max|x| / amax_to."""
    descale = float(x.float().abs().max()) / amax_to
    return (x.float() / descale).to(E4M3), descale


def _case(d, heads, B=3, S=300, causal=True, seed=71, sigma=0.5):
    w = W.scaled(BASE, batch=B, max_seqlen=S, len_lo=1, len_hi=S, dtype="bf16", head_dim=d,
                 num_heads_q=heads[0], num_heads_kv=heads[1], causal=causal, seed=seed,
                 sigma=sigma)
    return w, W.generate(w)


def _bound(qd, kd, vd, so, alpha, silu_scale, causal, nq, nk):
    """Per-row error bound of the module docstring, [T, Nq] (fp64, dense per sequence)."""
    G = nq // nk
    T = qd.shape[0]
    out = np.zeros((T, nq))
    ref_abs = np.zeros((T, nq))
    for b in range(len(so) - 1):
        a, e = int(so[b]), int(so[b + 1])
        L = e - a
        if L == 0:
            continue
        m = np.tril(np.ones((L, L))) if causal else np.ones((L, L))
        for h in range(nq):
            q = qd[a:e, h]
            k = kd[a:e, h // G]
            v = np.abs(vd[a:e, h // G])
            x = alpha * (q @ k.T)
            p = np.abs(x / (1.0 + np.exp(-x))) * m
            pv = (p @ v).max(axis=1)
            out[a:e, h] = silu_scale * ((2.0 ** -4 + 2.0 ** -8) * pv +
                                        2.0 ** -14 * (m @ v).max(axis=1))
    return out


@pytest.mark.parametrize("d,heads,causal", [(128, (4, 4), True), (64, (8, 2), True),
                                            (32, (2, 2), False), (128, (2, 1), False),
                                            (64, (4, 4), False)])
def test_fp8_matches_oracle_within_derived_bound(cuda_device, d, heads, causal):
    w, inp = _case(d, heads, causal=causal)
    q8, sq = _quant(inp["q"])
    k8, sk = _quant(inp["k"])
    v8, sv = _quant(inp["v"])
    dev = cuda_device
    out = hstu_fwd(q8.to(dev), k8.to(dev), v8.to(dev), inp["seq_offsets"].to(dev),
                   max_seqlen=w.max_seqlen, causal=causal, alpha=w.alpha_value,
                   silu_scale=w.silu_scale_value, q_descale=sq, k_descale=sk, v_descale=sv)
    torch.cuda.synchronize()
    assert out.dtype == torch.bfloat16
    qd, kd, vd = (t.double().numpy() * s for t, s in ((q8, sq), (k8, sk), (v8, sv)))
    ref = oracle.hstu_fwd(qd, kd, vd, inp["seq_offsets"],
                          mask_type=oracle.MASK_CAUSAL if causal else oracle.MASK_NONE,
                          alpha=w.alpha_value, silu_scale=w.silu_scale_value,
                          max_seqlen=w.max_seqlen, nthreads=8)
    got = out.double().cpu().numpy()
    T = int(inp["seq_offsets"][-1])
    err = np.abs(got[:T] - ref[:T]).max(axis=2)  # [T, Nq]
    bound = _bound(qd, kd, vd, inp["seq_offsets"].numpy(), w.alpha_value, w.silu_scale_value,
                   causal, heads[0], heads[1])[:T] + 2.0 ** -8 * np.abs(ref[:T]).max(axis=2)
    assert np.all(err <= bound), float((err / bound).max())
    assert np.abs(got[:T] - ref[:T]).max() / np.abs(ref[:T]).max() <= 2.0 ** -4


def test_fp8_targets_gqa_against_oracle(cuda_device):
    """Context and targets with GQA: the global check (error <= 2^-4 of max|O|)."""
    w = W.scaled(W.WORKLOADS["fp16_gqa8x2_targets_b8_s4096_d128"], batch=3, max_seqlen=400,
                 len_lo=50, len_hi=400, dtype="bf16", seed=72)
    inp = W.generate(w)
    q8, k8, v8 = (inp[n].float().to(E4M3) for n in ("q", "k", "v"))
    dev = cuda_device
    out = hstu_fwd(q8.to(dev), k8.to(dev), v8.to(dev), inp["seq_offsets"].to(dev),
                   max_seqlen=w.max_seqlen, num_context=inp["num_context"].to(dev),
                   num_targets=inp["num_targets"].to(dev), target_group_size=w.target_group_size,
                   alpha=w.alpha_value, silu_scale=w.silu_scale_value)
    torch.cuda.synchronize()
    ref = oracle.hstu_fwd(q8, k8, v8, inp["seq_offsets"], num_context=inp["num_context"],
                          num_targets=inp["num_targets"], mask_type=oracle.MASK_CAUSAL,
                          target_group_size=w.target_group_size, alpha=w.alpha_value,
                          silu_scale=w.silu_scale_value, max_seqlen=w.max_seqlen, nthreads=8)
    T = int(inp["seq_offsets"][-1])
    got = out.double().cpu().numpy()
    assert np.abs(got[:T] - ref[:T]).max() / np.abs(ref[:T]).max() <= 2.0 ** -4


def test_fp8_paged_cache_against_oracle(cuda_device):
    """E4M3 KV cache pages and new rows, queries at the end of the keys."""
    from dataclasses import replace
    kw = replace(W.KV_WORKLOADS["bf16_paged_b128_hist1k_4k_h4_d128"], batch=4,
                 hist_range=(100, 600), new_range=(10, 200), page_size=32, seed=73)
    inp = W.generate_kv(kw)
    for n in ("q", "k", "v", "kv_cache"):
        inp[n] = inp[n].float().to(E4M3)
    dev = cuda_device
    dv = {k: (v.to(dev) if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
    out = hstu_fwd(dv["q"], dv["k"], dv["v"], dv["seq_offsets"], max_seqlen=dv["max_seqlen"],
                   max_seqlen_k=dv["max_seqlen_k"], num_targets=dv["num_targets"],
                   target_group_size=1, alpha=dv["alpha"], silu_scale=dv["silu_scale"],
                   seq_offsets_k=dv["seq_offsets_k"], kv_cache=dv["kv_cache"],
                   page_offsets=dv["page_offsets"], page_ids=dv["page_ids"],
                   last_page_len=dv["last_page_len"])
    torch.cuda.synchronize()
    ref = oracle.hstu_fwd(inp["q"], inp["k"], inp["v"], inp["seq_offsets"],
                          seq_offsets_k=inp["seq_offsets_k"], kv_cache=inp["kv_cache"],
                          page_offsets=inp["page_offsets"], page_ids=inp["page_ids"],
                          last_page_len=inp["last_page_len"], num_targets=inp["num_targets"],
                          mask_type=oracle.MASK_CAUSAL, target_group_size=1, alpha=inp["alpha"],
                          silu_scale=inp["silu_scale"], max_seqlen=inp["max_seqlen_k"],
                          nthreads=8)
    got = out.double().cpu().numpy()
    assert np.abs(got - ref).max() / np.abs(ref).max() <= 2.0 ** -4


def test_fp8_full_size_sampled_rows(cuda_device):
    """The FP8 causal workload at full size (B = 32, L ~ U[256, 2048]), sampled rows."""
    w = W.WORKLOADS["fp8_causal_b32_s2048_h4_d128"]
    inp = W.generate(w)
    d = W.to_device(inp, cuda_device)
    out = hstu_fwd(d["q"], d["k"], d["v"], d["seq_offsets"], max_seqlen=w.max_seqlen,
                   alpha=w.alpha_value, silu_scale=w.silu_scale_value)
    torch.cuda.synchronize()
    so = inp["seq_offsets"]
    g = torch.Generator().manual_seed(5)
    rows = []
    for _ in range(64):
        b = int(torch.randint(0, w.batch, (1,), generator=g))
        i = int(torch.randint(0, int(so[b + 1] - so[b]), (1,), generator=g))
        rows.append((b, int(torch.randint(0, w.num_heads_q, (1,), generator=g)), i))
    ref = oracle.hstu_fwd_rows(inp["q"], inp["k"], inp["v"], so, np.array(rows),
                               mask_type=oracle.MASK_CAUSAL, alpha=w.alpha_value,
                               silu_scale=w.silu_scale_value, max_seqlen=w.max_seqlen,
                               nthreads=16)
    sel = torch.stack([out[int(so[b]) + i, h] for b, h, i in rows]).double().cpu().numpy()
    assert np.abs(sel - ref).max() / np.abs(ref).max() <= 2.0 ** -4


def test_fp8_rejects_key_side_rab_and_mask_with_rab(cuda_device):
    from hstu_dense_forward_gb300 import HstuError
    w, inp = _case(64, (2, 2), B=2, S=64)
    q8 = inp["q"].float().to(E4M3).to(cuda_device)
    so = inp["seq_offsets"].to(cuda_device)
    rab = torch.zeros(2, 2, 64, 64, dtype=torch.bfloat16, device=cuda_device)
    with pytest.raises(HstuError):
        hstu_fwd(q8, q8, q8, so, max_seqlen=64, rab=rab, seq_offsets_k=so)
    with pytest.raises(HstuError):
        hstu_fwd(q8, q8, q8, so, max_seqlen=64, rab=rab, mask=torch.ones_like(rab))


@pytest.mark.parametrize("gran", ["cast", "head"])
def test_fp8_custom_mask(cuda_device, gran):
    """A bf16 custom mask (weights in [-1, 2)) with FP8 inputs: P times the mask in fp32,
    then rounded to E4M3; against the oracle on the dequantized values (global bound)."""
    g = torch.Generator().manual_seed(501)
    w, inp = _case(64, (4, 2), B=3, S=264, causal=False, seed=502)
    so = inp["seq_offsets"]
    T = int(so[-1])
    spread = 1.0 if gran == "cast" else 64.0  # (cast: the values themselves are N(0, 1))
    q8, k8, v8 = (_e4m3((T, n, 64), g, spread) for n in (4, 2, 2))
    m = (torch.rand(3, 4, 264, 264, generator=g) * 3.0 - 1.0).to(torch.bfloat16)
    dev = cuda_device
    kw = {}
    if gran == "cast":
        qd, kd, vd = (x.double().numpy() for x in (q8, k8, v8))
    else:
        fq, fk, fv = (_factors("head", 3, n, 3, g) for n in (4, 2, 2))
        kw = dict(q_descale=fq.to(dev), k_descale=fk.to(dev), v_descale=fv.to(dev))
        qd, kd, vd = (oracle.dequantize(x.double().numpy(), f.double().numpy(), "head", so)
                      for x, f in ((q8, fq), (k8, fk), (v8, fv)))
    alpha = w.alpha_value
    out = hstu_fwd(q8.to(dev), k8.to(dev), v8.to(dev), so.to(dev), max_seqlen=264,
                   alpha=alpha, silu_scale=w.silu_scale_value, mask=m.to(dev), **kw)
    torch.cuda.synchronize()
    ref = oracle.hstu_fwd(qd, kd, vd, so, mask=m.double().numpy(), mask_type=oracle.MASK_CUSTOM,
                          alpha=alpha, silu_scale=w.silu_scale_value, max_seqlen=264, nthreads=8)
    got = out.double().cpu().numpy()[:T]
    assert np.abs(got - ref[:T]).max() / np.abs(ref[:T]).max() <= 2.0 ** -4


# ------------------------------------------------ descale granularities, rab, head dims
def _e4m3(shape, g, spread=64.0):
    """Random E4M3 values (normal, sigma = spread) as stored by a scaled cast."""
    return (torch.randn(*shape, generator=g) * spread).clamp(-440, 440).to(E4M3)


def _factors(gran, B, N, nblk, g, lo=-9.0, hi=-5.0):
    """Random descale factors 2^U[lo, hi] of a granularity's shape (fp32, CPU)."""
    shape = {"tensor": (1,), "batch": (B,), "head": (B, N), "block": (B, nblk, N)}[gran]
    return torch.exp2(torch.rand(*shape, generator=g) * (hi - lo) + lo)


def _bound_rows(qd, kd, vd, vsub, so, alpha, silu_scale, causal, nq, nk, rab=None):
    """Per-row error bound of the module docstring [T, Nq] (fp64): vsub [T, Nk, D] is what
    the subnormal term scales (|vd v| per element, or the sequence's largest v factor
    times |v| with block factors, where P carries vd / that factor)."""
    G = nq // nk
    out = np.zeros((qd.shape[0], nq))
    for b in range(len(so) - 1):
        a, e = int(so[b]), int(so[b + 1])
        L = e - a
        if L == 0:
            continue
        m = np.tril(np.ones((L, L))) if causal else np.ones((L, L))
        for h in range(nq):
            x = alpha * (qd[a:e, h] @ kd[a:e, h // G].T)
            if rab is not None:
                x = x + rab[b, h if rab.shape[1] > 1 else 0, :L, :L]
            p = np.abs(x / (1.0 + np.exp(-x))) * m
            out[a:e, h] = silu_scale * ((2.0 ** -4 + 2.0 ** -8) *
                                        (p @ np.abs(vd[a:e, h // G])).max(axis=1) +
                                        2.0 ** -14 * (m @ vsub[a:e, h // G]).max(axis=1))
    return out


def _run_descaled(dev, gran, d, heads, causal, seed, rab_mode=None, S=300, B=3):
    g = torch.Generator().manual_seed(seed)
    w, inp = _case(d, heads, B=B, S=S, causal=causal, seed=seed)
    so = inp["seq_offsets"]
    T = int(so[-1])
    nq, nk = heads
    nblk = -(-S // 128)
    q8, k8, v8 = _e4m3((T, nq, d), g), _e4m3((T, nk, d), g), _e4m3((T, nk, d), g)
    fq = _factors(gran, B, nq, nblk, g)
    fk = _factors(gran, B, nk, nblk, g)
    fv = _factors(gran, B, nk, nblk, g, lo=-10.0, hi=-5.0)  # (block: up to 32x apart)
    qd, kd, vd = (oracle.dequantize(x.double().numpy(), f.double().numpy(), gran, so)
                  for x, f in ((q8, fq), (k8, fk), (v8, fv)))
    rab = None
    if rab_mode is not None:
        rab = (torch.randn(B, 1 if rab_mode == "bcast" else nq, S, S, generator=g) * 0.5
               ).to(torch.bfloat16)
    out = hstu_fwd(q8.to(dev), k8.to(dev), v8.to(dev), so.to(dev), max_seqlen=S,
                   causal=causal, alpha=w.alpha_value, silu_scale=w.silu_scale_value,
                   rab=None if rab is None else rab.to(dev),
                   q_descale=fq.to(dev), k_descale=fk.to(dev), v_descale=fv.to(dev))
    torch.cuda.synchronize()
    assert out.dtype == torch.bfloat16
    rab64 = None if rab is None else rab.double().numpy()
    ref = oracle.hstu_fwd(qd, kd, vd, so, rab=rab64,
                          mask_type=oracle.MASK_CAUSAL if causal else oracle.MASK_NONE,
                          alpha=w.alpha_value, silu_scale=w.silu_scale_value, max_seqlen=S,
                          nthreads=8)
    if gran == "block":  # P carries vd / (the sequence-head's largest v factor)
        vmax = fv.abs().amax(dim=1).double().numpy()  # [B, Nk]
        vsub = np.abs(v8.double().numpy())
        for b in range(B):
            vsub[int(so[b]):int(so[b + 1])] *= vmax[b][None, :, None]
    else:
        vsub = np.abs(vd)
    got = out.double().cpu().numpy()[:T]
    err = np.abs(got - ref[:T]).max(axis=2)
    bound = _bound_rows(qd, kd, vd, vsub, so.numpy(), w.alpha_value, w.silu_scale_value,
                        causal, nq, nk, rab64)[:T] + 2.0 ** -8 * np.abs(ref[:T]).max(axis=2)
    assert np.all(err <= bound), float((err / bound).max())
    assert np.abs(got - ref[:T]).max() / np.abs(ref[:T]).max() <= 2.0 ** -4


@pytest.mark.parametrize("gran", oracle.DESCALE_GRANULARITIES)
@pytest.mark.parametrize("d,heads,causal", [(128, (4, 2), True), (64, (2, 2), False)])
def test_fp8_descale_granularities(cuda_device, gran, d, heads, causal):
    """Descale factors per tensor, sequence, sequence and head, and 128-row block, spread
    over 2^-9 .. 2^-5 (v: 2^-10 .. 2^-5), against the oracle on the dequantized values."""
    _run_descaled(cuda_device, gran, d, heads, causal, seed=200 + d + len(gran))


@pytest.mark.parametrize("gran,d,rab_mode", [("tensor", 128, "full"), ("block", 64, "full"),
                                             ("head", 32, "bcast"), ("batch", 96, "full")])
def test_fp8_with_rab(cuda_device, gran, d, rab_mode):
    """FP8 inputs with a bf16 rab (per head, or one plane broadcast to every head), added
    in fp32 to the SiLU argument: x = alpha (qd q).(kd k) + rab."""
    _run_descaled(cuda_device, gran, d, (4, 2), True, seed=300 + d, rab_mode=rab_mode, S=264)


@pytest.mark.parametrize("d", [16, 48, 80, 112])
def test_fp8_padded_head_dims(cuda_device, d):
    """Head dims between the built 32, 64, 128 (zero-filled extra columns)."""
    _run_descaled(cuda_device, "head", d, (2, 1), True, seed=400 + d)


def test_fp8_descale_shapes_are_checked(cuda_device):
    w, inp = _case(64, (2, 2), B=2, S=64)
    q8 = inp["q"].float().to(E4M3).to(cuda_device)
    so = inp["seq_offsets"].to(cuda_device)
    one = torch.ones(2, 2, dtype=torch.float32, device=cuda_device)
    with pytest.raises(ValueError):  # [B, N] for q, [B] for k and v
        hstu_fwd(q8, q8, q8, so, max_seqlen=64, q_descale=one, k_descale=one[:, 0].contiguous(),
                 v_descale=one[:, 0].contiguous())
    with pytest.raises(ValueError):  # all three or none
        hstu_fwd(q8, q8, q8, so, max_seqlen=64, q_descale=1.0)
    bf = inp["q"].to(cuda_device)
    with pytest.raises(ValueError):  # descales go with FP8 inputs
        hstu_fwd(bf, bf, bf, so, max_seqlen=64, q_descale=1.0, k_descale=1.0, v_descale=1.0)


@pytest.mark.parametrize("gran", ["head", "block"])
def test_fp8_descales_with_paged_cache(cuda_device, gran):
    """Descale factors on the key side: cached pages and new rows take the factor of their
    key position (per block: position // 128, cached history first), queries that of their
    row; against the oracle on the dequantized values (oracle.dequantize_kv)."""
    from dataclasses import replace
    kw = replace(W.KV_WORKLOADS["bf16_paged_b128_hist1k_4k_h4_d128"], batch=4,
                 hist_range=(100, 600), new_range=(10, 200), page_size=32, seed=74)
    inp = W.generate_kv(kw)
    g = torch.Generator().manual_seed(75)
    st = {n: (inp[n].float() * 64).clamp(-440, 440).to(E4M3) for n in ("q", "k", "v", "kv_cache")}
    B, Nq, Nk = kw.batch, kw.num_heads_q, kw.num_heads_kv
    Sq, Sk = int(inp["max_seqlen"]), int(inp["max_seqlen_k"])
    fq = _factors(gran, B, Nq, -(-Sq // 128), g)
    fk = _factors(gran, B, Nk, -(-Sk // 128), g)
    fv = _factors(gran, B, Nk, -(-Sk // 128), g, lo=-10.0, hi=-5.0)
    dev = cuda_device
    dv = {k: (v.to(dev) if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
    out = hstu_fwd(st["q"].to(dev), st["k"].to(dev), st["v"].to(dev), dv["seq_offsets"],
                   max_seqlen=Sq, max_seqlen_k=Sk, num_targets=dv["num_targets"],
                   target_group_size=1, alpha=dv["alpha"], silu_scale=dv["silu_scale"],
                   seq_offsets_k=dv["seq_offsets_k"], kv_cache=st["kv_cache"].to(dev),
                   page_offsets=dv["page_offsets"], page_ids=dv["page_ids"],
                   last_page_len=dv["last_page_len"], q_descale=fq.to(dev), k_descale=fk.to(dev),
                   v_descale=fv.to(dev))
    torch.cuda.synchronize()
    qd = oracle.dequantize(st["q"].double().numpy(), fq.double().numpy(), gran,
                           inp["seq_offsets"])
    kd, vd, cd = oracle.dequantize_kv(st["k"].double().numpy(), st["v"].double().numpy(),
                                      st["kv_cache"].double().numpy(), fk.double().numpy(),
                                      fv.double().numpy(), gran, inp["seq_offsets_k"],
                                      inp["page_offsets"], inp["page_ids"], inp["last_page_len"])
    ref = oracle.hstu_fwd(qd, kd, vd, inp["seq_offsets"], seq_offsets_k=inp["seq_offsets_k"],
                          kv_cache=cd, page_offsets=inp["page_offsets"], page_ids=inp["page_ids"],
                          last_page_len=inp["last_page_len"], num_targets=inp["num_targets"],
                          mask_type=oracle.MASK_CAUSAL, target_group_size=1, alpha=inp["alpha"],
                          silu_scale=inp["silu_scale"], max_seqlen=Sk, nthreads=8)
    T = int(inp["seq_offsets"][-1])
    got = out.double().cpu().numpy()[:T]
    assert np.abs(got - ref[:T]).max() / np.abs(ref[:T]).max() <= 2.0 ** -4
