"""GB300 (sm_103a) HSTU fused attention forward.

    out = hstu_fwd(q, k, v, seq_offsets, max_seqlen=S, causal=True, ...)

computes, per jagged sequence and query head ("RecOps Running Case
Documentation", Introduction to the HSTU_V1 Forward Operator and the feature
table): S = Q K^T scaled by alpha, plus the optional relative attention bias
rab, SiLU, the scaling silu_scale, the causal context/history/target mask or no
mask, and the product with V. MHA and GQA (Nq a multiple of Nk), fp32, fp16 and
bf16. Queries may be fewer than keys (seq_offsets_k: the queries are the last tokens of
their sequences), and the keys may start with a history held in a paged KV cache
(kv_cache, page_offsets, page_ids, last_page_len). The work runs in libhstu_fwd.so (tcgen05/TMA kernels for fp16/bf16, CUDA-core
FFMA for fp32); this module marshals torch tensors to its C ABI and uses torch
only for device memory and the current stream.
"""
from __future__ import annotations

import ctypes

import torch

from . import _abi
from ._abi import HstuError

__all__ = ["hstu_fwd", "hstu_fwd_noalloc", "HstuFwdPlan", "HstuError", "count_pairs",
           "count_pairs_kv", "useful_flops"]

_DTYPES = {torch.float32: _abi.HSTU_F32, torch.float16: _abi.HSTU_F16,
           torch.bfloat16: _abi.HSTU_BF16, torch.float8_e4m3fn: _abi.HSTU_FP8_E4M3}


def out_dtype(dtype: torch.dtype) -> torch.dtype:
    """Element type of out: the input type, bf16 for FP8 E4M3 inputs."""
    return torch.bfloat16 if dtype == torch.float8_e4m3fn else dtype


def _desc(*, dtype, batch, num_heads_q, num_heads_kv, head_dim, max_seqlen, index_is_int64,
          causal, target_group_size, has_rab, has_num_context, has_num_targets, watchdog_ms=0,
          layout="jagged", rab_heads=0, custom_mask=False, is_delta_qk=False, max_seqlen_k=0,
          page_size=0, descale=0):
    d = _abi.Desc()
    d.dtype = _DTYPES[dtype] if isinstance(dtype, torch.dtype) else int(dtype)
    d.batch = int(batch)
    d.num_heads_q = int(num_heads_q)
    d.num_heads_kv = int(num_heads_kv)
    d.head_dim = int(head_dim)
    d.max_seqlen = int(max_seqlen)
    d.index_is_int64 = int(bool(index_is_int64))
    d.mask_type = (_abi.HSTU_MASK_CUSTOM if custom_mask else
                   _abi.HSTU_MASK_CAUSAL if causal else _abi.HSTU_MASK_NONE)
    d.target_group_size = int(target_group_size)
    d.has_rab = int(bool(has_rab))
    d.has_num_context = int(bool(has_num_context))
    d.has_num_targets = int(bool(has_num_targets))
    d.watchdog_ms = int(watchdog_ms)
    if layout not in ("jagged", "normal"):
        raise ValueError(f"layout must be 'jagged' or 'normal', got {layout!r}")
    d.layout = _abi.HSTU_LAYOUT_NORMAL if layout == "normal" else _abi.HSTU_LAYOUT_JAGGED
    d.rab_heads = int(rab_heads)
    d.is_delta_qk = int(bool(is_delta_qk))
    d.max_seqlen_k = int(max_seqlen_k)
    d.page_size = int(page_size)
    d.descale = int(descale)
    return d


def _key_side(d) -> bool:
    return bool(d.is_delta_qk or d.page_size)


def _key_bound(d) -> int:
    """Bound on the keys of a sequence and the S of rab / mask."""
    return d.max_seqlen_k if _key_side(d) and d.max_seqlen_k > 0 else d.max_seqlen


class HstuFwdPlan:
    """One hstu_fwd_plan (validated descriptor + device workspace). Runs on one plan
    must not execute concurrently: keep one plan per stream."""

    def __init__(self, **desc_fields):
        self.desc = _desc(**desc_fields)
        self._keep = _abi.lib()
        h = ctypes.c_void_p()
        _abi.check(self._keep.hstu_fwd_create(ctypes.byref(self.desc), ctypes.byref(h)),
                   "hstu_fwd_create")
        self._h = h

    def run_ptr(self, q, k, v, seq_offsets, rab, num_context, num_targets, total_tokens,
                alpha, silu_scale, out, stream):
        """Raw entry: integer device addresses (0 for absent) and a cudaStream_t value."""
        _abi.check(self._keep.hstu_fwd_run(self._h, q, k, v, seq_offsets or None, rab or None,
                                           num_context or None, num_targets or None,
                                           int(total_tokens), float(alpha), float(silu_scale),
                                           out, stream or None), "hstu_fwd_run")

    def run(self, q, k, v, seq_offsets, out, *, rab=None, num_context=None, num_targets=None,
            alpha=1.0, silu_scale=None, stream=None, mask=None, seq_offsets_k=None,
            kv_cache=None, page_offsets=None, page_ids=None, last_page_len=None, descale=None):
        """descale: (q, k, v) fp32 device tensors of the plan's descale granularity (FP8
        plans whose granularity is not the plain cast)."""
        if silu_scale is None:
            silu_scale = 1.0 / _key_bound(self.desc)
        if stream is None:
            stream = torch.cuda.current_stream(q.device)
        ptr = lambda t: 0 if t is None else t.data_ptr()
        kv = None
        if _key_side(self.desc):
            kv = _abi.KV()
            kv.seq_offsets_k = ptr(seq_offsets_k) or None
            kv.total_tokens_k = k.shape[0] if seq_offsets_k is not None else q.shape[0]
            kv.kv_cache = ptr(kv_cache) or None
            kv.num_pages = 0 if kv_cache is None else kv_cache.shape[0]
            kv.page_offsets = ptr(page_offsets) or None
            kv.page_ids = ptr(page_ids) or None
            kv.last_page_len = ptr(last_page_len) or None
        custom = self.desc.mask_type == _abi.HSTU_MASK_CUSTOM
        if (custom and self.desc.has_rab) or (custom and
                                              self.desc.descale != _abi.HSTU_DESCALE_CAST):
            a = _abi.Args()  # a custom mask with rab or descales: the general entry point
            a.q, a.k, a.v, a.out = q.data_ptr(), ptr(k) or None, ptr(v) or None, out.data_ptr()
            a.seq_offsets = ptr(seq_offsets) or None
            if kv is not None:
                a.kv = ctypes.pointer(kv)
            a.rab, a.mask = ptr(rab) or None, ptr(mask) or None
            a.total_tokens, a.alpha, a.silu_scale = q.shape[0], float(alpha), float(silu_scale)
            if self.desc.descale != _abi.HSTU_DESCALE_CAST:
                ds = _abi.Descale()
                ds.q, ds.k, ds.v = (t.data_ptr() for t in descale)
                a.descale = ctypes.pointer(ds)
            _abi.check(self._keep.hstu_fwd_run_args(self._h, ctypes.byref(a),
                                                    stream.cuda_stream or None),
                       "hstu_fwd_run_args")
            return out
        if self.desc.descale != _abi.HSTU_DESCALE_CAST:
            ds = _abi.Descale()
            ds.q, ds.k, ds.v = (t.data_ptr() for t in descale)
            _abi.check(self._keep.hstu_fwd_run_fp8(
                self._h, q.data_ptr(), ptr(k) or None, ptr(v) or None, ptr(seq_offsets) or None,
                None if kv is None else ctypes.byref(kv), ptr(rab) or None,
                ptr(num_context) or None, ptr(num_targets) or None, ctypes.byref(ds),
                q.shape[0], float(alpha), float(silu_scale), out.data_ptr(),
                stream.cuda_stream or None), "hstu_fwd_run_fp8")
            return out
        if kv is not None:
            extra = mask if self.desc.mask_type == _abi.HSTU_MASK_CUSTOM else rab
            _abi.check(self._keep.hstu_fwd_run_kv(
                self._h, q.data_ptr(), ptr(k) or None, ptr(v) or None, ptr(seq_offsets) or None,
                ctypes.byref(kv), ptr(extra) or None, ptr(num_context) or None,
                ptr(num_targets) or None, q.shape[0], float(alpha), float(silu_scale),
                out.data_ptr(), stream.cuda_stream or None), "hstu_fwd_run_kv")
            return out
        if self.desc.mask_type == _abi.HSTU_MASK_CUSTOM:
            _abi.check(self._keep.hstu_fwd_run_masked(
                self._h, q.data_ptr(), k.data_ptr(), v.data_ptr(), ptr(seq_offsets) or None,
                ptr(mask) or None, q.shape[0], float(alpha), float(silu_scale), out.data_ptr(),
                stream.cuda_stream or None), "hstu_fwd_run_masked")
            return out
        self.run_ptr(q.data_ptr(), k.data_ptr(), v.data_ptr(), ptr(seq_offsets), ptr(rab),
                     ptr(num_context), ptr(num_targets), q.shape[0], alpha, silu_scale,
                     out.data_ptr(), stream.cuda_stream)
        return out

    def get_error(self) -> int:
        """Synchronise; return and clear the device error word (0 = none)."""
        w = ctypes.c_int(0)
        self._keep.hstu_fwd_get_error(self._h, ctypes.byref(w))
        return w.value

    def launches_per_run(self) -> int:
        n = ctypes.c_int(0)
        _abi.check(self._keep.hstu_fwd_launches_per_run(self._h, ctypes.byref(n)),
                   "hstu_fwd_launches_per_run")
        return n.value

    def close(self):
        if getattr(self, "_h", None) is not None and self._h.value:
            self._keep.hstu_fwd_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


_plans: dict = {}


def _check_tensor(t, name, dtype, device, ndim=None):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.device != device:
        raise ValueError(f"{name} must be on {device}, got {t.device}")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if ndim is not None and t.dim() != ndim:
        raise ValueError(f"{name} must have {ndim} dims, got {t.dim()}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def _rab_heads(rab, B, Nq, S):
    """0 for rab [B, Nq, S, S]; 1 for the broadcast form [B, 1, S, S] (feature table,
    "Support for rab broadcasting")."""
    if rab is None:
        return 0
    if rab.shape not in ((B, Nq, S, S), (B, 1, S, S)):
        raise ValueError(f"rab must be [B, Nq, S, S] or [B, 1, S, S] = [{B}, {Nq} or 1, {S}, "
                         f"{S}], got {list(rab.shape)}")
    return 1 if rab.shape[1] == 1 and Nq > 1 else 0


def _descales(q_descale, k_descale, v_descale, *, dev, B, Nq, Nk, Sq, Sk):
    """FP8 descale factors as the C ABI takes them: (granularity, (q, k, v) fp32 device
    tensors), from Python floats or one-element tensors (per tensor), [B] (per sequence),
    q [B, Nq] and k, v [B, Nk] (per sequence and head), or q [B, ceil(Sq / 128), Nq] and
    k, v [B, ceil(Sk / 128), Nk] (per block of 128 query rows / key positions). All
    three None: the plain cast."""
    given = [x is not None for x in (q_descale, k_descale, v_descale)]
    if not any(given):
        return _abi.HSTU_DESCALE_CAST, None
    if not all(given):
        raise ValueError("q_descale, k_descale and v_descale go together")
    ts = []
    for name, x in (("q_descale", q_descale), ("k_descale", k_descale), ("v_descale", v_descale)):
        if isinstance(x, torch.Tensor):
            _check_tensor(x, name, torch.float32, dev)
            ts.append(x)
        else:
            ts.append(torch.tensor([float(x)], dtype=torch.float32, device=dev))
    qd, kd, vd = ts
    if kd.shape != vd.shape:
        raise ValueError("k_descale and v_descale must have one shape")
    cdiv = lambda a, b: -(-a // b)
    if qd.numel() == 1 and qd.dim() <= 1 and kd.numel() == 1 and kd.dim() <= 1:
        return _abi.HSTU_DESCALE_TENSOR, ts
    shapes = {1: ((B,), (B,), _abi.HSTU_DESCALE_BATCH),
              2: ((B, Nq), (B, Nk), _abi.HSTU_DESCALE_HEAD),
              3: ((B, cdiv(Sq, 128), Nq), (B, cdiv(Sk, 128), Nk), _abi.HSTU_DESCALE_BLOCK)}
    want = shapes.get(qd.dim())
    if want is None or tuple(qd.shape) != want[0] or tuple(kd.shape) != want[1]:
        raise ValueError(f"descale shapes q {list(qd.shape)}, k/v {list(kd.shape)} match no "
                         "granularity (one factor, [B], [B, N] or [B, ceil(S/128), N])")
    return want[2], ts


def hstu_fwd(q, k, v, seq_offsets=None, *, max_seqlen=None, rab=None, num_context=None,
             num_targets=None, causal=True, target_group_size=0, alpha=1.0, silu_scale=None,
             out=None, watchdog_ms=0, layout="jagged", mask=None, seq_offsets_k=None,
             max_seqlen_k=None, kv_cache=None, page_offsets=None, page_ids=None,
             last_page_len=None, q_descale=None, k_descale=None, v_descale=None):
    """HSTU forward.

    layout "jagged" (default): q [T, Nq, D], k/v [T, Nk, D], seq_offsets [B+1] int32/int64,
    max_seqlen required. layout "normal" (Inputs and Outputs table, layout): q [B, S, Nq, D],
    k/v [B, S, Nk, D], every sequence of S tokens, no seq_offsets, max_seqlen = S.
    Same dtype for q, k, v: fp32, fp16 or bf16. num_context / num_targets [B] of the index
    dtype (int32/int64). rab [B, Nq, S, S] or [B, 1, S, S] (one plane for all heads) of q's
    dtype, or None. causal=False is mask_type 2 (no mask). mask [B, Nq, S, S] of q's dtype
    selects mask_type 3 (custom mask: P is multiplied by it after the SiLU; no context or
    target counts with it; rab, added before the SiLU, may come with it). silu_scale defaults to 1/max_seqlen. Returns out with q's
    shape; rows that belong to no sequence are left as allocated.

    Key side (jagged layout; Inputs and Outputs table, seq_offsets_k / kv_cache rows):
    seq_offsets_k [B+1] gives the new k/v rows of each sequence (k, v [Tk, Nk, D]; without
    it they are the query rows). kv_cache [num_pages, 2, page_size, Nk, D] (q's dtype; plane
    0 K, plane 1 V; page_size 32, 128 or 256) with page_offsets [B+1], page_ids and
    last_page_len [B] holds a history that precedes the new rows. The Lq queries of a
    sequence are the last Lq of its Lk keys; max_seqlen bounds Lq, max_seqlen_k (default
    max_seqlen) bounds Lk and is the S of rab and mask; silu_scale then defaults to
    1/max_seqlen_k.

    FP8 (feature table, "FP8 quantization types"): q, k, v (and kv_cache) of dtype
    torch.float8_e4m3fn, out bf16; rab (no key side) bf16. q_descale, k_descale, v_descale
    (all or none; none is the plain cast) give the values as factor * stored value: floats
    or one-element fp32 tensors (per tensor), [B] (per sequence), q [B, Nq] and k, v
    [B, Nk] (per sequence and head), q [B, ceil(max_seqlen / 128), Nq] and k, v
    [B, ceil(Sk / 128), Nk] (per block of 128 query rows / key positions). Head dims up to
    128; no custom mask.
    """
    dev = q.device
    if dev.type != "cuda":
        raise ValueError("hstu_fwd runs on CUDA tensors only")
    if q.dtype not in _DTYPES:
        raise TypeError(f"unsupported dtype {q.dtype}")
    if layout == "normal":
        _check_tensor(q, "q", None, dev, 4)
        _check_tensor(k, "k", q.dtype, dev, 4)
        _check_tensor(v, "v", q.dtype, dev, 4)
        if seq_offsets is not None:
            raise ValueError("the normal layout takes no seq_offsets")
        B, S = q.shape[0], q.shape[1]
        if max_seqlen is None:
            max_seqlen = S
        elif int(max_seqlen) != S:
            raise ValueError(f"the normal layout needs max_seqlen == S = {S}")
        if k.shape != v.shape or k.shape[:2] != q.shape[:2] or k.shape[3] != q.shape[3]:
            raise ValueError("k and v must be [B, S, Nk, D] with q's B, S and D")
        idx = [t for t in (num_context, num_targets) if t is not None]
        idx_dtype = idx[0].dtype if idx else torch.int64
        res = out
        if res is None:
            res = torch.empty(q.shape, dtype=out_dtype(q.dtype), device=dev)
        else:
            _check_tensor(res, "out", out_dtype(q.dtype), dev, 4)
            if res.shape != q.shape:
                raise ValueError("out must have q's shape")
        q3, k3, v3 = q.view(B * S, *q.shape[2:]), k.view(B * S, *k.shape[2:]), v.view(B * S, *v.shape[2:])
        out3 = res.view(B * S, *q.shape[2:])
    elif layout == "jagged":
        _check_tensor(q, "q", None, dev, 3)
        _check_tensor(k, "k", q.dtype, dev, 3)
        _check_tensor(v, "v", q.dtype, dev, 3)
        if seq_offsets is None or max_seqlen is None:
            raise ValueError("the jagged layout needs seq_offsets and max_seqlen")
        _check_tensor(seq_offsets, "seq_offsets", None, dev, 1)
        idx_dtype = seq_offsets.dtype
        rows_k = k.shape[0] if seq_offsets_k is not None else q.shape[0]
        if k.shape != v.shape or k.shape[0] != rows_k or k.shape[2] != q.shape[2]:
            raise ValueError("k and v must be [T, Nk, D] with q's T and D (or [Tk, Nk, D] "
                             "with seq_offsets_k)")
        B = seq_offsets.shape[0] - 1
        if out is None:
            out = torch.empty(q.shape, dtype=out_dtype(q.dtype), device=dev)
        else:
            _check_tensor(out, "out", out_dtype(q.dtype), dev, 3)
            if out.shape != q.shape:
                raise ValueError("out must have q's shape")
        q3, k3, v3, out3, res = q, k, v, out, out
    else:
        raise ValueError(f"layout must be 'jagged' or 'normal', got {layout!r}")
    if idx_dtype not in (torch.int32, torch.int64):
        raise TypeError("index tensors must be int32 or int64")
    for name, t in (("num_context", num_context), ("num_targets", num_targets),
                    ("seq_offsets_k", seq_offsets_k), ("page_offsets", page_offsets),
                    ("page_ids", page_ids), ("last_page_len", last_page_len)):
        if t is not None:
            _check_tensor(t, name, idx_dtype, dev, 1)
    T, Nq, D = q3.shape
    page_size = 0
    if kv_cache is not None:
        _check_tensor(kv_cache, "kv_cache", q.dtype, dev, 5)
        if kv_cache.shape[1] != 2 or tuple(kv_cache.shape[3:]) != (k3.shape[1], D):
            raise ValueError("kv_cache must be [num_pages, 2, page_size, Nk, D]")
        if page_offsets is None or page_ids is None or last_page_len is None:
            raise ValueError("kv_cache needs page_offsets, page_ids and last_page_len")
        page_size = kv_cache.shape[2]
    elif page_offsets is not None or page_ids is not None or last_page_len is not None:
        raise ValueError("a page table needs kv_cache")
    key_side = seq_offsets_k is not None or kv_cache is not None
    if key_side and layout != "jagged":
        raise ValueError("seq_offsets_k and kv_cache need the jagged layout")
    if max_seqlen_k is not None and not key_side:
        raise ValueError("max_seqlen_k goes with seq_offsets_k or kv_cache")
    Sk = int(max_seqlen_k) if max_seqlen_k is not None else int(max_seqlen)
    if rab is not None:
        _check_tensor(rab, "rab", out_dtype(q.dtype), dev, 4)  # (bf16 for FP8 inputs)
    rab_heads = _rab_heads(rab, B, Nq, Sk)
    if q.dtype == torch.float8_e4m3fn:
        descale, ds = _descales(q_descale, k_descale, v_descale, dev=dev, B=B, Nq=Nq,
                                Nk=k3.shape[1], Sq=int(max_seqlen), Sk=Sk)
    elif (q_descale, k_descale, v_descale) != (None, None, None):
        raise ValueError("descale factors go with FP8 E4M3 inputs")
    else:
        descale, ds = _abi.HSTU_DESCALE_CAST, None
    custom = mask is not None
    if custom:
        if num_context is not None or num_targets is not None:
            raise ValueError("a custom mask takes no num_context or num_targets")
        _check_tensor(mask, "mask", out_dtype(q.dtype), dev, 4)  # (bf16 for FP8 inputs)
        if tuple(mask.shape) != (B, Nq, Sk, Sk):
            raise ValueError(f"mask must be [B, Nq, S, S], got {list(mask.shape)}")
    stream = torch.cuda.current_stream(dev)
    key = (dev.index, stream.cuda_stream, q.dtype, B, Nq, k3.shape[1], D, int(max_seqlen),
           idx_dtype, bool(causal), int(target_group_size), rab is not None,
           num_context is not None, num_targets is not None, int(watchdog_ms), layout, rab_heads,
           custom, seq_offsets_k is not None, page_size, Sk if key_side else 0, descale)
    plan = _plans.get(key)
    if plan is None:
        with torch.cuda.device(dev):
            plan = HstuFwdPlan(dtype=q.dtype, batch=B, num_heads_q=Nq, num_heads_kv=k3.shape[1],
                               head_dim=D, max_seqlen=max_seqlen,
                               index_is_int64=idx_dtype == torch.int64, causal=causal,
                               target_group_size=target_group_size, has_rab=rab is not None,
                               has_num_context=num_context is not None,
                               has_num_targets=num_targets is not None, watchdog_ms=watchdog_ms,
                               layout=layout, rab_heads=rab_heads, custom_mask=custom,
                               is_delta_qk=seq_offsets_k is not None,
                               max_seqlen_k=Sk if key_side else 0, page_size=page_size,
                               descale=descale)
        _plans[key] = plan
    with torch.cuda.device(dev):
        plan.run(q3, k3, v3, seq_offsets, out3, rab=rab, num_context=num_context,
                 num_targets=num_targets, alpha=alpha, silu_scale=silu_scale, stream=stream,
                 mask=mask, seq_offsets_k=seq_offsets_k, kv_cache=kv_cache,
                 page_offsets=page_offsets, page_ids=page_ids, last_page_len=last_page_len,
                 descale=ds)
    return res


def hstu_fwd_noalloc(q, k, v, seq_offsets, out, *, max_seqlen=None, rab=None,
                     num_context=None, num_targets=None, causal=True, target_group_size=0,
                     alpha=1.0, silu_scale=None, layout="jagged"):
    """hstu_fwd through the library's allocation-free entry point (hstu_fwd_run_noalloc):
    no plan, the work list lives in a fixed device array of the library. `out` must be
    given (this call allocates nothing, torch included). Calls that may overlap on the GPU
    share that array and must be serialised by the caller. Arguments as for hstu_fwd
    (jagged or normal layout; fp32, fp16 or bf16; no custom mask, key side or FP8)."""
    dev = q.device
    if dev.type != "cuda":
        raise ValueError("hstu_fwd_noalloc runs on CUDA tensors only")
    if q.dtype not in (torch.float32, torch.float16, torch.bfloat16):
        raise TypeError(f"hstu_fwd_noalloc takes fp32, fp16 or bf16 inputs, got {q.dtype}")
    if layout == "normal":
        for name, t in (("q", q), ("k", k), ("v", v), ("out", out)):
            _check_tensor(t, name, q.dtype, dev, 4)
        if seq_offsets is not None:
            raise ValueError("the normal layout takes no seq_offsets")
        B, S = q.shape[0], q.shape[1]
        if max_seqlen is None:
            max_seqlen = S
        elif int(max_seqlen) != S:
            raise ValueError(f"the normal layout needs max_seqlen == S = {S}")
        if k.shape != v.shape or k.shape[:2] != q.shape[:2] or k.shape[3] != q.shape[3]:
            raise ValueError("k and v must be [B, S, Nk, D] with q's B, S and D")
        if out.shape != q.shape:
            raise ValueError("out must have q's shape")
        idx = [t for t in (num_context, num_targets) if t is not None]
        idx_dtype = idx[0].dtype if idx else torch.int64
        Nq, Nk, D, T = q.shape[2], k.shape[2], q.shape[3], B * S
    elif layout == "jagged":
        for name, t in (("q", q), ("k", k), ("v", v), ("out", out)):
            _check_tensor(t, name, q.dtype, dev, 3)
        if seq_offsets is None or max_seqlen is None:
            raise ValueError("the jagged layout needs seq_offsets and max_seqlen")
        _check_tensor(seq_offsets, "seq_offsets", None, dev, 1)
        if k.shape != v.shape or k.shape[0] != q.shape[0] or k.shape[2] != q.shape[2]:
            raise ValueError("k and v must be [T, Nk, D] with q's T and D")
        if out.shape != q.shape:
            raise ValueError("out must have q's shape")
        idx_dtype = seq_offsets.dtype
        B = seq_offsets.shape[0] - 1
        T, Nq, D = q.shape
        Nk = k.shape[1]
    else:
        raise ValueError(f"layout must be 'jagged' or 'normal', got {layout!r}")
    if idx_dtype not in (torch.int32, torch.int64):
        raise TypeError("index tensors must be int32 or int64")
    for name, t in (("num_context", num_context), ("num_targets", num_targets)):
        if t is not None:
            _check_tensor(t, name, idx_dtype, dev, 1)
            if t.shape[0] != B:
                raise ValueError(f"{name} must have B = {B} entries")
    if rab is not None:
        _check_tensor(rab, "rab", q.dtype, dev, 4)
    d = _desc(dtype=q.dtype, batch=B, num_heads_q=Nq, num_heads_kv=Nk, head_dim=D,
              max_seqlen=max_seqlen, index_is_int64=idx_dtype == torch.int64, causal=causal,
              target_group_size=target_group_size, has_rab=rab is not None,
              has_num_context=num_context is not None, has_num_targets=num_targets is not None,
              layout=layout, rab_heads=_rab_heads(rab, B, Nq, int(max_seqlen)))
    if silu_scale is None:
        silu_scale = 1.0 / max_seqlen
    ptr = lambda t: None if t is None else t.data_ptr()
    with torch.cuda.device(dev):
        stream = torch.cuda.current_stream(dev)
        _abi.check(_abi.lib().hstu_fwd_run_noalloc(
            ctypes.byref(d), q.data_ptr(), k.data_ptr(), v.data_ptr(), ptr(seq_offsets),
            ptr(rab), ptr(num_context), ptr(num_targets), T, float(alpha),
            float(silu_scale), out.data_ptr(), stream.cuda_stream), "hstu_fwd_run_noalloc")
    return out


def plan_for(**kw) -> HstuFwdPlan:
    """A fresh plan (see HstuFwdPlan); keyword arguments as the descriptor fields."""
    return HstuFwdPlan(**kw)


def count_pairs(seq_offsets, num_heads_q, *, max_seqlen, num_context=None, num_targets=None,
                causal=True, target_group_size=0, layout="jagged", batch=None) -> int:
    """Mask-aware (query head, i, j) pair count, computed by the library on the host
    from CPU integer tensors or sequences. For layout "normal" pass seq_offsets=None and
    batch=B (every sequence has max_seqlen tokens)."""
    so = None if seq_offsets is None else torch.as_tensor(seq_offsets, dtype=torch.int64).contiguous().cpu()
    nc = None if num_context is None else torch.as_tensor(num_context, dtype=torch.int64).contiguous().cpu()
    nt = None if num_targets is None else torch.as_tensor(num_targets, dtype=torch.int64).contiguous().cpu()
    B = int(batch) if so is None else so.numel() - 1
    d = _desc(dtype=_abi.HSTU_BF16, batch=B, num_heads_q=num_heads_q,
              num_heads_kv=1, head_dim=64, max_seqlen=max_seqlen, index_is_int64=True,
              causal=causal, target_group_size=target_group_size, has_rab=False,
              has_num_context=nc is not None, has_num_targets=nt is not None, layout=layout)
    out = ctypes.c_longlong(0)
    ptr = lambda t: None if t is None else ctypes.c_void_p(t.data_ptr())
    _abi.check(_abi.lib().hstu_fwd_count_pairs(ctypes.byref(d), ptr(so), ptr(nc), ptr(nt),
                                               ctypes.byref(out)), "hstu_fwd_count_pairs")
    return int(out.value)


def count_pairs_kv(seq_offsets, num_heads_q, *, max_seqlen, seq_offsets_k=None,
                   page_offsets=None, last_page_len=None, page_size=0, max_seqlen_k=None,
                   num_context=None, num_targets=None, causal=True, target_group_size=0) -> int:
    """count_pairs for calls whose queries are the last tokens of longer key sequences
    (seq_offsets_k and / or a KV cache page table), from CPU integer data."""
    t64 = lambda x: None if x is None else torch.as_tensor(x, dtype=torch.int64).contiguous().cpu()
    so, sok, po, last = t64(seq_offsets), t64(seq_offsets_k), t64(page_offsets), t64(last_page_len)
    nc, nt = t64(num_context), t64(num_targets)
    key_side = sok is not None or po is not None
    d = _desc(dtype=_abi.HSTU_BF16, batch=so.numel() - 1, num_heads_q=num_heads_q,
              num_heads_kv=1, head_dim=64, max_seqlen=max_seqlen, index_is_int64=True,
              causal=causal, target_group_size=target_group_size, has_rab=False,
              has_num_context=nc is not None, has_num_targets=nt is not None,
              is_delta_qk=sok is not None,
              max_seqlen_k=(max_seqlen_k or 0) if key_side else 0, page_size=page_size)
    out = ctypes.c_longlong(0)
    ptr = lambda t: None if t is None else ctypes.c_void_p(t.data_ptr())
    _abi.check(_abi.lib().hstu_fwd_count_pairs_kv(ctypes.byref(d), ptr(so), ptr(sok), ptr(po),
                                                  ptr(last), ptr(nc), ptr(nt),
                                                  ctypes.byref(out)), "hstu_fwd_count_pairs_kv")
    return int(out.value)


def useful_flops(pairs: int, head_dim: int) -> int:
    """Mask-aware useful flops: 2*D for Q.K and 2*D for P.V per valid pair."""
    return 4 * int(head_dim) * int(pairs)
