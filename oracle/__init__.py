"""fp64 CPU oracle for the HSTU fused attention forward.

TEST INFRASTRUCTURE ONLY: imported by ``tests/``, by ``__graft_entry__.smoke()``
and by the CPU-baseline leg of ``bench.py``; the product package never imports
it. The arithmetic lives in ``hstu_oracle.c`` (plain C, fp64 loops, in the
operation order of "RecOps Running Case Documentation", Introduction to the
HSTU_V1 Forward Operator: QK matmul, SiLU, scaling, mask, matmul with V). This
module only builds that file with gcc and marshals arrays to it.

Inputs are upcast to float64 exactly (every bf16/fp16/fp32 value is a double).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "hstu_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

MASK_CAUSAL = 0  # Inputs and Outputs table: "0: built-in lower triangular mask"
MASK_NONE = 2  # "2: do not use a mask"
MASK_CUSTOM = 3  # "3: use a custom mask ... the user must define and pass in the mask"


def build(force: bool = False) -> str:
    """Compile hstu_oracle.c into liboracle.so beside it (gcc, -O2, pthreads)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(
            ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-o", tmp, _SRC, "-lm", "-lpthread"]
        )
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            _lib = _bind(ctypes.CDLL(_LIB))
    return _lib


class use_library:
    """Context manager that points this module at another build of the oracle
    source (the mutation tests compile deliberately broken copies)."""

    def __init__(self, path):
        self._path = path

    def __enter__(self):
        global _lib
        _load()
        self._saved = _lib
        _lib = _bind(ctypes.CDLL(self._path))
        return self

    def __exit__(self, *exc):
        global _lib
        _lib = self._saved
        return False


def _bind(lib):
    d = ctypes.POINTER(ctypes.c_double)
    i64 = ctypes.POINTER(ctypes.c_int64)
    c64 = ctypes.c_int64
    lib.hstu_oracle_valid.restype = ctypes.c_int
    lib.hstu_oracle_valid.argtypes = [c64, c64, c64, ctypes.c_int, c64, c64, c64]
    kv = [i64, d, c64, i64, i64, i64, c64]  # seq_offsets_k, kv_cache, num_pages, page table
    lib.hstu_oracle_fwd.restype = ctypes.c_int
    lib.hstu_oracle_fwd.argtypes = [d, d, d, i64, c64, c64, c64, c64, d, c64, d, c64] + kv + [
        i64, i64, ctypes.c_int, c64, ctypes.c_double, ctypes.c_double, d, ctypes.c_int]
    lib.hstu_oracle_fwd_rows.restype = ctypes.c_int
    lib.hstu_oracle_fwd_rows.argtypes = [d, d, d, i64, c64, c64, c64, c64, d, c64, d,
                                         c64] + kv + [i64, i64, ctypes.c_int, c64,
                                                      ctypes.c_double, ctypes.c_double, i64,
                                                      c64, d, ctypes.c_int]
    lib.hstu_oracle_count_valid.restype = ctypes.c_int64
    lib.hstu_oracle_count_valid.argtypes = [i64, c64, c64, i64, i64, ctypes.c_int, c64]
    lib.hstu_oracle_count_valid_kv.restype = ctypes.c_int64
    lib.hstu_oracle_count_valid_kv.argtypes = [i64, i64, c64, c64, i64, i64, ctypes.c_int, c64]
    return lib


def _f64(x):
    if x is None:
        return None
    if hasattr(x, "detach"):  # torch tensor: exact upcast on the CPU
        x = x.detach().to("cpu").double().numpy()
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _i64(x):
    if x is None:
        return None
    if hasattr(x, "detach"):
        x = x.detach().to("cpu").numpy()
    return np.ascontiguousarray(np.asarray(x, dtype=np.int64))


def _p(a, ty):
    return None if a is None else a.ctypes.data_as(ctypes.POINTER(ty))


class _KV:
    """Key side of a call: offsets of the new k/v rows and the paged history."""

    def __init__(self, B, nk, d, seq_offsets_k, kv_cache, page_offsets, page_ids,
                 last_page_len):
        self.so_k = _i64(seq_offsets_k)
        if self.so_k is not None and self.so_k.shape != (B + 1,):
            raise ValueError("seq_offsets_k must be [B+1]")
        self.cache = _f64(kv_cache)
        self.num_pages, self.page_size = 0, 0
        self.po = self.ids = self.last = None
        if self.cache is not None:
            if self.cache.ndim != 5 or self.cache.shape[1] != 2 or \
                    self.cache.shape[3:] != (nk, d):
                raise ValueError("kv_cache must be [num_pages, 2, page_size, Nk, D]")
            self.num_pages, self.page_size = self.cache.shape[0], self.cache.shape[2]
            self.po, self.ids = _i64(page_offsets), _i64(page_ids)
            self.last = _i64(last_page_len)
            if self.po is None or self.ids is None or self.last is None or \
                    self.po.shape != (B + 1,) or self.last.shape != (B,):
                raise ValueError("page_offsets [B+1], page_ids and last_page_len [B] "
                                 "go with kv_cache")
            if self.ids.size < int(self.po[-1]):
                raise ValueError("page_ids shorter than page_offsets[B]")

    def args(self):
        return [_p(self.so_k, ctypes.c_int64), _p(self.cache, ctypes.c_double),
                self.num_pages, _p(self.po, ctypes.c_int64), _p(self.ids, ctypes.c_int64),
                _p(self.last, ctypes.c_int64), self.page_size]


def history_lengths(page_offsets, last_page_len, page_size):
    """Cached rows per sequence: (pages - 1) * page_size + last_page_len, 0 without pages."""
    po, last = _i64(page_offsets), _i64(last_page_len)
    pages = np.diff(po)
    return np.where(pages > 0, (pages - 1) * page_size + last, 0)


def _common(q, k, v, seq_offsets, rab, num_context, num_targets, max_seqlen, mask=None,
            mask_type=MASK_CAUSAL):
    q, k, v = _f64(q), _f64(k), _f64(v)
    so = _i64(seq_offsets)
    if q.ndim != 3 or k.ndim != 3 or v.shape != k.shape or q.shape[2] != k.shape[2]:
        raise ValueError("q [T, Nq, D], k/v [Tk, Nk, D] expected")
    B = so.shape[0] - 1
    nc, nt = _i64(num_context), _i64(num_targets)
    rab = _f64(rab)
    rab_heads = 0
    if rab is not None:
        if max_seqlen is None:
            raise ValueError("max_seqlen is required with rab")
        if rab.ndim != 4 or rab.shape[1] not in (1, q.shape[1]) or \
                rab.shape != (B, rab.shape[1], max_seqlen, max_seqlen):
            raise ValueError(f"rab must be [B, Nq, S, S] or [B, 1, S, S], got {rab.shape}")
        rab_heads = rab.shape[1]
    mask = _f64(mask)
    if (mask is not None) != (mask_type == MASK_CUSTOM):
        raise ValueError("a mask tensor is passed exactly with mask_type MASK_CUSTOM")
    if mask is not None and (max_seqlen is None or
                             mask.shape != (B, q.shape[1], max_seqlen, max_seqlen)):
        raise ValueError("mask must be [B, Nq, S, S] with S = max_seqlen")
    return q, k, v, so, B, rab, rab_heads, nc, nt, mask


def _key_lengths(so, kv):
    so_k = kv.so_k if kv.so_k is not None else so
    lk = np.diff(so_k)
    if kv.cache is not None:
        lk = lk + history_lengths(kv.po, kv.last, kv.page_size)
    return lk


def hstu_fwd(q, k, v, seq_offsets, *, rab=None, num_context=None, num_targets=None,
             mask_type=MASK_CAUSAL, target_group_size=0, alpha=1.0, silu_scale=None,
             max_seqlen=None, nthreads=1, mask=None, seq_offsets_k=None, kv_cache=None,
             page_offsets=None, page_ids=None, last_page_len=None):
    """Whole forward in fp64. Returns out [T, Nq, D] as float64 (rows outside
    every sequence are 0). silu_scale defaults to 1/max_seqlen (Inputs and
    Outputs table, silu_scale). max_seqlen is the key-side bound (the S of rab and
    mask); with seq_offsets_k and/or a kv_cache the keys of a sequence are its cached
    history followed by its new k/v rows, and its queries are the last ones."""
    q, k, v, so, B, rab, rab_heads, nc, nt, mask = _common(
        q, k, v, seq_offsets, rab, num_context, num_targets, max_seqlen, mask, mask_type)
    kv = _KV(B, k.shape[1], k.shape[2], seq_offsets_k, kv_cache, page_offsets, page_ids,
             last_page_len)
    if max_seqlen is None:
        max_seqlen = int(np.max(_key_lengths(so, kv))) if B > 0 else 1
    if silu_scale is None:
        silu_scale = 1.0 / max_seqlen
    out = np.zeros(q.shape, dtype=np.float64)
    rc = _load().hstu_oracle_fwd(_p(q, ctypes.c_double), _p(k, ctypes.c_double),
                                 _p(v, ctypes.c_double), _p(so, ctypes.c_int64), B, q.shape[1],
                                 k.shape[1], q.shape[2], _p(rab, ctypes.c_double), rab_heads,
                                 _p(mask, ctypes.c_double), max_seqlen, *kv.args(),
                                 _p(nc, ctypes.c_int64), _p(nt, ctypes.c_int64), mask_type,
                                 target_group_size, float(alpha), float(silu_scale),
                                 _p(out, ctypes.c_double), int(nthreads))
    if rc != 0:
        raise ValueError("oracle rejected its arguments")
    return out


def hstu_fwd_rows(q, k, v, seq_offsets, rows, *, rab=None, num_context=None, num_targets=None,
                  mask_type=MASK_CAUSAL, target_group_size=0, alpha=1.0, silu_scale=None,
                  max_seqlen=None, nthreads=1, mask=None, seq_offsets_k=None, kv_cache=None,
                  page_offsets=None, page_ids=None, last_page_len=None):
    """Selected output rows: rows is an int array [n, 3] of (b, h, i) (i local to
    sequence b). Returns [n, D] float64, row r = out[seq_offsets[b] + i, h, :]."""
    q, k, v, so, B, rab, rab_heads, nc, nt, mask = _common(
        q, k, v, seq_offsets, rab, num_context, num_targets, max_seqlen, mask, mask_type)
    kv = _KV(B, k.shape[1], k.shape[2], seq_offsets_k, kv_cache, page_offsets, page_ids,
             last_page_len)
    if max_seqlen is None:
        max_seqlen = int(np.max(_key_lengths(so, kv))) if B > 0 else 1
    if silu_scale is None:
        silu_scale = 1.0 / max_seqlen
    rows = np.ascontiguousarray(np.asarray(rows, dtype=np.int64).reshape(-1, 3))
    out = np.zeros((rows.shape[0], q.shape[2]), dtype=np.float64)
    rc = _load().hstu_oracle_fwd_rows(_p(q, ctypes.c_double), _p(k, ctypes.c_double),
                                      _p(v, ctypes.c_double), _p(so, ctypes.c_int64), B,
                                      q.shape[1], k.shape[1], q.shape[2],
                                      _p(rab, ctypes.c_double), rab_heads,
                                      _p(mask, ctypes.c_double), max_seqlen, *kv.args(),
                                      _p(nc, ctypes.c_int64), _p(nt, ctypes.c_int64), mask_type,
                                      target_group_size, float(alpha), float(silu_scale),
                                      _p(rows, ctypes.c_int64), rows.shape[0],
                                      _p(out, ctypes.c_double), int(nthreads))
    if rc != 0:
        raise ValueError("oracle rejected its arguments")
    return out


DESCALE_GRANULARITIES = ("tensor", "batch", "head", "block")


def dequantize(x, descale, granularity, seq_offsets, *, block=128):
    """Values of FP8 inputs with descale factors (feature table, "FP8 quantization types":
    per-tensor, per-batch, per-head, per-block): element (t, n, d) of the jagged tensor x
    [T, N, D] is factor * x[t, n, d], with the factor of its sequence b (seq_offsets[b] <=
    t < seq_offsets[b + 1]), head n and block (t - seq_offsets[b]) // block:
      "tensor" descale [1]; "batch" [B]; "head" [B, N]; "block" [B, nblocks, N].
    Rows outside every sequence become 0. Plain loops, fp64."""
    x = _f64(x)
    so = _i64(seq_offsets)
    f = np.asarray(descale, dtype=np.float64)
    if granularity not in DESCALE_GRANULARITIES:
        raise ValueError(f"granularity must be one of {DESCALE_GRANULARITIES}")
    out = np.zeros_like(x)
    for b in range(so.shape[0] - 1):
        for t in range(int(so[b]), int(so[b + 1])):
            i = t - int(so[b])  # position within the sequence
            for n in range(x.shape[1]):
                if granularity == "tensor":
                    c = f.reshape(-1)[0]
                elif granularity == "batch":
                    c = f[b]
                elif granularity == "head":
                    c = f[b, n]
                else:
                    c = f[b, i // block, n]
                out[t, n] = c * x[t, n]
    return out


def dequantize_kv(k, v, kv_cache, k_descale, v_descale, granularity, seq_offsets_k,
                  page_offsets, page_ids, last_page_len, *, block=128):
    """FP8 descale factors on the key side: the keys of sequence b are its cached history
    (pages page_ids[page_offsets[b]] .. in order, rows of each page, the last one holding
    last_page_len[b] rows) followed by its new rows k/v [seq_offsets_k[b] ..). Key position
    p (0 for the first cached row) takes the factor of (b, p // block, kv head) ("block"),
    (b, kv head) ("head"), b ("batch") or the one factor ("tensor"). Returns the values
    (k, v, kv_cache) in fp64; cache rows that belong to no sequence keep their stored
    values (they are never read as keys). Plain loops."""
    k, v, cache = _f64(k), _f64(v), _f64(kv_cache)
    so = _i64(seq_offsets_k)
    po, ids, last = _i64(page_offsets), _i64(page_ids), _i64(last_page_len)
    fk = np.asarray(k_descale, dtype=np.float64)
    fv = np.asarray(v_descale, dtype=np.float64)
    if granularity not in DESCALE_GRANULARITIES:
        raise ValueError(f"granularity must be one of {DESCALE_GRANULARITIES}")
    page_size = cache.shape[2]

    def factor(f, b, pos, h):
        if granularity == "tensor":
            return f.reshape(-1)[0]
        if granularity == "batch":
            return f[b]
        if granularity == "head":
            return f[b, h]
        return f[b, pos // block, h]

    ko, vo, co = k.copy(), v.copy(), cache.copy()
    for b in range(so.shape[0] - 1):
        pages = [int(x) for x in ids[int(po[b]):int(po[b + 1])]]
        hist = 0
        for s_, pg in enumerate(pages):
            rows = page_size if s_ + 1 < len(pages) else int(last[b])
            for r in range(rows):
                pos = s_ * page_size + r
                for h in range(cache.shape[3]):
                    co[pg, 0, r, h] = factor(fk, b, pos, h) * cache[pg, 0, r, h]
                    co[pg, 1, r, h] = factor(fv, b, pos, h) * cache[pg, 1, r, h]
            hist += rows
        for t in range(int(so[b]), int(so[b + 1])):
            pos = hist + t - int(so[b])
            for h in range(k.shape[1]):
                ko[t, h] = factor(fk, b, pos, h) * k[t, h]
                vo[t, h] = factor(fv, b, pos, h) * v[t, h]
    return ko, vo, co


def valid(i, j, L, mask_type=MASK_CAUSAL, num_context=0, num_targets=0, target_group_size=0):
    """The oracle's mask predicate for one pair (0 or 1)."""
    return _load().hstu_oracle_valid(i, j, L, mask_type, num_context, num_targets,
                                     target_group_size)


def mask_matrix(L, mask_type=MASK_CAUSAL, num_context=0, num_targets=0, target_group_size=0):
    """[L, L] 0/1 matrix of the oracle's predicate (small L only)."""
    return np.array([[valid(i, j, L, mask_type, num_context, num_targets, target_group_size)
                      for j in range(L)] for i in range(L)], dtype=np.int64)


def count_valid(seq_offsets, num_heads_q, *, num_context=None, num_targets=None,
                mask_type=MASK_CAUSAL, target_group_size=0):
    """Sum over sequences of Nq * #valid(i, j): the mask-aware pair count."""
    so = _i64(seq_offsets)
    nc, nt = _i64(num_context), _i64(num_targets)
    return int(_load().hstu_oracle_count_valid(_p(so, ctypes.c_int64), so.shape[0] - 1,
                                               num_heads_q, _p(nc, ctypes.c_int64),
                                               _p(nt, ctypes.c_int64), mask_type,
                                               target_group_size))


def count_valid_kv(query_lengths, key_lengths, num_heads_q, *, num_context=None,
                   num_targets=None, mask_type=MASK_CAUSAL, target_group_size=0):
    """Pair count with per-sequence query and key lengths, queries at the end of the keys."""
    lq, lk = _i64(query_lengths), _i64(key_lengths)
    nc, nt = _i64(num_context), _i64(num_targets)
    return int(_load().hstu_oracle_count_valid_kv(_p(lq, ctypes.c_int64),
                                                  _p(lk, ctypes.c_int64), lq.shape[0],
                                                  num_heads_q, _p(nc, ctypes.c_int64),
                                                  _p(nt, ctypes.c_int64), mask_type,
                                                  target_group_size))
