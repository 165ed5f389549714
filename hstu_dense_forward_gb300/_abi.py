"""ctypes binding of libhstu_fwd.so (include/hstu_fwd.h). Argument marshalling only:
every step of the forward runs in the library's CUDA kernels."""
from __future__ import annotations

import ctypes
import os
import re
import threading

PKG = os.path.dirname(os.path.abspath(__file__))
# HSTU_FWD_TRACE=1 loads the tracing build of the library (build.build(trace=True));
# HSTU_FWD_LIB=<path> loads another build of it (for comparing builds)
LIB_PATH = os.environ.get("HSTU_FWD_LIB") or os.path.join(
    PKG, "libhstu_fwd_trace.so" if os.environ.get("HSTU_FWD_TRACE") == "1" else "libhstu_fwd.so")
HEADER = os.path.join(os.path.dirname(PKG), "include", "hstu_fwd.h")

HSTU_OK, HSTU_ERR_INVALID_ARG, HSTU_ERR_UNSUPPORTED, HSTU_ERR_CUDA, HSTU_ERR_TIMEOUT, \
    HSTU_ERR_DEVICE_CHECK = range(6)
HSTU_F32, HSTU_F16, HSTU_BF16, HSTU_FP8_E4M3 = 0, 1, 2, 3
HSTU_MASK_CAUSAL, HSTU_MASK_UPPER, HSTU_MASK_NONE, HSTU_MASK_CUSTOM = 0, 1, 2, 3
HSTU_DEVERR_NONE, HSTU_DEVERR_OFFSETS, HSTU_DEVERR_TIMEOUT = 0, 1, 2
HSTU_LAYOUT_JAGGED, HSTU_LAYOUT_NORMAL = 0, 1
(HSTU_DESCALE_CAST, HSTU_DESCALE_TENSOR, HSTU_DESCALE_BATCH, HSTU_DESCALE_HEAD,
 HSTU_DESCALE_BLOCK) = 0, 1, 2, 3, 4


class Desc(ctypes.Structure):
    _fields_ = [
        ("dtype", ctypes.c_int),
        ("batch", ctypes.c_int),
        ("num_heads_q", ctypes.c_int),
        ("num_heads_kv", ctypes.c_int),
        ("head_dim", ctypes.c_int),
        ("max_seqlen", ctypes.c_int),
        ("index_is_int64", ctypes.c_int),
        ("mask_type", ctypes.c_int),
        ("target_group_size", ctypes.c_int),
        ("has_rab", ctypes.c_int),
        ("has_num_context", ctypes.c_int),
        ("has_num_targets", ctypes.c_int),
        ("watchdog_ms", ctypes.c_int),
        ("layout", ctypes.c_int),
        ("rab_heads", ctypes.c_int),
        ("is_delta_qk", ctypes.c_int),
        ("max_seqlen_k", ctypes.c_int),
        ("page_size", ctypes.c_int),
        ("descale", ctypes.c_int),
        ("reserved", ctypes.c_int),
    ]


class KV(ctypes.Structure):
    """hstu_fwd_kv: the key side of hstu_fwd_run_kv (device pointers)."""
    _fields_ = [
        ("seq_offsets_k", ctypes.c_void_p),
        ("total_tokens_k", ctypes.c_longlong),
        ("kv_cache", ctypes.c_void_p),
        ("num_pages", ctypes.c_longlong),
        ("page_offsets", ctypes.c_void_p),
        ("page_ids", ctypes.c_void_p),
        ("last_page_len", ctypes.c_void_p),
    ]


class Descale(ctypes.Structure):
    """hstu_fwd_descale: FP8 descale factor arrays (device fp32 pointers)."""
    _fields_ = [("q", ctypes.c_void_p), ("k", ctypes.c_void_p), ("v", ctypes.c_void_p)]


class Args(ctypes.Structure):
    """hstu_fwd_args: every input of one forward (hstu_fwd_run_args)."""
    _fields_ = [
        ("q", ctypes.c_void_p), ("k", ctypes.c_void_p), ("v", ctypes.c_void_p),
        ("out", ctypes.c_void_p), ("seq_offsets", ctypes.c_void_p),
        ("kv", ctypes.POINTER(KV)), ("rab", ctypes.c_void_p), ("mask", ctypes.c_void_p),
        ("num_context", ctypes.c_void_p), ("num_targets", ctypes.c_void_p),
        ("descale", ctypes.POINTER(Descale)), ("total_tokens", ctypes.c_longlong),
        ("alpha", ctypes.c_float), ("silu_scale", ctypes.c_float),
    ]


class HstuError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {status_string(status)} (status {status})")


_lock = threading.Lock()
_lib = None


def declared_symbols() -> list[str]:
    """Entry points declared in include/hstu_fwd.h (the HSTU_API functions)."""
    text = open(HEADER).read()
    return re.findall(r"HSTU_API\s+[\w\s\*]+?\b(\w+)\s*\(", text)


def lib():
    """Load libhstu_fwd.so; raises if it has not been built (there is no fallback)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                f"{LIB_PATH} is missing: build it with hstu_dense_forward_gb300.build.build() "
                "(nvcc, sm_103a). The HSTU forward has no non-CUDA implementation.")
        L = ctypes.CDLL(LIB_PATH)
        vp, ll, f = ctypes.c_void_p, ctypes.c_longlong, ctypes.c_float
        L.hstu_fwd_create.restype = ctypes.c_int
        L.hstu_fwd_create.argtypes = [ctypes.POINTER(Desc), ctypes.POINTER(vp)]
        L.hstu_fwd_run.restype = ctypes.c_int
        L.hstu_fwd_run.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, ll, f, f, vp, vp]
        L.hstu_fwd_destroy.restype = ctypes.c_int
        L.hstu_fwd_destroy.argtypes = [vp]
        L.hstu_fwd_get_error.restype = ctypes.c_int
        L.hstu_fwd_get_error.argtypes = [vp, ctypes.POINTER(ctypes.c_int)]
        L.hstu_fwd_launches_per_run.restype = ctypes.c_int
        L.hstu_fwd_launches_per_run.argtypes = [vp, ctypes.POINTER(ctypes.c_int)]
        L.hstu_fwd_count_pairs.restype = ctypes.c_int
        L.hstu_fwd_count_pairs.argtypes = [ctypes.POINTER(Desc), vp, vp, vp,
                                           ctypes.POINTER(ctypes.c_longlong)]
        L.hstu_fwd_run_masked.restype = ctypes.c_int
        L.hstu_fwd_run_masked.argtypes = [vp, vp, vp, vp, vp, vp, ll, f, f, vp, vp]
        L.hstu_fwd_run_kv.restype = ctypes.c_int
        L.hstu_fwd_run_kv.argtypes = [vp, vp, vp, vp, vp, ctypes.POINTER(KV), vp, vp, vp, ll, f, f,
                                      vp, vp]
        L.hstu_fwd_count_pairs_kv.restype = ctypes.c_int
        L.hstu_fwd_count_pairs_kv.argtypes = [ctypes.POINTER(Desc), vp, vp, vp, vp, vp, vp,
                                              ctypes.POINTER(ctypes.c_longlong)]
        L.hstu_fwd_run_noalloc.restype = ctypes.c_int
        L.hstu_fwd_run_noalloc.argtypes = [ctypes.POINTER(Desc), vp, vp, vp, vp, vp, vp, vp, ll, f,
                                           f, vp, vp]
        L.hstu_fwd_run_fp8.restype = ctypes.c_int
        L.hstu_fwd_run_fp8.argtypes = [vp, vp, vp, vp, vp, ctypes.POINTER(KV), vp, vp, vp,
                                       ctypes.POINTER(Descale), ll, f, f, vp, vp]
        L.hstu_fwd_run_args.restype = ctypes.c_int
        L.hstu_fwd_run_args.argtypes = [vp, ctypes.POINTER(Args), vp]
        L.hstu_fwd_trace_read.restype = ctypes.c_int
        L.hstu_fwd_trace_read.argtypes = [vp, vp, ll]
        L.hstu_status_string.restype = ctypes.c_char_p
        L.hstu_status_string.argtypes = [ctypes.c_int]
        _lib = L
        return _lib


def status_string(status: int) -> str:
    try:
        return lib().hstu_status_string(status).decode()
    except Exception:  # the library may be what failed to load
        return "status"


def check(status: int, what: str) -> None:
    if status != HSTU_OK:
        raise HstuError(status, what)
