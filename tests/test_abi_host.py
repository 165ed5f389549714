"""Host-side checks of the C ABI (no GPU needed): the library builds for sm_103a,
loads, exports every entry point the header declares, validates descriptors
before touching the device, and counts mask-aware work like the oracle."""
import ctypes

import numpy as np
import pytest

import oracle
from hstu_dense_forward_gb300 import _abi, count_pairs, useful_flops


def test_library_exports_every_declared_symbol(built_lib):
    L = ctypes.CDLL(built_lib)
    names = _abi.declared_symbols()
    assert {"hstu_fwd_create", "hstu_fwd_run", "hstu_fwd_destroy", "hstu_fwd_get_error",
            "hstu_status_string"} <= set(names)
    for n in names:
        assert hasattr(L, n), f"{n} declared in include/hstu_fwd.h but not exported"


def _desc(**kw):
    d = _abi.Desc()
    base = dict(dtype=_abi.HSTU_BF16, batch=2, num_heads_q=4, num_heads_kv=2, head_dim=128,
                max_seqlen=256, index_is_int64=1, mask_type=_abi.HSTU_MASK_CAUSAL,
                target_group_size=0, has_rab=0, has_num_context=0, has_num_targets=0,
                watchdog_ms=0)
    base.update(kw)
    for k, v in base.items():
        setattr(d, k, v)
    return d


@pytest.mark.parametrize("kw,status", [
    (dict(num_heads_q=3, num_heads_kv=2), _abi.HSTU_ERR_INVALID_ARG),   # Nq % Nk != 0
    (dict(mask_type=_abi.HSTU_MASK_UPPER), _abi.HSTU_ERR_UNSUPPORTED),  # "currently not supported"
    (dict(mask_type=_abi.HSTU_MASK_CUSTOM, has_rab=1, head_dim=256), _abi.HSTU_ERR_UNSUPPORTED),
    (dict(mask_type=_abi.HSTU_MASK_CUSTOM, has_num_targets=1), _abi.HSTU_ERR_INVALID_ARG),
    (dict(mask_type=_abi.HSTU_MASK_CUSTOM, rab_heads=1), _abi.HSTU_ERR_INVALID_ARG),
    (dict(mask_type=_abi.HSTU_MASK_CUSTOM, max_seqlen=100), _abi.HSTU_ERR_UNSUPPORTED),
    (dict(mask_type=7), _abi.HSTU_ERR_INVALID_ARG),
    (dict(head_dim=40), _abi.HSTU_ERR_UNSUPPORTED),                      # not a multiple of 16
    (dict(head_dim=528), _abi.HSTU_ERR_UNSUPPORTED),
    (dict(head_dim=512, has_rab=1), _abi.HSTU_ERR_UNSUPPORTED),          # 512: built-in masks
    (dict(head_dim=384, mask_type=_abi.HSTU_MASK_CUSTOM), _abi.HSTU_ERR_UNSUPPORTED),
    (dict(head_dim=512, is_delta_qk=1), _abi.HSTU_ERR_UNSUPPORTED),
    (dict(dtype=_abi.HSTU_FP8_E4M3, head_dim=144), _abi.HSTU_ERR_UNSUPPORTED),  # FP8: <= 128
    (dict(dtype=_abi.HSTU_FP8_E4M3, mask_type=_abi.HSTU_MASK_CUSTOM, has_rab=1),
     _abi.HSTU_ERR_UNSUPPORTED),                                         # FP8: mask or rab
    (dict(dtype=_abi.HSTU_FP8_E4M3, mask_type=_abi.HSTU_MASK_CUSTOM, is_delta_qk=1),
     _abi.HSTU_ERR_UNSUPPORTED),
    (dict(dtype=_abi.HSTU_FP8_E4M3, has_rab=1, is_delta_qk=1), _abi.HSTU_ERR_UNSUPPORTED),
    (dict(descale=_abi.HSTU_DESCALE_HEAD), _abi.HSTU_ERR_INVALID_ARG),  # descales: FP8 only
    (dict(dtype=_abi.HSTU_FP8_E4M3, descale=5), _abi.HSTU_ERR_INVALID_ARG),
    (dict(dtype=_abi.HSTU_FP8_E4M3, descale=-1), _abi.HSTU_ERR_INVALID_ARG),
    (dict(dtype=_abi.HSTU_F32, head_dim=300), _abi.HSTU_ERR_UNSUPPORTED),
    (dict(head_dim=0), _abi.HSTU_ERR_INVALID_ARG),
    (dict(max_seqlen=0), _abi.HSTU_ERR_INVALID_ARG),
    (dict(max_seqlen=200000), _abi.HSTU_ERR_INVALID_ARG),
    (dict(has_rab=1, max_seqlen=100), _abi.HSTU_ERR_UNSUPPORTED),        # TMA row stride
    (dict(dtype=9), _abi.HSTU_ERR_INVALID_ARG),
    (dict(batch=-1), _abi.HSTU_ERR_INVALID_ARG),
    (dict(target_group_size=-2), _abi.HSTU_ERR_INVALID_ARG),
    (dict(layout=2), _abi.HSTU_ERR_INVALID_ARG),
    (dict(has_rab=1, rab_heads=2), _abi.HSTU_ERR_INVALID_ARG),          # neither 1 nor Nq
    (dict(reserved=1), _abi.HSTU_ERR_INVALID_ARG),
    (dict(is_delta_qk=2), _abi.HSTU_ERR_INVALID_ARG),
    (dict(page_size=64), _abi.HSTU_ERR_INVALID_ARG),                    # not in {32, 128, 256}
    (dict(max_seqlen_k=512), _abi.HSTU_ERR_INVALID_ARG),                # without a key side
    (dict(is_delta_qk=1, max_seqlen_k=-1), _abi.HSTU_ERR_INVALID_ARG),
    (dict(is_delta_qk=1, layout=1), _abi.HSTU_ERR_UNSUPPORTED),         # jagged only
    (dict(page_size=128, layout=1), _abi.HSTU_ERR_UNSUPPORTED),
    (dict(is_delta_qk=1, max_seqlen_k=1001, has_rab=1), _abi.HSTU_ERR_UNSUPPORTED),  # Sk % 8
])
def test_create_rejects_bad_descriptors(built_lib, kw, status):
    lib = _abi.lib()
    h = ctypes.c_void_p()
    d = _desc(**kw)
    assert lib.hstu_fwd_create(ctypes.byref(d), ctypes.byref(h)) == status
    assert not h.value


def test_null_arguments(built_lib):
    lib = _abi.lib()
    assert lib.hstu_fwd_destroy(None) == _abi.HSTU_OK
    assert lib.hstu_fwd_create(None, None) == _abi.HSTU_ERR_INVALID_ARG
    h = ctypes.c_void_p()
    assert lib.hstu_fwd_create(None, ctypes.byref(h)) == _abi.HSTU_ERR_INVALID_ARG
    assert lib.hstu_fwd_run(None, None, None, None, None, None, None, None, 0, 1.0, 1.0,
                            None, None) == _abi.HSTU_ERR_INVALID_ARG
    n = ctypes.c_int()
    assert lib.hstu_fwd_get_error(None, ctypes.byref(n)) == _abi.HSTU_ERR_INVALID_ARG
    a = _abi.Args()
    assert lib.hstu_fwd_run_args(None, ctypes.byref(a), None) == _abi.HSTU_ERR_INVALID_ARG
    assert lib.hstu_fwd_run_fp8(None, None, None, None, None, None, None, None, None, None, 0,
                                1.0, 1.0, None, None) == _abi.HSTU_ERR_INVALID_ARG
    assert lib.hstu_fwd_trace_read(None, None, 0) == _abi.HSTU_ERR_INVALID_ARG
    for s in range(6):
        assert lib.hstu_status_string(s)


@pytest.mark.parametrize("seed", range(6))
def test_count_pairs_matches_oracle(built_lib, seed):
    rng = np.random.default_rng(100 + seed)
    B = int(rng.integers(1, 6))
    S = 64
    lengths = rng.integers(0, S + 1, B)
    so = np.concatenate([[0], np.cumsum(lengths)])
    causal = seed % 3 != 0
    nc = rng.integers(0, 10, B) if seed % 2 else None
    nt = rng.integers(0, 20, B) if seed >= 2 else None
    g = int(rng.integers(0, 5)) if causal else 0
    want = oracle.count_valid(so, 3, num_context=nc, num_targets=nt,
                              mask_type=oracle.MASK_CAUSAL if causal else oracle.MASK_NONE,
                              target_group_size=g)
    got = count_pairs(so, 3, max_seqlen=S, num_context=nc, num_targets=nt, causal=causal,
                      target_group_size=g)
    assert got == want
    assert useful_flops(got, 128) == 4 * 128 * want


def test_count_pairs_closed_forms(built_lib):
    so = [0, 100, 250]
    assert count_pairs(so, 2, max_seqlen=150) == 2 * (100 * 101 // 2 + 150 * 151 // 2)
    assert count_pairs(so, 2, max_seqlen=150, causal=False) == 2 * (100 ** 2 + 150 ** 2)


def test_count_pairs_normal_layout(built_lib):
    """The normal layout is B sequences of max_seqlen tokens: the count equals the jagged
    count with offsets b * S, and no offsets may be passed."""
    S, B = 96, 3
    nc, nt = [5, 0, 20], [10, 30, 0]
    want = count_pairs([b * S for b in range(B + 1)], 4, max_seqlen=S, num_context=nc,
                       num_targets=nt, target_group_size=3)
    got = count_pairs(None, 4, max_seqlen=S, num_context=nc, num_targets=nt,
                      target_group_size=3, layout="normal", batch=B)
    assert got == want
    lib = _abi.lib()
    d = _desc(batch=B, max_seqlen=S, layout=_abi.HSTU_LAYOUT_NORMAL)
    so = (ctypes.c_longlong * (B + 1))(*[b * S for b in range(B + 1)])
    out = ctypes.c_longlong(0)
    assert lib.hstu_fwd_count_pairs(ctypes.byref(d), so, None, None,
                                    ctypes.byref(out)) == _abi.HSTU_ERR_INVALID_ARG


def test_rab_broadcast_descriptor_accepted(built_lib):
    lib = _abi.lib()
    for rab_heads in (0, 1, 4):
        h = ctypes.c_void_p()
        d = _desc(has_rab=1, rab_heads=rab_heads)
        st = lib.hstu_fwd_create(ctypes.byref(d), ctypes.byref(h))
        # a plan needs a GB300; without one creation stops at the device check
        assert st in (_abi.HSTU_OK, _abi.HSTU_ERR_UNSUPPORTED, _abi.HSTU_ERR_CUDA)
        if h.value:
            lib.hstu_fwd_destroy(h)


def test_count_pairs_custom_mask_counts_every_pair(built_lib):
    """With a custom mask every (i, j) of a sequence is computed (its values act as
    weights), so the work count is that of no mask."""
    lib = _abi.lib()
    so = (ctypes.c_longlong * 3)(0, 100, 250)
    out = ctypes.c_longlong(0)
    d = _desc(mask_type=_abi.HSTU_MASK_CUSTOM, max_seqlen=256)
    assert lib.hstu_fwd_count_pairs(ctypes.byref(d), so, None, None,
                                    ctypes.byref(out)) == _abi.HSTU_OK
    assert out.value == 4 * (100 ** 2 + 150 ** 2)


def _kv_case(rng, B, page_size):
    """Random query lengths, new k/v rows and a page table (histories of 0 to 5 pages)."""
    lnew = rng.integers(0, 300, B)
    lq = np.minimum(rng.integers(0, 300, B), lnew)
    pages = rng.integers(0, 6, B)
    last = rng.integers(1, page_size + 1, B)
    hist = np.where(pages > 0, (pages - 1) * page_size + last, 0)
    lq = np.minimum(lq + rng.integers(0, 50, B), hist + lnew)  # queries may reach into history
    so_q = np.concatenate([[0], np.cumsum(lq)])
    so_k = np.concatenate([[0], np.cumsum(lnew)])
    po = np.concatenate([[0], np.cumsum(pages)])
    return lq, lnew, hist, so_q, so_k, po, last


@pytest.mark.parametrize("seed", range(4))
def test_count_pairs_kv_matches_oracle(built_lib, seed):
    """Pairs of calls whose queries are the last tokens of longer key sequences (own k/v
    offsets and a paged history), against the oracle's brute-force count."""
    from hstu_dense_forward_gb300 import count_pairs_kv
    rng = np.random.default_rng(seed)
    B, ps = 5, [32, 128, 256, 32][seed]
    lq, lnew, hist, so_q, so_k, po, last = _kv_case(rng, B, ps)
    lk = hist + lnew
    nc = rng.integers(0, 40, B)
    nt = rng.integers(0, 60, B)
    for causal, g in ((True, 0), (True, 2), (False, 0)):
        kw = dict(num_context=nc, num_targets=nt, target_group_size=g) if causal else {}
        got = count_pairs_kv(so_q, 3, max_seqlen=512, seq_offsets_k=so_k, page_offsets=po,
                             last_page_len=last, page_size=ps, max_seqlen_k=int(lk.max()) + 1,
                             causal=causal, **kw)
        ref = oracle.count_valid_kv(lq, lk, 3, mask_type=oracle.MASK_CAUSAL if causal
                                    else oracle.MASK_NONE, **kw)
        assert got == ref


def test_count_pairs_kv_without_key_side_matches_count_pairs(built_lib):
    from hstu_dense_forward_gb300 import count_pairs_kv
    so = [0, 100, 350, 351]
    kw = dict(num_context=[3, 0, 1], num_targets=[10, 20, 0], target_group_size=3)
    assert count_pairs_kv(so, 2, max_seqlen=256, **kw) == count_pairs(so, 2, max_seqlen=256, **kw)


def test_key_side_entry_points_validate_before_the_device(built_lib):
    """hstu_fwd_run_kv without a plan, and the allocation-free entry point with a key-side
    descriptor, fail before any CUDA call (the key-side plan checks run in the GPU tests)."""
    lib = _abi.lib()
    fake = ctypes.c_void_p(1 << 20)  # never dereferenced: the calls fail validation first
    kv = _abi.KV()
    assert lib.hstu_fwd_run_kv(None, fake, fake, fake, fake, ctypes.byref(kv), None, None, None,
                               10, 1.0, 1.0, fake, None) == _abi.HSTU_ERR_INVALID_ARG
    for kw in (dict(is_delta_qk=1), dict(page_size=128), dict(is_delta_qk=1, page_size=32)):
        d = _desc(**kw)
        assert lib.hstu_fwd_run_noalloc(ctypes.byref(d), fake, fake, fake, fake, None, None,
                                        None, 10, 1.0, 1.0, fake, None) == \
            _abi.HSTU_ERR_UNSUPPORTED
