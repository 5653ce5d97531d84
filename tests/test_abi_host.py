"""C-ABI tests that need no GPU: the library loads and exports every symbol
include/fd_decode.h declares; the pure host functions equal the oracle's
mirrors bit for bit; argument validation returns the documented status
before touching the device."""

import ctypes
import math
import os
import re

import pytest

import oracle
from decode_attention_20_b300 import _lib
from decode_attention_20_b300._lib import FD_BF16, FD_F32, FD_I32, raw_descriptor

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "fd_decode.h")


@pytest.fixture(scope="module")
def L():
    if not os.path.exists(_lib.LIB_PATH):
        from decode_attention_20_b300 import build
        build.build()
    return _lib.lib()


def declared_functions():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"FD_API\s+[\w\s\*]+?\b(fd_\w+)\s*\(", text)))


def test_header_declares_entry_points():
    names = declared_functions()
    for n in ["fd_decode_attention", "fd_bifurcated_attention", "fd_choose_num_splits",
              "fd_split_bounds", "fd_check_device_error", "fd_lse_combine"]:
        assert n in names


def test_library_exports_every_declared_symbol(L):
    missing = [n for n in declared_functions() if not hasattr(L, n)]
    assert not missing, missing


def test_version_and_status_strings(L):
    assert b"sm_103a" in L.fd_version()
    for s in range(0, 11):
        assert L.fd_status_string(s)
    assert L.fd_status_string(999) == b"unknown status"


def _bounds(L, length, ns, i):
    b = ctypes.c_int64(-7)
    e = ctypes.c_int64(-7)
    st = L.fd_split_bounds(length, ns, i, ctypes.byref(b), ctypes.byref(e))
    return st, b.value, e.value


def test_split_bounds_bit_exact_vs_oracle(L):
    lengths = list(range(0, 260)) + [1000, 1023, 1024, 1025, 4095, 65536, 131071, 131072,
                                    2_000_000_000]
    for length in lengths:
        for ns in [1, 2, 3, 4, 5, 7, 8, 9, 16, 37, 64, 128, 255, 256]:
            for i in range(ns):
                st, b, e = _bounds(L, length, ns, i)
                assert st == 0
                assert (b, e) == oracle.split_bounds_ref(length, ns, i), (length, ns, i)


def test_split_bounds_at_the_largest_accepted_length(L):
    """The largest cache length the entry points accept (INT32_MAX - 128),
    where len + ns - 1 no longer fits a 32-bit int: the host partition (and
    the device copy, computed in 64 bits the same way) still covers [0, len)
    exactly, in order, with the oracle's bounds."""
    top = (1 << 31) - 1 - 128
    for length in [top, top - 1, top - 63, (1 << 31) - 1 - 255]:
        for ns in [2, 3, 37, 255, 256]:
            prev = 0
            for i in range(ns):
                st, b, e = _bounds(L, length, ns, i)
                assert st == 0
                assert (b, e) == oracle.split_bounds_ref(length, ns, i)
                assert b == prev and b <= e <= length
                prev = e
            assert prev == length


def test_split_bounds_errors(L):
    for args in [(10, 0, 0), (10, 2, 2), (10, 2, -1), (-1, 2, 0)]:
        st, b, e = _bounds(L, *args)
        assert st == 5 and b == -7 and e == -7           # FD_ERR_ARG, outputs untouched
    assert L.fd_split_bounds(10, 1, 0, None, None) == 1  # FD_ERR_NULL


def test_heuristic_bit_exact_vs_oracle(L):
    for sms in [1, 2, 8, 132, 148, 160]:
        for B in [0, 1, 2, 3, 4, 8, 32, 64, 100, 1000]:
            for hkv in [0, 1, 2, 8, 32]:
                for Lmax in [0, 1, 100, 256, 257, 512, 4096, 65536, 131072, 1 << 22]:
                    assert L.fd_choose_num_splits(B, hkv, Lmax, sms) == \
                        oracle.choose_num_splits_ref(B, hkv, Lmax, sms), (B, hkv, Lmax, sms)


def test_workspace_bytes(L):
    assert L.fd_workspace_bytes(1, 64, 128, 1) == 0
    b = L.fd_workspace_bytes(1, 64, 128, 37)
    assert b >= 64 * 37 * 129 * 4 and b % 256 == 0


# ------------------------------------------------------------------ validation

FAKE = 0x10000  # never dereferenced: every case below fails validation first


def _t(shape, dtype=FD_BF16, stride=None, ptr=FAKE):
    if stride is None:
        stride = []
        acc = 1
        for s in reversed(shape):
            stride.insert(0, acc)
            acc *= s
    return raw_descriptor(ptr, dtype, list(shape), list(stride))


def _decode(L, q, k, v, sl, ns, scale, o, lse):
    r = lambda x: ctypes.byref(x) if x is not None else None
    return L.fd_decode_attention(r(q), r(k), r(v), r(sl), ns, scale, r(o), r(lse), None)


def good():
    return dict(q=_t([2, 8, 128]), k=_t([2, 64, 2, 128]), v=_t([2, 64, 2, 128]),
                sl=_t([2], FD_I32), ns=0, scale=0.1, o=_t([2, 8, 128], FD_F32),
                lse=_t([2, 8], FD_F32))


CASES = [
    ("null q", dict(q=None), 1),
    ("null data", dict(q=_t([2, 8, 128], ptr=0)), 1),
    ("q rank", dict(q=_t([2, 8, 128, 1])), 2),
    ("k/v shapes", dict(v=_t([2, 65, 2, 128])), 2),
    ("batch mismatch", dict(k=_t([3, 64, 2, 128]), v=_t([3, 64, 2, 128])), 2),
    ("head dim mismatch", dict(k=_t([2, 64, 2, 64]), v=_t([2, 64, 2, 64])), 2),
    ("out shape", dict(o=_t([2, 8, 64], FD_F32)), 2),
    ("lse shape", dict(lse=_t([2, 9], FD_F32)), 2),
    ("seqlens shape", dict(sl=_t([3], FD_I32)), 2),
    ("k/v dtype differ", dict(v=_t([2, 64, 2, 128], FD_F32)), 3),
    ("int q", dict(q=_t([2, 8, 128], FD_I32)), 3),
    ("bf16 out", dict(o=_t([2, 8, 128], FD_BF16)), 3),
    ("seqlens dtype", dict(sl=_t([2], FD_F32)), 3),
    ("unknown dtype", dict(q=_t([2, 8, 128], 9)), 3),
    ("inner stride", dict(k=_t([2, 64, 2, 128], stride=[32768, 256, 128, 2])), 4),
    ("negative stride", dict(k=_t([2, 64, 2, 128], stride=[-32768, 256, 128, 1])), 4),
    ("misaligned ptr", dict(q=_t([2, 8, 128], ptr=FAKE + 1)), 4),
    ("num_splits high", dict(ns=257), 5),
    ("num_splits negative", dict(ns=-1), 5),
    ("nan scale", dict(scale=float("nan")), 5),
    ("inf scale", dict(scale=float("inf")), 5),
    ("head dim 96", dict(q=_t([2, 8, 96]), k=_t([2, 64, 2, 96]), v=_t([2, 64, 2, 96]),
                         o=_t([2, 8, 96], FD_F32)), 6),
    ("Hq % Hkv", dict(k=_t([2, 64, 3, 128]), v=_t([2, 64, 3, 128])), 6),
]


@pytest.mark.parametrize("name,override,status", CASES, ids=[c[0] for c in CASES])
def test_decode_validation(L, name, override, status):
    a = good()
    a.update(override)
    assert _decode(L, a["q"], a["k"], a["v"], a["sl"], a["ns"], a["scale"], a["o"], a["lse"]) == status
    assert L.fd_last_error()


def test_valid_call_without_gpu_reports_cuda_error(L):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    a = good()
    st = _decode(L, a["q"], a["k"], a["v"], a["sl"], a["ns"], a["scale"], a["o"], a["lse"])
    assert st == 8  # FD_ERR_CUDA: validation passed, no device to run on


def test_bifurcated_validation(L):
    r = ctypes.byref
    q = _t([4, 8, 128])
    kc = _t([100, 1, 128])
    kd = _t([4, 16, 1, 128])
    o = _t([4, 8, 128], FD_F32)
    call = lambda q_, kc_, vc_, kd_, vd_, o_, scale=0.1: L.fd_bifurcated_attention(
        r(q_), r(kc_), r(vc_), r(kd_), r(vd_), None, scale, r(o_), None)
    assert call(q, kc, kc, kd, _t([4, 17, 1, 128]), o) == 2
    assert call(q, kc, kc, _t([5, 16, 1, 128]), _t([5, 16, 1, 128]), o) == 2
    assert call(q, _t([0, 1, 128]), _t([0, 1, 128]), kd, kd, o) == 2        # empty context
    assert call(q, _t([100, 1, 128], FD_F32), _t([100, 1, 128], FD_F32), kd, kd, o) == 3
    assert call(q, kc, kc, kd, kd, o, scale=math.inf) == 5
    assert call(_t([4, 6, 128]), _t([100, 4, 128]), _t([100, 4, 128]), _t([4, 16, 4, 128]),
                _t([4, 16, 4, 128]), _t([4, 6, 128], FD_F32)) == 6


def test_combine_validation(L):
    r = ctypes.byref
    po = _t([10, 4, 128], FD_F32)
    pl = _t([10, 4], FD_F32)
    o = _t([10, 128], FD_F32)
    assert L.fd_lse_combine(r(po), r(_t([10, 5], FD_F32)), r(o), None, None) == 2
    assert L.fd_lse_combine(r(_t([10, 4, 130], FD_F32)), r(pl), r(_t([10, 130], FD_F32)), None, None) == 6
    assert L.fd_lse_combine(r(po), r(pl), r(_t([10, 128], FD_BF16)), None, None) == 3


def test_profile_api_without_launches(L):
    assert L.fd_profile_enable(1) == 0
    n = ctypes.c_int64(-1)
    ms = ctypes.c_double(-1)
    assert L.fd_profile_read(0, ctypes.byref(n), ctypes.byref(ms)) == 0
    assert n.value == 0 and ms.value == 0.0
    assert L.fd_profile_read(7, ctypes.byref(n), ctypes.byref(ms)) == 5
    assert L.fd_profile_enable(0) == 0


def test_python_binding_rejects_cpu_tensors():
    import torch
    import decode_attention_20_b300 as fd
    q = torch.zeros(1, 4, 64)
    k = torch.zeros(1, 16, 4, 64)
    with pytest.raises(ValueError):
        fd.decode_attention(q, k, k)


def test_paged_validation(L):
    """fd_decode_attention_paged refuses bad descriptors before touching the
    device (the pointers below are never dereferenced)."""
    r = lambda x: ctypes.byref(x) if x is not None else None
    q = _t([2, 8, 128])
    kp = _t([10, 64, 2, 128])
    bt = _t([2, 5], FD_I32)
    o = _t([2, 8, 128], FD_F32)
    call = lambda q_=q, k_=kp, v_=kp, bt_=bt, sl=None, ns=0, scale=0.1, o_=o: \
        L.fd_decode_attention_paged(r(q_), r(k_), r(v_), r(bt_), r(sl), ns, scale, r(o_), None, None)
    assert call(v_=_t([10, 32, 2, 128])) == 2                       # page shapes differ
    assert call(bt_=_t([3, 5], FD_I32)) == 2                        # table rows != B
    assert call(bt_=_t([2, 5], FD_F32)) == 3                        # table dtype
    assert call(bt_=_t([2, 5], FD_I32, stride=[10, 2])) == 4        # table rows not contiguous
    assert call(sl=_t([3], FD_I32)) == 2                            # seqlens shape
    assert call(k_=_t([10, 64, 3, 128]), v_=_t([10, 64, 3, 128])) == 6   # Hq % Hkv
    assert call(ns=300) == 5
    assert call(scale=math.nan) == 5
    assert call(k_=_t([0, 64, 2, 128]), v_=_t([0, 64, 2, 128])) == 2     # no pages
    assert L.fd_last_error()
    import torch
    if not torch.cuda.is_available():
        assert call() == 8                                          # valid: no device here


def test_quant_validation(L):
    """fd_decode_attention_quant refuses bad descriptors on the host (the
    pointers below are never dereferenced), and the plain entry point
    refuses 8-bit caches."""
    from decode_attention_20_b300._lib import FD_E4M3, FD_I8
    r = lambda x: ctypes.byref(x) if x is not None else None
    q = _t([2, 8, 128])
    k = _t([2, 256, 2, 128], FD_I8)
    ks = _t([2], FD_F32)
    o = _t([2, 8, 128], FD_F32)
    call = lambda q_=q, k_=k, v_=k, ks_=ks, vs_=ks, sl=None, ns=0, scale=0.1, o_=o: \
        L.fd_decode_attention_quant(r(q_), r(k_), r(v_), r(ks_), r(vs_), r(sl), ns, scale, r(o_),
                                    None, None)
    assert call(k_=_t([2, 256, 2, 128])) == 3                          # bf16 cache
    assert call(v_=_t([2, 256, 2, 128], FD_E4M3)) == 3                 # K / V kinds differ
    assert call(ks_=None) == 1
    assert call(vs_=_t([2], FD_BF16)) == 3                              # scale dtype
    assert call(ks_=_t([3], FD_F32)) == 2                               # one scale per kv head
    assert call(ks_=_t([2, 1], FD_F32)) == 2                            # scale rank
    assert call(ns=-1) == 5
    assert call(scale=math.inf) == 5
    assert call(q_=_t([2, 8, 96])) == 2                                 # head dims differ
    assert L.fd_last_error()
    # the plain entry point takes bf16 / f32 caches only
    assert _decode(L, q, k, k, None, 0, 0.1, o, None) == 3
    import torch
    if not torch.cuda.is_available():
        assert call() == 8                                              # valid: no device here
        assert call(k_=_t([2, 256, 2, 128], FD_E4M3), v_=_t([2, 256, 2, 128], FD_E4M3)) == 8


def test_multi_validation(L):
    """fd_decode_attention_multi refuses bad descriptors on the host."""
    r = lambda x: ctypes.byref(x) if x is not None else None
    q = _t([2, 3, 8, 128])
    k = _t([2, 256, 2, 128])
    o = _t([2, 3, 8, 128], FD_F32)
    call = lambda q_=q, k_=k, v_=k, sl=None, ns=0, scale=0.1, o_=o, l_=None: \
        L.fd_decode_attention_multi(r(q_), r(k_), r(v_), r(sl), ns, scale, r(o_), r(l_), None)
    assert call(q_=_t([2, 8, 128])) == 2                            # q rank
    assert call(o_=_t([2, 2, 8, 128], FD_F32)) == 2                 # out tokens
    assert call(l_=_t([2, 8], FD_F32)) == 2                         # lse rank
    assert call(l_=_t([2, 2, 8], FD_F32)) == 2                      # lse tokens
    assert call(k_=_t([2, 256, 3, 128]), v_=_t([2, 256, 3, 128])) == 6
    assert call(q_=_t([2, 0, 8, 128]), o_=_t([2, 0, 8, 128], FD_F32)) == 2
    assert call(q_=_t([2, 9000, 8, 128]), o_=_t([2, 9000, 8, 128], FD_F32)) == 6
    assert call(o_=_t([2, 3, 8, 128])) == 3                          # out dtype
    assert call(ns=257) == 5
    import torch
    if not torch.cuda.is_available():
        assert call() == 8
        assert call(l_=_t([2, 3, 8], FD_F32)) == 8
