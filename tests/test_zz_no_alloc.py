"""GPU test of fd_decode_attention_noalloc, the entry point for callers that
cannot allocate device memory while they run (a runtime that owns all device
memory, a region where no pool may grow, a loop that cannot risk an
allocation stall).  Call after call, it must match the fp64 oracle and give
the same result as fd_decode_attention, while keeping its partial results
in the library's fixed scratch array.

The file is named so that pytest collects it last: a run that stops at the
first failure has then already run every other test.  It also passes on its
own in a fresh process (the first call on the device does the one-time
scratch set-up).
"""

import ctypes

import pytest
import torch

import oracle
from decode_attention_20_b300 import _lib, inputs
from decode_attention_20_b300.api import _desc

from _convert import assert_parity, to_f64

pytestmark = pytest.mark.gpu

FD_ERR_UNSUPPORTED = 6
SCRATCH_BYTES = 8 * 1024 * 1024


def _call(fn, case, q, k, v, sl, ns):
    out = torch.full((q.shape[0], q.shape[1], q.shape[2]), float("nan"), device="cuda")
    lse = torch.full((q.shape[0], q.shape[1]), float("nan"), device="cuda")
    d = [_desc(x, n) for x, n in [(q, "q"), (k, "k"), (v, "v"), (sl, "sl"), (out, "out"), (lse, "lse")]]
    r = lambda x: ctypes.byref(x) if x is not None else None
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    st = fn(r(d[0]), r(d[1]), r(d[2]), r(d[3]), ns, ctypes.c_float(case.scale), r(d[4]), r(d[5]), stream)
    assert st == 0, _lib.lib().fd_last_error().decode()
    torch.cuda.synchronize()
    return out, lse


def _oracle(case):
    lens = case.seqlens.numpy() if case.seqlens is not None else None
    return oracle.decode_attention_ref(to_f64(case.q), to_f64(case.k), to_f64(case.v), lens,
                                       case.scale)


def test_noalloc_matches_allocating_entry_two_calls_in_a_row(cuda_device):
    """Both calls in a row match the fp64 oracle and the allocating entry
    point, within the bf16 tolerances."""
    L = _lib.lib()
    cases = [
        (inputs.flash_decoding_b1(4096, seed=5), 0),                                 # heuristic splits
        (inputs.decode_case(3, 32, 8, 128, 1500, seed=6, seqlens=[1500, 17, 900]), 7),
    ]
    for case, ns in cases:
        q, k, v = case.q.cuda(), case.k.cuda(), case.v.cuda()
        sl = case.seqlens.cuda() if case.seqlens is not None else None
        O_ref, L_ref = _oracle(case)
        ref_o, ref_l = _call(L.fd_decode_attention, case, q, k, v, sl, ns)
        assert_parity(to_f64(ref_o), to_f64(ref_l), O_ref, L_ref, torch.bfloat16,
                      f"allocating entry {case.name}")
        for call in range(2):                       # the scratch keeps the last call's contents
            o, l = _call(L.fd_decode_attention_noalloc, case, q, k, v, sl, ns)
            assert_parity(to_f64(o), to_f64(l), O_ref, L_ref, torch.bfloat16,
                          f"noalloc vs oracle {case.name} call {call}")
            assert_parity(to_f64(o), to_f64(l), to_f64(ref_o), to_f64(ref_l), torch.bfloat16,
                          f"noalloc vs allocating entry {case.name} call {call}")


def test_noalloc_lowers_the_heuristic_split_count_to_the_scratch(cuda_device):
    """With num_splits = 0 the library's own choice is never refused: one kv
    head with 64 query heads over 65536 tokens makes the heuristic pick 256
    splits, whose partials (8.45 MB) exceed the 8 MiB scratch; the call runs
    with fewer splits and still matches the oracle."""
    L = _lib.lib()
    case = inputs.decode_case(1, 64, 1, 128, 65536, seed=8)
    assert L.fd_choose_num_splits(1, 1, 65536, 148) == 256
    assert L.fd_workspace_bytes(1, 64, 128, 256) > SCRATCH_BYTES
    q, k, v = case.q.cuda(), case.k.cuda(), case.v.cuda()
    O_ref, L_ref = _oracle(case)
    for call in range(2):
        o, l = _call(L.fd_decode_attention_noalloc, case, q, k, v, None, 0)
        assert_parity(to_f64(o), to_f64(l), O_ref, L_ref, torch.bfloat16, f"capped call {call}")


def test_noalloc_rejects_work_beyond_the_scratch(cuda_device):
    """A call whose partial results exceed the fixed scratch is refused before
    anything is enqueued (the descriptors below are never dereferenced)."""
    L = _lib.lib()
    B, Hq, Hkv, D, Lcap, ns = 32, 32, 8, 128, 32768, 64
    assert L.fd_workspace_bytes(B, Hq, D, ns) > SCRATCH_BYTES
    fake = 0x100000
    t = lambda shape, dt: _lib.raw_descriptor(fake, dt, shape, [
        int(torch.tensor(shape[i + 1:]).prod()) if i + 1 < len(shape) else 1 for i in range(len(shape))])
    q = t([B, Hq, D], _lib.FD_BF16)
    k = t([B, Lcap, Hkv, D], _lib.FD_BF16)
    out = t([B, Hq, D], _lib.FD_F32)
    r = ctypes.byref
    st = L.fd_decode_attention_noalloc(r(q), r(k), r(k), None, ns, ctypes.c_float(0.1), r(out), None, None)
    assert st == FD_ERR_UNSUPPORTED
    assert b"static scratch" in L.fd_last_error()
