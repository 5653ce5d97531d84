"""GPU parity at the full workload sizes, in the launch configuration the
benchmark times (heuristic split count): every output where the oracle is
cheap, sampled (sequence, kv head) slices where it is not."""

import numpy as np
import pytest
import torch

import oracle
import decode_attention_20_b300 as fd
from decode_attention_20_b300 import inputs

from _convert import assert_parity, to_f64

pytestmark = pytest.mark.gpu


def _slice_ref(case, b, g, lens):
    """Oracle for one (sequence, kv head) slice, from device tensors."""
    G = case.q.shape[1] // case.k.shape[2]
    n = lens[b]
    q = to_f64(case.q[b:b + 1, g * G:(g + 1) * G])
    k = to_f64(case.k[b:b + 1, :n, g:g + 1])
    v = to_f64(case.v[b:b + 1, :n, g:g + 1])
    return oracle.decode_attention_ref(q, k, v, None, case.scale)


def test_flash_decoding_b1_64k_full(cuda_device):
    case = inputs.flash_decoding_b1(65536, device="cuda")
    O, L = fd.decode_attention(case.q, case.k, case.v, None, 0, case.scale)
    fd.check_device_error()
    O_ref, L_ref = oracle.decode_attention_ref(to_f64(case.q), to_f64(case.k), to_f64(case.v),
                                               None, case.scale)
    assert_parity(to_f64(O), to_f64(L), O_ref, L_ref, torch.bfloat16, "b1 64K")


def test_ragged_batch_full_size_sampled(cuda_device):
    """Every kv head of the shortest, median and longest sequences, and of
    two fixed ones, in the benchmark's launch configuration."""
    case = inputs.ragged_batch(device="cuda")
    lens = case.lens
    O, L = fd.decode_attention(case.q, case.k, case.v, case.seqlens.cuda(), 0, case.scale)
    fd.check_device_error()
    G = case.q.shape[1] // case.k.shape[2]
    order = np.argsort(lens)
    picks = sorted({int(order[0]), int(order[-1]), int(order[len(order) // 2]), 5, 17})
    for b in picks:
        for g in range(case.k.shape[2]):
            O_ref, L_ref = _slice_ref(case, b, g, lens)
            assert_parity(to_f64(O[b:b + 1, g * G:(g + 1) * G]), to_f64(L[b:b + 1, g * G:(g + 1) * G]),
                          O_ref, L_ref, torch.bfloat16, f"ragged b={b} g={g} len={lens[b]}")


_LONG = {}


def _long_case_and_refs():
    """The long peaked workload and the oracle of all its 4 x 8 (sequence,
    kv head) slices, computed once for the parametrised tests below."""
    if "case" not in _LONG:
        case = inputs.long_context_peaked(device="cuda")
        lens = case.lens
        refs = {(b, g): _slice_ref(case, b, g, lens)
                for b in range(case.k.shape[0]) for g in range(case.k.shape[2])}
        _LONG["case"], _LONG["refs"] = case, refs
    return _LONG["case"], _LONG["refs"]


@pytest.mark.parametrize("ns", [0, 1, 64, 256])
def test_long_context_peaked_every_slice(cuda_device, ns):
    """All 32 (sequence, kv head) slices of the 4 x 131072 peaked workload."""
    case, refs = _long_case_and_refs()
    O, L = fd.decode_attention(case.q, case.k, case.v, None, ns, case.scale)
    fd.check_device_error()
    G = case.q.shape[1] // case.k.shape[2]
    for (b, g), (O_ref, L_ref) in refs.items():
        assert_parity(to_f64(O[b:b + 1, g * G:(g + 1) * G]), to_f64(L[b:b + 1, g * G:(g + 1) * G]),
                      O_ref, L_ref, torch.bfloat16, f"long b={b} g={g} ns={ns}")
