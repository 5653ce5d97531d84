"""GPU parity: split-KV decode attention over a paged KV cache
(fd_decode_attention_paged) against the fp64 paged oracle, for page sizes
the tensor-core split kernel streams (16, 32, 64, 128, 256) and ones that
fall back to the generic kernel, scattered and shared pages, ragged and
empty sequences, every split-kernel variant, and bad page ids caught on the
device."""

import pytest
import torch

import oracle
import decode_attention_20_b300 as fd
from decode_attention_20_b300 import inputs
from decode_attention_20_b300.api import FdError

from _convert import assert_parity, to_f64

pytestmark = pytest.mark.gpu


def _run(case, ns=0):
    sl = case.seqlens.cuda() if case.seqlens is not None else None
    O, L = fd.decode_attention_paged(case.q.cuda(), case.k_pages.cuda(), case.v_pages.cuda(),
                                     case.block_table.cuda(), sl, ns, case.scale)
    fd.check_device_error()
    return O, L


def _check(case, ns=0, label=""):
    O, L = _run(case, ns)
    lens = None if case.seqlens is None else case.seqlens.numpy()
    O_ref, L_ref = oracle.paged_decode_attention_ref(to_f64(case.q), to_f64(case.k_pages),
                                                     to_f64(case.v_pages),
                                                     case.block_table.numpy(), lens,
                                                     case.page_size, case.scale)
    assert_parity(to_f64(O), to_f64(L), O_ref, L_ref, case.k_pages.dtype, label or case.name)


@pytest.fixture(params=["default", "mma0", "mma1", "cuda"])
def variant(request, monkeypatch):
    if request.param != "default":
        monkeypatch.setenv("FD_SPLIT_VARIANT", request.param)
    else:
        monkeypatch.delenv("FD_SPLIT_VARIANT", raising=False)
    return request.param


@pytest.mark.parametrize("ps", [16, 32, 64, 128, 256])
@pytest.mark.parametrize("ns", [0, 1, 5])
def test_paged_page_sizes(cuda_device, variant, ps, ns):
    case = inputs.paged_case(3, 32, 4, 128, ps, 2048 // ps, seed=ps + ns, ragged=(1, 2048))
    _check(case, ns, f"{variant} ps={ps} ns={ns}")


@pytest.mark.parametrize("ps,dtype,D,G", [
    (48, torch.bfloat16, 128, 8),     # page size the TMA kernel does not stream
    (64, torch.float32, 128, 4),      # fp32 pages
    (32, torch.bfloat16, 64, 4),      # head dim 64
    (64, torch.bfloat16, 128, 1),     # G = 1 (generic kernel)
    (7, torch.bfloat16, 128, 16),     # odd page size
])
def test_paged_generic_paths(cuda_device, ps, dtype, D, G):
    case = inputs.paged_case(2, 2 * G, 2, D, ps, 300 // ps + 1, dtype=dtype, seed=ps,
                             seqlens=[300 - 300 % ps, 123])
    for ns in [1, 3]:
        _check(case, ns, f"ps={ps} {dtype} D={D} G={G} ns={ns}")


def test_paged_shared_prefix_and_empty(cuda_device):
    case = inputs.paged_case(4, 16, 2, 128, 64, 8, seed=3, seqlens=[512, 0, 300, 65],
                             shared_prefix_pages=3)
    for ns in [0, 1, 4]:
        _check(case, ns, f"shared prefix ns={ns}")


def test_paged_batch1_64k_matches_oracle_and_contiguous(cuda_device):
    """The benchmark's paged layer, in the benchmark's launch configuration
    (heuristic split count): every output against the fp64 paged oracle;
    and, as a second property, scattered 64-token pages give the same result
    as the contiguous cache holding the same tokens."""
    case = inputs.paged_flash_decoding_b1(65536, 64, device="cuda")
    O, L = _run(case)
    O_ref, L_ref = oracle.paged_decode_attention_ref(to_f64(case.q), to_f64(case.k_pages),
                                                     to_f64(case.v_pages),
                                                     case.block_table.cpu().numpy(), None,
                                                     case.page_size, case.scale)
    assert_parity(to_f64(O), to_f64(L), O_ref, L_ref, torch.bfloat16, "paged b1 64K vs oracle")
    kc = case.k_pages[case.block_table.cuda().long()].reshape(1, 65536, 8, 128)
    vc = case.v_pages[case.block_table.cuda().long()].reshape(1, 65536, 8, 128)
    O2, L2 = fd.decode_attention(case.q, kc, vc, None, 0, case.scale)
    fd.check_device_error()
    assert torch.allclose(O, O2, atol=1e-6, rtol=0)
    assert torch.allclose(L, L2, atol=1e-6, rtol=0)


def test_paged_bad_page_id_is_reported(cuda_device):
    case = inputs.paged_case(2, 16, 2, 128, 64, 4, seed=4, seqlens=[256, 100])
    case.block_table[1, 1] = 1000                 # used by sequence 1 (tokens 64..99)
    sl = case.seqlens.cuda()
    for var in ["mma0", "cuda"]:
        import os
        os.environ["FD_SPLIT_VARIANT"] = var
        try:
            fd.decode_attention_paged(case.q.cuda(), case.k_pages.cuda(), case.v_pages.cuda(),
                                      case.block_table.cuda(), sl, 2, case.scale)
            with pytest.raises(FdError) as ei:
                fd.check_device_error()
            assert ei.value.status == 9
        finally:
            del os.environ["FD_SPLIT_VARIANT"]


def test_nan_past_the_lengths_is_ignored(cuda_device, variant):
    """Page rows at or past a sequence's length may hold anything, NaN
    included: the tail of its last page and every later page of its table."""
    ps, pages, lens = 64, 8, [333, 70]
    case = inputs.paged_case(2, 16, 2, 128, ps, pages, seed=21, seqlens=lens)
    for b, n in enumerate(lens):
        for p in range(pages):
            first = max(0, n - p * ps)
            if first < ps:
                page = int(case.block_table[b, p])
                case.k_pages[page, first:] = float("nan")
                case.v_pages[page, first:] = float("nan")
    for ns in [0, 1, 3]:
        _check(case, ns, f"{variant} nan past lengths ns={ns}")
