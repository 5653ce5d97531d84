"""GPU parity: multi-token decode attention (fd_decode_attention_multi:
several new query positions per sequence, each attending causally to the
history up to itself) against the fp64 oracle on the same seeded inputs.
Covers 1..8 query tokens, group sizes with and without a tensor-core
tiling (rows = tokens x group size up to 64 on the tensor cores, beyond on
the CUDA-core kernel), histories shorter than the number of new tokens,
split counts whose last split ends inside the new tokens, strided outputs
and the batch-1 64K-token layer."""

import numpy as np
import pytest
import torch

import oracle
import decode_attention_20_b300 as fd
from decode_attention_20_b300 import inputs

from _convert import assert_parity, to_f64

pytestmark = pytest.mark.gpu


@pytest.fixture(params=["default", "cuda"])
def path(request, monkeypatch):
    if request.param == "cuda":
        monkeypatch.setenv("FD_SPLIT_VARIANT", "cuda")
    else:
        monkeypatch.delenv("FD_SPLIT_VARIANT", raising=False)
    return request.param


def _run(c, ns=0, out=None, lse=None):
    sl = c.seqlens.cuda() if c.seqlens is not None else None
    O, L = fd.decode_attention_multi(c.q.cuda(), c.k.cuda(), c.v.cuda(), sl, num_splits=ns,
                                     scale=c.scale, out=out, lse=lse)
    fd.check_device_error()
    return O, L


def _check(c, ns=0, label=""):
    O, L = _run(c, ns)
    lens = None if c.seqlens is None else c.seqlens.numpy()
    O_ref, L_ref = oracle.multi_token_decode_ref(to_f64(c.q), to_f64(c.k), to_f64(c.v), lens, c.scale)
    assert_parity(to_f64(O), to_f64(L), O_ref, L_ref, c.k.dtype, label or c.name)


@pytest.mark.parametrize("tq", [1, 2, 3, 4, 8])
@pytest.mark.parametrize("G", [1, 4, 8])
@pytest.mark.parametrize("ns", [1, 3, 0])
def test_tokens_groups_splits(cuda_device, path, tq, G, ns):
    c = inputs.multi_token_case(3, tq, 2 * G, 2, 128, 700, seed=tq * 10 + G,
                                seqlens=[700, 129, max(1, tq - 1)])
    _check(c, ns, f"{path} tq={tq} G={G} ns={ns}")


@pytest.mark.parametrize("tq,G", [(8, 16), (5, 16), (3, 32)])
def test_more_rows_than_the_tensor_core_tiles(cuda_device, tq, G):
    c = inputs.multi_token_case(2, tq, 2 * G, 2, 128, 500, seed=tq + G, seqlens=[500, 300])
    _check(c, 0, f"tq={tq} G={G}")


@pytest.mark.parametrize("dtype,D", [(torch.float32, 128), (torch.bfloat16, 64)])
def test_generic_dtypes(cuda_device, dtype, D):
    c = inputs.multi_token_case(2, 4, 8, 2, D, 300, dtype=dtype, seed=5, seqlens=[300, 64])
    _check(c, 3, f"{dtype} D={D}")


def test_splits_ending_inside_the_new_tokens(cuda_device, path):
    """ns chosen so that split boundaries fall among the last Tq tokens."""
    c = inputs.multi_token_case(1, 8, 64, 8, 128, 4096 + 5, seed=2)
    for ns in [1, 2, 64, 65]:
        _check(c, ns, f"{path} boundaries ns={ns}")


def test_single_token_matches_plain_decode(cuda_device):
    c = inputs.multi_token_case(2, 1, 64, 8, 128, 3000, seed=9, seqlens=[3000, 1500])
    O1, L1 = _run(c, 0)
    sl = c.seqlens.cuda()
    O2, L2 = fd.decode_attention(c.q[:, 0].cuda(), c.k.cuda(), c.v.cuda(), sl, scale=c.scale)
    assert torch.equal(O1[:, 0], O2) and torch.equal(L1[:, 0], L2)


def test_strided_outputs(cuda_device):
    c = inputs.multi_token_case(2, 3, 16, 2, 128, 800, seed=11, seqlens=[800, 2])
    big = torch.full((2, 3, 16, 130), float("nan"), device="cuda")
    out = big[..., 1:129]                       # rows not 16-byte aligned
    lse_big = torch.full((2, 3, 18), float("nan"), device="cuda")
    lse = lse_big[..., 1:17]                    # unit inner stride, odd offset
    _run(c, 4, out=out, lse=lse)
    O_ref, L_ref = oracle.multi_token_decode_ref(to_f64(c.q), to_f64(c.k), to_f64(c.v),
                                                 c.seqlens.numpy(), c.scale)
    assert_parity(to_f64(out), to_f64(lse), O_ref, L_ref, c.k.dtype, "strided")
    assert torch.isnan(big[..., 0]).all() and torch.isnan(big[..., 129]).all()


@pytest.mark.parametrize("tq", [2, 4])
def test_full_size_verification_b1(cuda_device, tq):
    """Batch 1, 65536 cached tokens, 64 query heads over 8 kv heads (the
    benchmark's verification workload) against the oracle, every row."""
    c = inputs.speculative_b1(65536, tq=tq, device="cuda")
    O, L = _run(c, 0)
    O_ref, L_ref = oracle.multi_token_decode_ref(to_f64(c.q), to_f64(c.k), to_f64(c.v), None, c.scale)
    assert_parity(to_f64(O), to_f64(L), O_ref, L_ref, c.k.dtype, f"verify tq={tq}")


def test_nan_padding_past_the_lengths_is_ignored(cuda_device, path):
    """Cache rows at or past a sequence's length may hold anything, NaN
    included: the partial last tile of a split clears them before the PV
    product, and the causal limits keep them out of the scores."""
    c = inputs.multi_token_case(2, 4, 16, 2, 128, 700, seed=77, seqlens=[333, 70])
    for b, n in enumerate([333, 70]):
        c.k[b, n:] = float("nan")
        c.v[b, n:] = float("nan")
    for ns in (1, 3, 0):
        _check(c, ns, f"{path} nan past lengths ns={ns}")
