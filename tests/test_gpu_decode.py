"""GPU parity: split-KV decode attention (C ABI through the Python binding)
against the fp64 oracle on the same seeded inputs.  Sizes span several
64-token tiles with ragged tails; edge cases cover empty histories, empty
splits, every group-size variant, strided and misaligned caches and
out-of-range lengths."""

import numpy as np
import pytest
import torch

import oracle
import decode_attention_20_b300 as fd
from decode_attention_20_b300 import inputs
from decode_attention_20_b300.api import FdError

from _convert import assert_parity, to_f64

pytestmark = pytest.mark.gpu

VARIANTS = ["mma0", "mma1", "mma2", "cuda"]


@pytest.fixture(params=VARIANTS)
def variant(request, monkeypatch):
    """Split-kernel variant (tensor-core tilings or the CUDA-core kernel)."""
    monkeypatch.setenv("FD_SPLIT_VARIANT", request.param)
    return request.param


def _lens_np(case):
    return None if case.seqlens is None else case.seqlens.numpy()


def _run(case, ns=0):
    q, k, v = case.q.cuda(), case.k.cuda(), case.v.cuda()
    sl = case.seqlens.cuda() if case.seqlens is not None else None
    O, L = fd.decode_attention(q, k, v, sl, num_splits=ns, scale=case.scale)
    fd.check_device_error()
    return O, L


def _check(case, ns=0, label=""):
    O, L = _run(case, ns)
    O_ref, L_ref = oracle.decode_attention_ref(to_f64(case.q), to_f64(case.k), to_f64(case.v),
                                               _lens_np(case), case.scale)
    assert_parity(to_f64(O), to_f64(L), O_ref, L_ref, case.k.dtype, label or case.name)


@pytest.mark.parametrize("ns", [1, 4, 0])
def test_tiny_mha_fp32(cuda_device, ns):
    _check(inputs.tiny_mha(), ns, f"tiny ns={ns}")


@pytest.mark.parametrize("L", [512, 1024, 4096, 16384])
def test_flash_decoding_b1_lengths(cuda_device, L):
    _check(inputs.flash_decoding_b1(L), 0)


@pytest.mark.parametrize("ns", [1, 2, 5, 16, 37, 64, 128])
def test_flash_decoding_b1_split_sweep(cuda_device, variant, ns):
    _check(inputs.flash_decoding_b1(8192, seed=3), ns, f"L8192 ns={ns}")


@pytest.mark.parametrize("G", [1, 2, 4, 8, 16, 32, 64])
@pytest.mark.parametrize("ns", [1, 3])
def test_group_sizes_tma_path(cuda_device, variant, G, ns):
    case = inputs.decode_case(2, 2 * G, 2, 128, 300, seed=G, seqlens=[300, 77])
    _check(case, ns, f"{variant} G={G} ns={ns}")


@pytest.mark.parametrize("dtype,D,G,Lcap", [
    (torch.bfloat16, 64, 4, 300),     # head dim 64
    (torch.float32, 128, 4, 300),     # fp32 cache
    (torch.bfloat16, 128, 8, 50),     # shorter than one tile
    (torch.bfloat16, 128, 3, 200),    # group size without a TMA variant
    (torch.float32, 64, 1, 129),
])
@pytest.mark.parametrize("ns", [1, 4])
def test_generic_paths(cuda_device, dtype, D, G, Lcap, ns):
    case = inputs.decode_case(2, 2 * G, 2, D, Lcap, dtype=dtype, seed=7, seqlens=[Lcap, Lcap // 3])
    _check(case, ns, f"{dtype} D={D} G={G} L={Lcap} ns={ns}")


def test_q_fp32_with_bf16_cache(cuda_device):
    case = inputs.decode_case(1, 16, 2, 128, 400, dtype=torch.bfloat16, q_dtype=torch.float32, seed=9)
    _check(case, 3)


def test_seqlens_edges(cuda_device, variant):
    case = inputs.decode_case(4, 16, 2, 128, 200, seed=11, seqlens=[0, 1, 200, 65])
    for ns in [1, 2, 7]:
        _check(case, ns, f"edges ns={ns}")


def test_many_empty_splits(cuda_device, variant):
    case = inputs.decode_case(1, 8, 1, 128, 512, seed=12)
    _check(case, 256, "ns=256 over 512 tokens")


def test_partials_match_oracle_per_split(cuda_device, variant):
    """Each split's partial (O_i, lse_i) equals exact attention over exactly
    the oracle's [begin_i, end_i): pins the partition bounds on the device."""
    for case, nss in [
        (inputs.decode_case(2, 16, 2, 128, 1000, seed=13, seqlens=[1000, 333]), [1, 3, 4, 7, 16]),
        (inputs.decode_case(1, 4, 4, 64, 256, dtype=torch.float32, seed=14), [4, 5]),
    ]:
        q, k, v = case.q.cuda(), case.k.cuda(), case.v.cuda()
        sl = case.seqlens.cuda() if case.seqlens is not None else None
        for ns in nss:
            po, pl = fd.decode_attention_partials(q, k, v, ns, sl, case.scale)
            torch.cuda.synchronize()
            Or, Lr = oracle.split_partials_ref(to_f64(case.q), to_f64(case.k), to_f64(case.v),
                                               _lens_np(case), case.scale, ns)
            assert_parity(to_f64(po), to_f64(pl), Or, Lr, case.k.dtype, f"partials ns={ns}")


def test_strided_cache_layout(cuda_device, variant):
    """Cache stored head-major [B, Hkv, L, D] and passed as a [B, L, Hkv, D]
    view: the tensor maps take the strides as given."""
    case = inputs.decode_case(2, 16, 2, 128, 700, seed=15, seqlens=[700, 123])
    kt = case.k.permute(0, 2, 1, 3).contiguous().cuda()   # [B, Hkv, L, D]
    vt = case.v.permute(0, 2, 1, 3).contiguous().cuda()
    k_view = kt.permute(0, 2, 1, 3)
    v_view = vt.permute(0, 2, 1, 3)
    assert not k_view.is_contiguous()
    O, L = fd.decode_attention(case.q.cuda(), k_view, v_view, case.seqlens.cuda(), 5, case.scale)
    O_ref, L_ref = oracle.decode_attention_ref(to_f64(case.q), to_f64(case.k), to_f64(case.v),
                                               _lens_np(case), case.scale)
    assert_parity(to_f64(O), to_f64(L), O_ref, L_ref, torch.bfloat16, "head-major cache")


def test_misaligned_cache_uses_plain_loads(cuda_device):
    case = inputs.decode_case(1, 8, 1, 128, 300, seed=16)
    big_k = torch.zeros((1, 300, 1, 129), dtype=torch.bfloat16, device="cuda")
    big_v = torch.zeros_like(big_k)
    big_k[..., 1:] = case.k.cuda()
    big_v[..., 1:] = case.v.cuda()
    k, v = big_k[..., 1:], big_v[..., 1:]                 # 2-byte offset, odd strides
    O, L = fd.decode_attention(case.q.cuda(), k, v, None, 3, case.scale)
    O_ref, L_ref = oracle.decode_attention_ref(to_f64(case.q), to_f64(case.k), to_f64(case.v),
                                               None, case.scale)
    assert_parity(to_f64(O), to_f64(L), O_ref, L_ref, torch.bfloat16, "misaligned")


def test_strided_q_and_out(cuda_device):
    case = inputs.decode_case(2, 16, 2, 128, 256, seed=17)
    qbig = torch.zeros((2, 16, 256), dtype=torch.bfloat16, device="cuda")
    qbig[..., :128] = case.q.cuda()
    out_big = torch.full((2, 16, 200), 7.0, device="cuda")
    out = out_big[..., 10:138]
    lse_big = torch.full((2, 40), 7.0, device="cuda")
    lse = lse_big[:, 4:20]
    fd.decode_attention(qbig[..., :128], case.k.cuda(), case.v.cuda(), None, 2, case.scale,
                        out=out, lse=lse)
    O_ref, L_ref = oracle.decode_attention_ref(to_f64(case.q), to_f64(case.k), to_f64(case.v),
                                               None, case.scale)
    assert_parity(to_f64(out), to_f64(lse), O_ref, L_ref, torch.bfloat16, "strided q/out")
    assert torch.all(out_big[..., :10] == 7.0) and torch.all(out_big[..., 138:] == 7.0)
    assert torch.all(lse_big[:, :4] == 7.0) and torch.all(lse_big[:, 20:] == 7.0)


def test_bounded_wait_running_out_is_reported_and_the_context_survives(cuda_device, monkeypatch):
    """The bounded-wait error path of the tensor-core split kernel.  Under
    the test knobs its producer thread spins 200 us before issuing its first
    copies while every other thread may wait only 1 us for them, so those
    waits run out: the kernel sets the device error word, drains the copies
    it issued (those waits keep the full limit), writes empty partials and
    returns.  Nothing faults and nothing is left waiting; the host reads
    FD_ERR_DEVICE_TIMEOUT, and the next call without the knobs matches the
    oracle."""
    case = inputs.decode_case(1, 8, 1, 128, 4096, seed=19)
    q, k, v = case.q.cuda(), case.k.cuda(), case.v.cuda()
    monkeypatch.delenv("FD_SPLIT_VARIANT", raising=False)
    fd.check_device_error()                              # start clean
    monkeypatch.setenv("FD_TEST_WAIT_LIMIT_NS", "1000")
    monkeypatch.setenv("FD_TEST_PRODUCER_DELAY_NS", "200000")
    fd.decode_attention(q, k, v, None, 4, case.scale)
    with pytest.raises(FdError) as ei:
        fd.check_device_error()
    assert ei.value.status_name == "FD_ERR_DEVICE_TIMEOUT"
    monkeypatch.delenv("FD_TEST_WAIT_LIMIT_NS")
    monkeypatch.delenv("FD_TEST_PRODUCER_DELAY_NS")
    fd.check_device_error()                              # the word was cleared
    O, L = fd.decode_attention(q, k, v, None, 4, case.scale)
    fd.check_device_error()
    O_ref, L_ref = oracle.decode_attention_ref(to_f64(case.q), to_f64(case.k), to_f64(case.v),
                                               None, case.scale)
    assert_parity(to_f64(O), to_f64(L), O_ref, L_ref, torch.bfloat16, "after the timeout")


def test_out_of_range_seqlens_are_clamped_and_flagged(cuda_device):
    case = inputs.decode_case(3, 8, 1, 128, 150, seed=18)
    sl = torch.tensor([-5, 10 ** 6, 40], dtype=torch.int32)
    fd.check_device_error()                              # start clean
    O, L = fd.decode_attention(case.q.cuda(), case.k.cuda(), case.v.cuda(), sl.cuda(), 2, case.scale)
    with pytest.raises(FdError) as ei:
        fd.check_device_error()
    assert ei.value.status_name == "FD_ERR_DEVICE_BOUNDS"
    fd.check_device_error()                              # the word was cleared
    O_ref, L_ref = oracle.decode_attention_ref(to_f64(case.q), to_f64(case.k), to_f64(case.v),
                                               [0, 150, 40], case.scale)
    assert_parity(to_f64(O), to_f64(L), O_ref, L_ref, torch.bfloat16, "clamped")


def test_empty_batch_and_empty_cache(cuda_device):
    q = torch.zeros((0, 8, 128), dtype=torch.bfloat16, device="cuda")
    k = torch.zeros((0, 64, 1, 128), dtype=torch.bfloat16, device="cuda")
    O, L = fd.decode_attention(q, k, k)
    assert O.shape == (0, 8, 128)
    q = torch.randn((2, 8, 128), device="cuda").to(torch.bfloat16)
    k = torch.zeros((2, 0, 1, 128), dtype=torch.bfloat16, device="cuda")
    O, L = fd.decode_attention(q, k, k)
    torch.cuda.synchronize()
    assert torch.all(O == 0) and torch.all(torch.isneginf(L))


def test_lse_combine_standalone(cuda_device):
    g = torch.Generator().manual_seed(19)
    R, S, D = 37, 9, 128
    po = torch.randn((R, S, D), generator=g)
    pl = torch.randn((R, S), generator=g) * 5
    pl[3, :] = -float("inf")                            # row with every split empty
    pl[5, ::2] = -float("inf")
    O, L = fd.lse_combine(po.cuda(), pl.cuda())
    O_ref, L_ref = oracle.lse_combine_ref(to_f64(po), to_f64(pl))
    assert_parity(to_f64(O), to_f64(L), O_ref, L_ref, torch.float32, "combine")


@pytest.mark.parametrize("R,S,D", [
    (1, 1, 128), (64, 37, 128), (5, 100, 128), (3, 300, 64),      # one and several load batches
    (2, 4096, 512), (4, 33, 4), (7, 20, 12), (3, 17, 512),         # widest rows, 1 and 3 chunks per row
    (1500, 9, 128), (1100, 70, 64),                                # grids of many rows
    (2048, 9, 128), (600, 1, 128), (777, 16, 128), (513, 17, 64),  # warp-per-row layout: one
    (1000, 32, 128), (900, 31, 4), (530, 20, 100),                 # and two batches, D < 128
])
def test_lse_combine_shapes(cuda_device, R, S, D):
    """Split counts and head dims across the combine's thread layouts: one
    or several batches of partial rows per thread, rows of 1 to 128 float4
    chunks (threads left over when the chunks do not divide the block),
    grids of few and many rows (a warp per row for up to 32 splits and head
    dims up to 128); empty splits hold NaN, which must not reach the
    result."""
    g = torch.Generator().manual_seed(R * 7 + S * 3 + D)
    po = torch.randn((R, S, D), generator=g)
    pl = torch.randn((R, S), generator=g) * 8
    pl[0, ::3] = -float("inf")
    po[0, ::3] = float("nan")
    if R > 2:
        pl[2, :] = -float("inf")                        # every split empty
        po[2, :] = float("nan")
    O, L = fd.lse_combine(po.cuda(), pl.cuda())
    # An empty split's row is undefined; the oracle gets zeros there.
    po_def = torch.where(torch.isneginf(pl)[..., None], torch.zeros_like(po), po)
    O_ref, L_ref = oracle.lse_combine_ref(to_f64(po_def), to_f64(pl))
    assert_parity(to_f64(O), to_f64(L), O_ref, L_ref, torch.float32, f"combine R={R} S={S} D={D}")


def test_stream_ordering_on_side_stream(cuda_device):
    case = inputs.flash_decoding_b1(2048, seed=20)
    s = torch.cuda.Stream()
    q, k, v = case.q.cuda(), case.k.cuda(), case.v.cuda()
    torch.cuda.synchronize()
    with torch.cuda.stream(s):
        O, L = fd.decode_attention(q, k, v, None, 0, case.scale)
    s.synchronize()
    O_ref, L_ref = oracle.decode_attention_ref(to_f64(case.q), to_f64(case.k), to_f64(case.v),
                                               None, case.scale)
    assert_parity(to_f64(O), to_f64(L), O_ref, L_ref, torch.bfloat16, "side stream")


def test_kernel_timing_hooks(cuda_device):
    case = inputs.flash_decoding_b1(4096, seed=21)
    q, k, v = case.q.cuda(), case.k.cuda(), case.v.cuda()
    fd.profile_enable(True)
    for _ in range(3):
        fd.decode_attention(q, k, v, None, 8, case.scale)
    n_split, ms_split = fd.profile_read(fd.FD_KERNEL_SPLIT)
    n_comb, ms_comb = fd.profile_read(fd.FD_KERNEL_COMBINE)
    fd.profile_enable(False)
    assert n_split == 3 and n_comb == 3
    assert ms_split > 0 and ms_comb > 0


def test_nan_padding_past_the_lengths_is_ignored(cuda_device, variant):
    """Cache rows at or past each sequence's length may hold anything, NaN
    included: they must not reach the output."""
    case = inputs.decode_case(2, 16, 2, 128, 400, seed=22, seqlens=[333, 70])
    k = case.k.clone()
    v = case.v.clone()
    k[0, 333:] = float("nan")
    v[0, 333:] = float("nan")
    k[1, 70:] = float("inf")
    v[1, 70:] = float("nan")
    for ns in [1, 3]:
        O, L = fd.decode_attention(case.q.cuda(), k.cuda(), v.cuda(), case.seqlens.cuda(), ns,
                                   case.scale)
        O_ref, L_ref = oracle.decode_attention_ref(to_f64(case.q), to_f64(case.k), to_f64(case.v),
                                                   _lens_np(case), case.scale)
        assert_parity(to_f64(O), to_f64(L), O_ref, L_ref, torch.bfloat16, f"{variant} nan pad ns={ns}")


def test_descriptor_cache_is_by_value(cuda_device):
    """The binding caches fd_tensor descriptors by (pointer, dtype, shape,
    strides): the same values give the same descriptor, another view of the
    same memory its own one, with that view's strides."""
    from decode_attention_20_b300 import api
    t = torch.zeros((2, 3, 4), device="cuda")
    a = api._desc(t, "t")
    assert api._desc(t.view(2, 3, 4), "t") is a
    v = t.transpose(0, 1)
    d = api._desc(v, "v")
    assert d is not a
    assert [d.shape[i] for i in range(3)] == list(v.shape)
    assert [d.stride[i] for i in range(3)] == list(v.stride())
    assert d.data == a.data == t.data_ptr()
