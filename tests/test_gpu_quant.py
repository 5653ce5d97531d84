"""GPU parity: decode attention over an 8-bit KV cache (int8 or e4m3 codes,
one scale per kv head; fd_decode_attention_quant) against the fp64 oracle on
the same seeded inputs.  Sizes span several 128-token tiles with ragged
tails; edge cases cover empty histories, every group-size variant, the
CUDA-core fallback, f32 queries, extreme query magnitudes, NaN codes past
the lengths, signs and zeros of the scales, and out-of-range lengths.

Tolerance.  The kernels turn every code into its exact f16 value, so the
dequantised K and V are exact; what rounds is the probability p (f16, 11
significant bits, relative error <= 2^-11) and the fp32 accumulations.  The
output error is then at most about 2^-11 * max |V| (V dequantised); the
tests ask for 2^-10 * max |V| + 1e-5 with bf16 queries (exact in f16 after
the per-head power-of-two rescale) and the bf16-cache tolerances (max 2e-2,
mean 2e-3) with f32 queries, whose f16 rounding perturbs the scores.  LSE
within 1e-3 as everywhere."""

import numpy as np
import pytest
import torch

import oracle
import decode_attention_20_b300 as fd
from decode_attention_20_b300 import inputs
from decode_attention_20_b300.api import FdError

from _convert import TOL_BF16_MAX, TOL_BF16_MEAN, TOL_LSE, to_f64

pytestmark = pytest.mark.gpu

KINDS = ["int8", "e4m3"]


@pytest.fixture(params=["mma", "mma0", "mma2", "cuda"])
def path(request, monkeypatch):
    """Tensor-core split kernel: the default tiling (8 warps, 128-token
    tiles for 8-bit caches), the 4-warp 128-token one (mma0), the 64-token
    6-stage one (mma2); or the CUDA-core kernel."""
    if request.param == "mma":
        monkeypatch.delenv("FD_SPLIT_VARIANT", raising=False)
    else:
        monkeypatch.setenv("FD_SPLIT_VARIANT", request.param)
    return request.param


def _codes_np(t):
    t = t.detach().cpu().contiguous()
    if t.dtype == torch.float8_e4m3fn:
        return t.view(torch.uint8).numpy()
    return t.numpy()


def _oracle(c):
    lens = None if c.seqlens is None else c.seqlens.numpy()
    return oracle.quant_decode_attention_ref(to_f64(c.q), _codes_np(c.k), _codes_np(c.v),
                                             c.k_scale.cpu().numpy(), c.v_scale.cpu().numpy(),
                                             c.kind, lens, c.scale)


def _run(c, ns=0, k=None, v=None):
    k = c.k.cuda() if k is None else k
    v = c.v.cuda() if v is None else v
    sl = c.seqlens.cuda() if c.seqlens is not None else None
    O, L = fd.decode_attention_quant(c.q.cuda(), k, v, c.k_scale.cuda(), c.v_scale.cuda(), sl,
                                     num_splits=ns, scale=c.scale)
    fd.check_device_error()
    return to_f64(O), to_f64(L)


def _assert(c, O, L, O_ref, L_ref, label):
    assert O.shape == O_ref.shape
    assert np.all(np.isfinite(O)), f"{label}: non-finite output"
    err = np.abs(O - O_ref)
    if c.q.dtype == torch.bfloat16:
        vmax = float(np.nanmax(np.abs(oracle.dequantize_kv_ref(_codes_np(c.v), c.v_scale.cpu().numpy(), c.kind))))
        tol = 2.0 ** -10 * vmax + 1e-5
        assert err.max() <= tol, f"{label}: max |dO| {err.max():.3e} > {tol:.3e}"
    else:
        assert err.max() <= TOL_BF16_MAX, f"{label}: max |dO| {err.max():.3e}"
        assert err.mean() <= TOL_BF16_MEAN, f"{label}: mean |dO| {err.mean():.3e}"
    inf_ref = np.isneginf(L_ref)
    assert np.array_equal(np.isneginf(L), inf_ref), f"{label}: -inf pattern differs"
    if (~inf_ref).any():
        d = np.abs(L[~inf_ref] - L_ref[~inf_ref])
        assert d.max() <= TOL_LSE, f"{label}: max |dLSE| {d.max():.3e}"
    assert np.all(O[inf_ref] == 0), f"{label}: empty rows must be exactly 0"


def _check(c, ns=0, label=""):
    O, L = _run(c, ns)
    O_ref, L_ref = _oracle(c)
    _assert(c, O, L, O_ref, L_ref, label or c.name)


@pytest.mark.parametrize("kind", KINDS)
@pytest.mark.parametrize("L", [512, 4096, 16384])
def test_b1_lengths(cuda_device, kind, L):
    _check(inputs.quant_flash_decoding_b1(L, kind=kind, seed=L), 0, f"{kind} L={L}")


@pytest.mark.parametrize("kind", KINDS)
@pytest.mark.parametrize("ns", [1, 2, 5, 37, 128])
def test_split_sweep(cuda_device, path, kind, ns):
    c = inputs.quant_case(1, 64, 8, 128, 8192, kind=kind, seed=3)
    _check(c, ns, f"{path} {kind} ns={ns}")


@pytest.mark.parametrize("kind", KINDS)
@pytest.mark.parametrize("G", [1, 2, 4, 8, 16, 32, 64])
@pytest.mark.parametrize("ns", [1, 3])
def test_group_sizes(cuda_device, path, kind, G, ns):
    c = inputs.quant_case(2, 2 * G, 2, 128, 700, kind=kind, seed=G, seqlens=[700, 77])
    _check(c, ns, f"{path} {kind} G={G} ns={ns}")


@pytest.mark.parametrize("kind", KINDS)
@pytest.mark.parametrize("D,G,Lcap,q_dtype", [
    (64, 4, 300, torch.bfloat16),     # head dim 64: CUDA-core kernel
    (128, 3, 300, torch.bfloat16),    # group size without a tensor-core variant
    (128, 8, 100, torch.bfloat16),    # shorter than one 128-token tile
    (128, 8, 1000, torch.float32),    # f32 queries on the tensor-core kernel
    (64, 2, 129, torch.float32),
])
@pytest.mark.parametrize("ns", [1, 4])
def test_other_shapes(cuda_device, kind, D, G, Lcap, q_dtype, ns):
    c = inputs.quant_case(2, 2 * G, 2, D, Lcap, kind=kind, seed=9, seqlens=[Lcap, Lcap // 3],
                          q_dtype=q_dtype)
    _check(c, ns, f"{kind} D={D} G={G} Lcap={Lcap} {q_dtype}")


@pytest.mark.parametrize("kind", KINDS)
def test_ragged_batch(cuda_device, path, kind):
    c = inputs.quant_case(6, 32, 8, 128, 3000, kind=kind, seed=21, ragged=(0, 3000))
    _check(c, 0, f"{path} {kind} ragged")


@pytest.mark.parametrize("kind", KINDS)
def test_empty_and_short_histories(cuda_device, path, kind):
    c = inputs.quant_case(5, 16, 2, 128, 1000, kind=kind, seed=4, seqlens=[0, 1, 127, 129, 1000])
    for ns in [1, 7, 0]:
        _check(c, ns, f"{path} {kind} short ns={ns}")


@pytest.mark.parametrize("kind", KINDS)
@pytest.mark.parametrize("exp", [-60, -20, 20, 60])
def test_query_magnitudes(cuda_device, path, kind, exp):
    """Queries times 2^exp (exact in bf16) with the score scale times 2^-exp:
    the same scores, through the kernel's per-head query rescale."""
    c = inputs.quant_case(2, 16, 2, 128, 600, kind=kind, seed=30 + exp, seqlens=[600, 311])
    c.q = c.q * (2.0 ** exp)
    c.scale = c.scale * 2.0 ** -exp
    _check(c, 0, f"{path} {kind} q*2^{exp}")


@pytest.mark.parametrize("kind", KINDS)
@pytest.mark.parametrize("scale", [-0.125, 0.0, 0.7])
def test_score_scale_sign_and_zero(cuda_device, kind, scale):
    c = inputs.quant_case(2, 16, 2, 128, 500, kind=kind, seed=12, seqlens=[500, 250], scale=scale)
    _check(c, 0, f"{kind} scale={scale}")


def test_e4m3_nan_codes_past_lengths_unused(cuda_device, path):
    c = inputs.quant_case(3, 16, 2, 128, 900, kind="e4m3", seed=8, seqlens=[900, 400, 130])
    k, v = c.k.clone(), c.v.clone()
    kb, vb = k.view(torch.uint8), v.view(torch.uint8)
    for b, n in enumerate([900, 400, 130]):
        kb[b, n:] = 0x7F
        vb[b, n:] = 0xFF
    O, L = _run(c, 0, k.cuda(), v.cuda())
    O_ref, L_ref = _oracle(c)
    _assert(c, O, L, O_ref, L_ref, f"{path} NaN codes past lengths")


def test_per_head_scales_are_per_head(cuda_device):
    """Scales differing by orders of magnitude between kv heads."""
    c = inputs.quant_case(1, 32, 4, 128, 2000, kind="int8", seed=14)
    c.k_scale = torch.tensor([1e-3, 0.05, 0.3, 0.01], dtype=torch.float32)
    c.v_scale = torch.tensor([10.0, 1e-2, 1.0, 0.1], dtype=torch.float32)
    _check(c, 0, "per-head scales")


def test_lengths_outside_capacity_are_clamped_and_flagged(cuda_device):
    c = inputs.quant_case(3, 16, 2, 128, 300, kind="int8", seed=2)
    sl = torch.tensor([-5, 10 ** 6, 40], dtype=torch.int32)
    fd.check_device_error()                              # start clean
    O, L = fd.decode_attention_quant(c.q.cuda(), c.k.cuda(), c.v.cuda(), c.k_scale.cuda(),
                                     c.v_scale.cuda(), sl.cuda(), 2, c.scale)
    with pytest.raises(FdError) as ei:
        fd.check_device_error()
    assert ei.value.status_name == "FD_ERR_DEVICE_BOUNDS"
    fd.check_device_error()                              # the word was cleared
    c.seqlens = torch.tensor([0, 300, 40], dtype=torch.int32)
    O_ref, L_ref = _oracle(c)
    _assert(c, to_f64(O), to_f64(L), O_ref, L_ref, "clamped")


def test_misaligned_cache_takes_the_cuda_core_kernel(cuda_device):
    """A cache whose base is not 16-byte aligned cannot be streamed by TMA;
    the CUDA-core kernel takes it and the result must not change."""
    c = inputs.quant_case(2, 16, 2, 128, 300, kind="int8", seed=6, seqlens=[300, 100])
    big = torch.zeros((2 * 300 * 2 * 128 + 1,), dtype=torch.int8, device="cuda")
    k = big[1:].view(2, 300, 2, 128)
    k.copy_(c.k.cuda())
    O, L = _run(c, 0, k, c.v.cuda())
    O_ref, L_ref = _oracle(c)
    _assert(c, O, L, O_ref, L_ref, "misaligned")


@pytest.mark.parametrize("kind", KINDS)
def test_full_size_b1_sampled_heads(cuda_device, kind):
    """Batch 1, 65536 cached tokens (the benchmark's 8-bit workload, default
    split count): every query head against the oracle."""
    c = inputs.quant_flash_decoding_b1(65536, kind=kind, device="cuda")
    O, L = _run(c, 0)
    O_ref, L_ref = _oracle(c)
    _assert(c, O, L, O_ref, L_ref, f"{kind} b1 L=65536")
