"""GPU parity: bifurcated attention (shared context + per-sample decode
tokens) against the fp64 oracle, at small shapes spanning several tiles with
ragged decode lengths, and at the single-context MQA sampling workload."""

import numpy as np
import pytest
import torch

import oracle
import decode_attention_20_b300 as fd
from decode_attention_20_b300 import inputs

from _convert import assert_parity, to_f64

pytestmark = pytest.mark.gpu


def _ref(case):
    lens = None if case.dec_lens is None else case.dec_lens.numpy()
    return oracle.bifurcated_attention_ref(to_f64(case.q), to_f64(case.k_ctx), to_f64(case.v_ctx),
                                           to_f64(case.k_dec), to_f64(case.v_dec), lens, case.scale)


def _run(case, ctx_splits=0):
    dl = case.dec_lens.cuda() if case.dec_lens is not None else None
    O, L = fd.bifurcated_attention(case.q.cuda(), case.k_ctx.cuda(), case.v_ctx.cuda(),
                                   case.k_dec.cuda(), case.v_dec.cuda(), dl, case.scale,
                                   ctx_splits=ctx_splits, return_lse=True)
    fd.check_device_error()
    return O, L


@pytest.mark.parametrize("hkv,G", [(1, 32), (1, 8), (2, 4), (2, 16), (1, 3)])
@pytest.mark.parametrize("ctx_splits", [0, 1, 3])
def test_bifurcated_small(cuda_device, hkv, G, ctx_splits):
    case = inputs.bifurcated_case(5, hkv * G, hkv, 128, 300, 70, seed=31 + G,
                                  dec_lens=[70, 0, 1, 33, 64])
    O, L = _run(case, ctx_splits)
    O_ref, L_ref = _ref(case)
    assert_parity(to_f64(O), to_f64(L), O_ref, L_ref, torch.bfloat16, f"hkv={hkv} G={G}")


def test_bifurcated_no_decode_tokens_is_plain_decode(cuda_device):
    case = inputs.bifurcated_case(1, 16, 2, 128, 257, 8, seed=40, dec_lens=[0])
    O, L = _run(case)
    O2, L2 = fd.decode_attention(case.q.cuda(), case.k_ctx.unsqueeze(0).cuda(),
                                 case.v_ctx.unsqueeze(0).cuda(), None, 1, case.scale)
    O_ref, L_ref = _ref(case)
    assert_parity(to_f64(O), to_f64(L), O_ref, L_ref, torch.bfloat16, "n=1 dec=0")
    assert_parity(to_f64(O2), to_f64(L2), O_ref, L_ref, torch.bfloat16, "plain decode")


def test_bifurcated_head_dim_64(cuda_device):
    case = inputs.bifurcated_case(3, 8, 1, 64, 200, 40, seed=41, ragged_dec=(0, 40))
    O, L = _run(case)
    O_ref, L_ref = _ref(case)
    assert_parity(to_f64(O), to_f64(L), O_ref, L_ref, torch.bfloat16, "D=64")


def test_bifurcated_mqa_sampling_workload(cuda_device):
    """n = 64 samples, shared context of 8192 tokens, 256 decode tokens each,
    32 query heads on 1 kv head: every output checked, and the
    replicated-context decode path gives the same answer."""
    case = inputs.bifurcated_mqa(device="cuda")
    O, L = _run(case)
    O_ref, L_ref = _ref(case)
    assert_parity(to_f64(O), to_f64(L), O_ref, L_ref, torch.bfloat16, "bifurcated MQA")
    rep = inputs.replicate_context(case)
    O2, L2 = fd.decode_attention(rep.q, rep.k, rep.v, rep.seqlens.cuda(), 0, rep.scale)
    assert_parity(to_f64(O2), to_f64(L2), O_ref, L_ref, torch.bfloat16, "replicated")


# ---------------------------------------------------------------------------
# Context part on the tensor cores (default) and on the split kernel over a
# batch-broadcast view of the context (FD_BIF_CTX=split): both against the
# oracle, across M-tile tails, context tails, split counts and a peaked
# softmax that makes the running max jump (accumulator rescaling).

@pytest.fixture(params=["tc", "tc_nofold", "tc_rowio", "split"])
def ctx_path(request, monkeypatch):
    """tc: tensor-core context kernel, one partial per split, with the decode
    part folded into it where G >= 16, the query tile loaded and the partial
    rows stored by TMA where the maps apply (default); tc_nofold: the same
    with the decode part on the split kernel; tc_rowio: query rows loaded
    and partial rows stored by each thread; split: the split kernel over a
    broadcast view of the context."""
    monkeypatch.setenv("FD_BIF_CTX", "split" if request.param == "split" else "tc")
    monkeypatch.setenv("FD_BIF_FOLD", "0" if request.param == "tc_nofold" else "1")
    rowio = "0" if request.param == "tc_rowio" else "1"
    monkeypatch.setenv("FD_BIF_Q_TMA", rowio)
    monkeypatch.setenv("FD_BIF_O_TMA", rowio)
    return request.param


@pytest.mark.parametrize("n,hkv,G,lc,ld,ctx_splits", [
    (5, 1, 32, 300, 70, 0),        # rows 160: two M-tiles, second one ragged
    (4, 1, 32, 256, 16, 1),        # rows 128: exactly one M-tile, whole tiles
    (40, 4, 8, 1000, 33, 0),       # GQA, 3 M-tiles per kv head, context tail of 104
    (3, 2, 64, 129, 5, 2),         # G = 64, second split holds one token
    (16, 1, 8, 4173, 20, 1),       # one split streams 33 tiles (rings wrap many times)
    (2, 1, 1, 700, 9, 0),          # G = 1
    (12, 1, 32, 2000, 17, 4),      # 4 splits of 512 tokens
    (12, 1, 32, 2000, 17, 8),      # 8 splits, the last holds 208 tokens
    (9, 2, 16, 1500, 3, 2),        # GQA, M-tile tail
    (10, 2, 12, 900, 40, 3),       # G = 12: no query / output tensor map applies
    (3, 1, 256, 500, 9, 0),        # G = 256: a query tile is half a sample's heads
])
def test_bifurcated_ctx_paths(cuda_device, ctx_path, n, hkv, G, lc, ld, ctx_splits):
    case = inputs.bifurcated_case(n, hkv * G, hkv, 128, lc, ld, seed=n * 7 + G,
                                  ragged_dec=(0, ld))
    O, L = _run(case, ctx_splits)
    O_ref, L_ref = _ref(case)
    assert_parity(to_f64(O), to_f64(L), O_ref, L_ref, torch.bfloat16,
                  f"{ctx_path} n={n} hkv={hkv} G={G} lc={lc} ns={ctx_splits}")


@pytest.mark.parametrize("ctx_splits", [0, 1])
def test_bifurcated_peaked_context(cuda_device, ctx_path, ctx_splits):
    """Context keys at a seeded 2% of positions scaled by 8 (exact in bf16):
    scores jump late in a split, so the running max moves by far more than
    the lazy-rescale threshold."""
    case = inputs.bifurcated_case(8, 32, 1, 128, 2048, 40, seed=77, ragged_dec=(1, 40))
    gen = torch.Generator().manual_seed(78)
    pos = torch.randperm(2048, generator=gen)[:41]
    case.k_ctx[pos] = case.k_ctx[pos] * 8
    O, L = _run(case, ctx_splits)
    O_ref, L_ref = _ref(case)
    assert_parity(to_f64(O), to_f64(L), O_ref, L_ref, torch.bfloat16,
                  f"{ctx_path} peaked ns={ctx_splits}")


@pytest.mark.parametrize("scale", [-0.07, 0.0, 0.3])
def test_bifurcated_scale_sign_and_zero(cuda_device, ctx_path, scale):
    """A negative scale (the tensor-core path negates Q in the MMA), a zero
    scale (uniform weights) and a large one."""
    case = inputs.bifurcated_case(6, 16, 1, 128, 700, 20, seed=91, ragged_dec=(0, 20),
                                  scale=scale)
    O, L = _run(case)
    O_ref, L_ref = _ref(case)
    assert_parity(to_f64(O), to_f64(L), O_ref, L_ref, torch.bfloat16, f"{ctx_path} scale={scale}")


@pytest.mark.parametrize("n,G,ld,dec_lens", [
    (8, 16, 300, [300, 0, 129, 128, 127, 1, 256, 299]),   # 8 samples per tile, every tail kind
    (7, 24, 260, [260, 3, 0, 131, 200, 259, 64]),          # samples straddle query tiles
    (5, 48, 400, [0, 0, 0, 0, 0]),                         # no decode token anywhere
    (3, 32, 130, None),                                    # all Ld
    (11, 64, 200, [5, 199, 128, 0, 77, 200, 1, 2, 150, 129, 64]),
])
@pytest.mark.parametrize("ctx_splits", [0, 1, 4, 40])
def test_decode_folded_into_context_kernel(cuda_device, monkeypatch, n, G, ld, dec_lens, ctx_splits):
    """The decode part streamed by the context kernel: decode tiles of every
    length, samples spanning two query tiles, empty decode histories, NaN
    left in the caches past each sample's length (never used), and the
    tile list of a query tile cut into 1, 4 or 40 runs (40: some splits get
    nothing) or the library's count."""
    monkeypatch.setenv("FD_BIF_CTX", "tc")
    monkeypatch.setenv("FD_BIF_FOLD", "1")
    case = inputs.bifurcated_case(n, G, 1, 128, 700, ld, seed=n * 13 + G, dec_lens=dec_lens)
    lens = [ld] * n if dec_lens is None else dec_lens
    for i, L in enumerate(lens):
        case.k_dec[i, L:] = float("nan")
        case.v_dec[i, L:] = float("nan")
    O, L = _run(case, ctx_splits)
    O_ref, L_ref = _ref(case)
    assert_parity(to_f64(O), to_f64(L), O_ref, L_ref, torch.bfloat16,
                  f"fold n={n} G={G} ld={ld} ns={ctx_splits}")


@pytest.mark.parametrize("lc,ctx_splits", [(1, 0), (57, 0), (57, 3), (127, 2)])
def test_decode_folded_with_context_shorter_than_a_tile(cuda_device, monkeypatch, lc, ctx_splits):
    """The folded decode part when the whole shared context is shorter than
    one 128-token tile: the context run of every query tile is a single
    partial tile (one token at the least), followed by the samples' decode
    tiles; split counts that leave some runs with decode tiles only."""
    monkeypatch.setenv("FD_BIF_CTX", "tc")
    monkeypatch.setenv("FD_BIF_FOLD", "1")
    case = inputs.bifurcated_case(9, 32, 1, 128, lc, 300, seed=lc + 5,
                                  dec_lens=[300, 1, 0, 129, 128, 257, 64, 2, 299])
    O, L = _run(case, ctx_splits)
    O_ref, L_ref = _ref(case)
    assert_parity(to_f64(O), to_f64(L), O_ref, L_ref, torch.bfloat16,
                  f"short context lc={lc} ns={ctx_splits}")


@pytest.mark.parametrize("ctx_splits", [0, 1, 5])
def test_decode_folded_with_peaked_decode_keys(cuda_device, monkeypatch, ctx_splits):
    """Decode keys scaled by 8 (exact in bf16) at a seeded 5% of each
    sample's own positions: the running maximum jumps inside a sample's
    decode tiles, after the context tiles of the same run, so the O
    accumulator is rescaled mid-run for some rows and not for others."""
    monkeypatch.setenv("FD_BIF_CTX", "tc")
    monkeypatch.setenv("FD_BIF_FOLD", "1")
    case = inputs.bifurcated_case(12, 32, 1, 128, 1000, 384, seed=91,
                                  dec_lens=[384, 200, 0, 1, 383, 256, 129, 64, 300, 17, 128, 250])
    gen = torch.Generator().manual_seed(92)
    for i, n in enumerate(case.lens):
        if n:
            pos = torch.randperm(n, generator=gen)[:max(1, n // 20)]
            case.k_dec[i, pos] = case.k_dec[i, pos] * 8
    O, L = _run(case, ctx_splits)
    O_ref, L_ref = _ref(case)
    assert_parity(to_f64(O), to_f64(L), O_ref, L_ref, torch.bfloat16,
                  f"peaked decode keys ns={ctx_splits}")
