"""The seeded input recipe, checked on the CPU: the shapes, dtypes, draw
order and value distributions that the design notes state for every
workload, so that the GPU parity tests and the benchmark are fed what the
recipe says.  (The generators hold no attention arithmetic; these tests
check layout and statistics only.)"""

import inspect
import math

import pytest
import torch

from decode_attention_20_b300 import inputs


def _draws(seed, shapes, dtype):
    """Consecutive N(0,1) float32 draws from one generator, rounded to dtype."""
    g = torch.Generator().manual_seed(seed)
    return [torch.randn(s, generator=g, dtype=torch.float32).to(dtype) for s in shapes]


def test_same_seed_same_tensors_other_seed_other_tensors():
    a = inputs.flash_decoding_b1(512, seed=5)
    b = inputs.flash_decoding_b1(512, seed=5)
    c = inputs.flash_decoding_b1(512, seed=6)
    for x, y in [(a.q, b.q), (a.k, b.k), (a.v, b.v)]:
        assert torch.equal(x, y)
    assert not torch.equal(a.k, c.k)


def test_draw_order_q_then_k_then_v():
    """Bulk tensors are consecutive N(0,1) draws of one generator, q first,
    rounded to bf16."""
    c = inputs.decode_case(2, 8, 2, 64, 96, seed=11)
    q, k, v = _draws(11, [(2, 8, 64), (2, 96, 2, 64), (2, 96, 2, 64)], torch.bfloat16)
    assert torch.equal(c.q, q) and torch.equal(c.k, k) and torch.equal(c.v, v)


def test_draw_order_multi_token_and_bifurcated():
    m = inputs.multi_token_case(1, 4, 8, 2, 64, 80, seed=3)
    q, k, v = _draws(3, [(1, 4, 8, 64), (1, 80, 2, 64), (1, 80, 2, 64)], torch.bfloat16)
    assert torch.equal(m.q, q) and torch.equal(m.k, k) and torch.equal(m.v, v)
    b = inputs.bifurcated_case(3, 8, 1, 64, 50, 20, seed=4)
    q, kc, vc, kd, vd = _draws(4, [(3, 8, 64), (50, 1, 64), (50, 1, 64), (3, 20, 1, 64),
                                   (3, 20, 1, 64)], torch.bfloat16)
    assert torch.equal(b.q, q) and torch.equal(b.k_ctx, kc) and torch.equal(b.v_ctx, vc)
    assert torch.equal(b.k_dec, kd) and torch.equal(b.v_dec, vd)


def test_named_workload_shapes():
    t = inputs.tiny_mha()
    assert t.q.shape == (1, 4, 64) and t.k.shape == (1, 256, 4, 64) and t.q.dtype == torch.float32
    assert t.scale == pytest.approx(1 / 8)
    f = inputs.flash_decoding_b1(512)
    assert f.q.shape == (1, 64, 128) and f.k.shape == (1, 512, 8, 128) and f.k.dtype == torch.bfloat16
    assert f.scale == pytest.approx(1 / math.sqrt(128))
    b = inputs.bifurcated_mqa()
    assert b.q.shape == (64, 32, 128) and b.k_ctx.shape == (8192, 1, 128)
    assert b.k_dec.shape == (64, 256, 1, 128) and b.dec_lens is None
    s = inputs.speculative_b1(256, tq=4)
    assert s.q.shape == (1, 4, 64, 128) and s.k.shape == (1, 256, 8, 128)


def test_named_workload_defaults():
    """The large workloads are too big to draw here; their defaults are the
    recipe's sizes."""
    r = inspect.signature(inputs.ragged_batch).parameters
    assert (r["batch"].default, r["lcap"].default, r["lo"].default, r["hi"].default) == (
        32, 32768, 1024, 32768)
    lp = inspect.signature(inputs.long_context_peaked).parameters
    assert (lp["batch"].default, lp["L"].default) == (4, 131072)
    pg = inspect.signature(inputs.paged_flash_decoding_b1).parameters
    assert (pg["L"].default, pg["page_size"].default) == (65536, 64)
    qf = inspect.signature(inputs.quant_flash_decoding_b1).parameters
    assert qf["L"].default == 65536


def test_values_are_standard_normal_in_bf16():
    f = inputs.flash_decoding_b1(4096, seed=1)
    x = f.k.float()
    assert abs(x.mean().item()) < 0.01
    assert abs(x.std().item() - 1.0) < 0.01
    # bf16: every value has at most 8 significant bits
    assert torch.equal(x.to(torch.bfloat16).float(), x)


def test_ragged_lengths_uniform_in_range():
    r = inputs.ragged_batch(batch=400, lcap=64, lo=10, hi=64)
    lens = r.seqlens
    assert lens.dtype == torch.int32 and lens.shape == (400,)
    assert int(lens.min()) >= 10 and int(lens.max()) <= 64
    assert len(set(lens.tolist())) > 40          # spread over the range, not a constant
    assert abs(lens.float().mean().item() - 37.0) < 3.0


def test_peaked_keys_are_exactly_eight_times_the_draw():
    """1% of each sequence's positions have their keys (every head and dim)
    multiplied by 8; everything else is the plain draw."""
    p = inputs.decode_case(2, 8, 2, 64, 1000, seed=7, peaked_frac=0.01)
    plain = inputs.decode_case(2, 8, 2, 64, 1000, seed=7)
    for b in range(2):
        pos = p.meta["peaks"][b]
        assert len(pos) == 10 and len(set(pos.tolist())) == 10
        mask = torch.zeros(1000, dtype=torch.bool)
        mask[pos] = True
        assert torch.equal(p.k[b, mask], plain.k[b, mask] * 8)
        assert torch.equal(p.k[b, ~mask], plain.k[b, ~mask])
    assert torch.equal(p.v, plain.v) and torch.equal(p.q, plain.q)


def test_paged_block_table_is_a_permutation_slice():
    c = inputs.paged_case(3, 8, 2, 64, 16, 10, num_pages=40, seed=2)
    bt = c.block_table
    assert bt.dtype == torch.int32 and bt.shape == (3, 10)
    ids = bt.flatten().tolist()
    assert len(set(ids)) == 30 and min(ids) >= 0 and max(ids) < 40   # distinct pages
    assert c.k_pages.shape == (40, 16, 2, 64)
    s = inputs.paged_case(3, 8, 2, 64, 16, 10, num_pages=40, seed=2, shared_prefix_pages=2)
    assert torch.equal(s.block_table[:, :2], s.block_table[0:1, :2].expand(3, 2))


def test_paged_b1_covers_all_pages_once():
    c = inputs.paged_case(1, 8, 2, 64, 64, 32, seed=0)           # 2048 tokens in 32 pages
    assert sorted(c.block_table[0].tolist()) == list(range(32))
    assert c.block_table[0].tolist() != list(range(32))          # scattered, not in order


def test_int8_codes_and_scales():
    c = inputs.quant_case(1, 8, 4, 128, 2048, kind="int8", seed=3)
    assert c.k.dtype == torch.int8
    x = c.k.float()
    assert int(x.min()) >= -127 and int(x.max()) <= 127
    assert abs(x.std().item() - 32.0) < 0.5                      # round(N(0, 32^2))
    for s in (c.k_scale, c.v_scale):
        assert s.shape == (4,) and s.dtype == torch.float32
        assert bool(((s >= 0.5 / 32) & (s <= 1.5 / 32)).all())


def test_e4m3_codes_and_scales():
    c = inputs.quant_case(1, 8, 4, 128, 2048, kind="e4m3", seed=3)
    assert c.k.dtype == torch.float8_e4m3fn
    bits = c.k.view(torch.uint8)
    assert not bool(((bits & 0x7F) == 0x7F).any())               # no NaN codes drawn
    assert abs(c.k.float().std().item() - 1.0) < 0.02            # N(0,1) rounded to e4m3
    for s in (c.k_scale, c.v_scale):
        assert bool(((s >= 0.5) & (s <= 1.5)).all())
