"""Pins for the fp64 CPU oracle (CPU only).

The oracle is checked against what the pages and the mathematics fix:
hand-derived worked examples (tests/golden/worked_examples.json), closed
forms, a brute-force loop oracle, library routines for special cases, and the
invariants the pages state (split + log-sum-exp combine == unsplit;
bifurcated == concatenated).
"""

import math

import numpy as np
import pytest
import torch

import oracle
from oracle import attention as oa

import _pins


# ------------------------------------------------------------------ bf16 decode

@pytest.mark.parametrize("bits,val", [
    (0x3F80, 1.0), (0xBF80, -1.0), (0x4000, 2.0), (0x3F00, 0.5), (0x3FC0, 1.5),
    (0x4049, 3.140625), (0x0000, 0.0), (0x7F80, math.inf), (0xFF80, -math.inf),
    (0x0001, 2.0 ** -133), (0x0080, 2.0 ** -126), (0x7F7F, (2 - 2 ** -7) * 2.0 ** 127),
])
def test_bf16_decode_known_patterns(bits, val):
    got = oracle.bf16_bits_to_f64(np.array([bits], np.uint16))[0]
    assert got == val


def test_bf16_negative_zero():
    got = oracle.bf16_bits_to_f64(np.array([0x8000], np.uint16))[0]
    assert got == 0.0 and math.copysign(1.0, got) < 0


def test_bf16_decode_matches_torch():
    rng = np.random.default_rng(0)
    bits = rng.integers(0, 1 << 16, size=20000, dtype=np.uint32).astype(np.uint16)
    bits = bits[(bits & 0x7F80) != 0x7F80]          # drop inf/NaN patterns
    ref = torch.from_numpy(bits.view(np.int16).copy()).view(torch.bfloat16).to(torch.float64).numpy()
    assert np.array_equal(oracle.bf16_bits_to_f64(bits), ref)


# ------------------------------------------------------------- worked examples

def test_golden_decode():
    assert _pins.golden_decode_ok(oracle.decode_attention_ref)


def test_golden_combine():
    assert _pins.golden_combine_ok(oracle.lse_combine_ref)


def test_golden_bifurcated():
    assert _pins.golden_bifurcated_ok(oracle.bifurcated_attention_ref)


# ---------------------------------------------------------------- closed forms

def test_closed_forms():
    assert _pins.closed_forms_ok(oracle.decode_attention_ref)


def test_bruteforce_tiny_shapes():
    assert _pins.bruteforce_ok(oracle.decode_attention_ref, oracle.attention_bruteforce)


def test_bruteforce_tiny_fp32_config():
    """The tiny MHA workload's shape, cut to 16 tokens, against brute force."""
    rng = np.random.default_rng(5)
    q = rng.standard_normal((1, 4, 64)).astype(np.float32).astype(np.float64)
    k = rng.standard_normal((1, 16, 4, 64)).astype(np.float32).astype(np.float64)
    v = rng.standard_normal((1, 16, 4, 64)).astype(np.float32).astype(np.float64)
    O, L = oracle.decode_attention_ref(q, k, v, None, 1 / 8)
    Ob, Lb = oracle.attention_bruteforce(q.tolist(), k.tolist(), v.tolist(), None, 1 / 8)
    np.testing.assert_allclose(O, np.array(Ob), rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(L, np.array(Lb), rtol=1e-12, atol=1e-13)


def test_weights_sum_to_one_and_reproduce_O():
    rng = np.random.default_rng(7)
    q = rng.standard_normal((2, 6, 16))
    k = rng.standard_normal((2, 50, 3, 16))
    v = rng.standard_normal((2, 50, 3, 16))
    lens = [50, 9]
    P = oracle.attention_weights_ref(q, k, lens, 0.3)
    s = P.sum(axis=-1)
    assert np.all(np.abs(s - 1.0) <= 1e-12)
    assert np.all(P[1, :, 9:] == 0)
    O, _ = oracle.decode_attention_ref(q, k, v, lens, 0.3)
    G = 2
    for b in range(2):
        for h in range(6):
            ref = P[b, h, :lens[b]] @ v[b, :lens[b], h // G]
            np.testing.assert_allclose(O[b, h], ref, rtol=1e-12, atol=1e-13)


def test_permutation_invariance():
    rng = np.random.default_rng(8)
    q = rng.standard_normal((1, 4, 8))
    k = rng.standard_normal((1, 40, 2, 8))
    v = rng.standard_normal((1, 40, 2, 8))
    O, L = oracle.decode_attention_ref(q, k, v, None, 0.5)
    perm = rng.permutation(40)
    O2, L2 = oracle.decode_attention_ref(q, k[:, perm], v[:, perm], None, 0.5)
    np.testing.assert_allclose(O2, O, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(L2, L, rtol=1e-12, atol=1e-13)


def test_peaked_softmax_large_dynamic_range():
    """Scores up to ~300 (no overflow thanks to the max shift): one dominant
    key returns its value."""
    rng = np.random.default_rng(9)
    D = 16
    q = rng.standard_normal((1, 1, D))
    k = rng.standard_normal((1, 30, 1, D))
    k[0, 11, 0] = 40 * q[0, 0] / np.linalg.norm(q[0, 0])
    v = rng.standard_normal((1, 30, 1, D))
    O, L = oracle.decode_attention_ref(q, k, v, None, 1.0)
    assert np.all(np.isfinite(O)) and np.isfinite(L).all()
    np.testing.assert_allclose(O[0, 0], v[0, 11, 0], atol=1e-12)


# ------------------------------------------------------ library special cases

def test_matches_torch_sdpa_float64():
    """Single-query MHA attention equals PyTorch's scaled_dot_product_attention
    (math path, float64 on CPU)."""
    rng = np.random.default_rng(10)
    B, H, D, L = 2, 3, 32, 70
    q = rng.standard_normal((B, H, D))
    k = rng.standard_normal((B, L, H, D))
    v = rng.standard_normal((B, L, H, D))
    O, _ = oracle.decode_attention_ref(q, k, v, None, 1 / math.sqrt(D))
    tq = torch.from_numpy(q)[:, :, None, :]                  # [B,H,1,D]
    tk = torch.from_numpy(k).permute(0, 2, 1, 3)             # [B,H,L,D]
    tv = torch.from_numpy(v).permute(0, 2, 1, 3)
    ref = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv)[:, :, 0, :].numpy()
    np.testing.assert_allclose(O, ref, rtol=1e-10, atol=1e-12)


def test_lse_matches_scipy_logsumexp():
    from scipy.special import logsumexp
    rng = np.random.default_rng(11)
    q = rng.standard_normal((1, 2, 8))
    k = rng.standard_normal((1, 25, 1, 8))
    v = rng.standard_normal((1, 25, 1, 8))
    _, L = oracle.decode_attention_ref(q, k, v, None, 0.9)
    for h in range(2):
        s = 0.9 * (k[0, :, 0] @ q[0, h])
        assert abs(L[0, h] - logsumexp(s)) <= 1e-12 * (1 + abs(L[0, h]))


def test_combine_scalar_is_logsumexp():
    from scipy.special import logsumexp
    rng = np.random.default_rng(12)
    lse = rng.standard_normal((3, 5, 9)) * 4
    o = rng.standard_normal((3, 5, 9, 4))
    O, L = oracle.lse_combine_ref(o, lse)
    np.testing.assert_allclose(L, logsumexp(lse, axis=-1), rtol=1e-13, atol=1e-13)
    w = np.exp(lse - logsumexp(lse, axis=-1, keepdims=True))
    np.testing.assert_allclose(O, (w[..., None] * o).sum(-2), rtol=1e-12, atol=1e-13)


# --------------------------------------------------- invariants from the pages

def test_split_combine_equals_unsplit():
    assert _pins.split_combine_ok(oracle.split_partials_ref, oracle.lse_combine_ref,
                                  oracle.decode_attention_ref)


def test_bifurcated_equals_concatenated():
    assert _pins.bifurcated_concat_ok(oracle.bifurcated_attention_ref,
                                      oracle.decode_attention_ref)


def test_bifurcated_single_sample_no_decode_is_plain_decode():
    rng = np.random.default_rng(13)
    q = rng.standard_normal((1, 4, 8))
    kc = rng.standard_normal((20, 1, 8))
    vc = rng.standard_normal((20, 1, 8))
    kd = rng.standard_normal((1, 3, 1, 8))
    vd = rng.standard_normal((1, 3, 1, 8))
    O, L = oracle.bifurcated_attention_ref(q, kc, vc, kd, vd, [0], 0.5)
    Or, Lr = oracle.decode_attention_ref(q, kc[None], vc[None], None, 0.5)
    np.testing.assert_allclose(O, Or, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(L, Lr, rtol=1e-12, atol=1e-13)


# ------------------------------------------------------ split bounds / heuristic

def test_split_bounds_partition_brute_force():
    A = oracle.SPLIT_ALIGN
    for length in list(range(0, 300)) + [1023, 1024, 1025, 65536, 131071, 131072]:
        for ns in [1, 2, 3, 4, 5, 7, 8, 16, 37, 64, 100, 256]:
            covered = []
            prev_end = 0
            for i in range(ns):
                lo, hi = oracle.split_bounds_ref(length, ns, i)
                assert 0 <= lo <= hi <= length
                assert lo == prev_end                       # contiguous, in order
                assert lo % A == 0 or lo == length          # aligned starts
                covered.append(hi - lo)
                prev_end = hi
            assert prev_end == length and sum(covered) == length
            per = -(-length // ns) if length else 0
            chunk = -(-per // A) * A
            assert max(covered) <= max(chunk, 0)
            # chunk is the smallest multiple of A that is >= ceil(length/ns)
            assert chunk >= per and chunk - per < A


def test_split_bounds_rejects_bad_args():
    for args in [(10, 0, 0), (10, 2, 2), (10, 2, -1), (-1, 2, 0)]:
        with pytest.raises(ValueError):
            oracle.split_bounds_ref(*args)


def test_heuristic_properties():
    sms = 148
    for B in [1, 2, 4, 8, 32, 64, 256]:
        for hkv in [1, 8]:
            for L in [1, 64, 256, 512, 1024, 4096, 65536, 131072, 1 << 20]:
                ns = oracle.choose_num_splits_ref(B, hkv, L, sms)
                assert 1 <= ns <= oracle.MAX_SPLITS
                assert ns <= max(1, -(-L // oracle.MIN_CHUNK))   # chunks of >= 64 tokens
    # a history of one tile -> no splitting
    assert oracle.choose_num_splits_ref(1, 8, 64, sms) == 1
    assert oracle.choose_num_splits_ref(0, 8, 65536, 148) == 1


def _makespan(units, L, ns, sms):
    chunk = -(-(-(-L // ns)) // oracle.SPLIT_ALIGN) * oracle.SPLIT_ALIGN
    used = -(-L // chunk)
    return -(-(units * used) // (2 * sms)) * (chunk + oracle.SPLIT_OVERHEAD_TOKENS)


def test_heuristic_is_the_makespan_minimiser():
    """Brute force over every admissible ns: the choice has the lowest
    modelled makespan, and no smaller ns ties it."""
    for sms in [148, 132]:
        for units in [1, 8, 16, 32, 64, 256, 1000]:
            for L in [300, 4096, 65536, 131072]:
                ns = oracle.choose_num_splits_ref(units, 1, L, sms)
                costs = {k: _makespan(units, L, k, sms)
                         for k in range(1, min(oracle.MAX_SPLITS, -(-L // oracle.MIN_CHUNK)) + 1)}
                assert costs[ns] == min(costs.values())
                assert all(costs[k] > costs[ns] for k in costs if k < ns)


def test_heuristic_workload_choices():
    # two CTAs per SM: one wave of 296 CTAs for the batch-1 64K layer, one of
    # 288 at batch 4 over 128K, seven for the batch-32 cache of 32K
    assert oracle.choose_num_splits_ref(1, 8, 65536, 148) == 37
    assert oracle.choose_num_splits_ref(4, 8, 131072, 148) == 9
    assert oracle.choose_num_splits_ref(32, 8, 32768, 148) == 8
    # short batch-1 histories: one 64-token tile per split where one wave
    # holds them (the fastest calls of the sweeps at 512 .. 2048 tokens)
    assert [oracle.choose_num_splits_ref(1, 8, L, 148) for L in (512, 1024, 2048, 4096, 8192)] == \
        [8, 16, 32, 32, 32]


def test_required_bytes_config_flash_decoding_64k():
    # 64K tokens x 8 kv heads x 128 dims x 2 (K,V) x 2 B + q + O + LSE
    b = oracle.required_bytes_ref(2, 2, 1, 64, 8, 128, [65536])
    assert b == 65536 * 8 * 128 * 2 * 2 + 64 * 128 * 2 + 64 * 128 * 4 + 64 * 4
    assert b == 268484864
