"""Pins for the paged-cache oracle (CPU only).

The paged reference reads keys and values through a block table.  It is
checked against a token-at-a-time brute force (math.fsum, no max shift),
against the contiguous reference on a cache whose pages are laid out in
order (identity table), and a planted off-by-one in the page lookup must
fail the brute-force comparison.
"""

import numpy as np
import pytest

import oracle
from oracle import attention as oa


def _case(rng, B, Hq, Hkv, D, ps, max_pages, num_pages, lens):
    q = rng.standard_normal((B, Hq, D))
    kp = rng.standard_normal((num_pages, ps, Hkv, D))
    vp = rng.standard_normal((num_pages, ps, Hkv, D))
    bt = np.stack([rng.permutation(num_pages)[:max_pages] for _ in range(B)]).astype(np.int64)
    return q, kp, vp, bt, lens


@pytest.mark.parametrize("ps,lens", [(2, [5, 0, 8]), (3, [9, 4, 1]), (4, [12, 7, 3])])
def test_paged_ref_matches_bruteforce(ps, lens):
    rng = np.random.default_rng(ps)
    q, kp, vp, bt, lens = _case(rng, 3, 4, 2, 3, ps, 12 // ps + 1, 16, lens)
    O, L = oracle.paged_decode_attention_ref(q, kp, vp, bt, lens, ps, 0.7)
    Ob, Lb = oracle.paged_attention_bruteforce(q.tolist(), kp.tolist(), vp.tolist(), bt.tolist(),
                                               lens, ps, 0.7)
    np.testing.assert_allclose(O, np.array(Ob), rtol=1e-12, atol=1e-13)
    Lb = np.array(Lb)
    assert np.array_equal(np.isneginf(L), np.isneginf(Lb))
    fin = ~np.isneginf(Lb)
    np.testing.assert_allclose(L[fin], Lb[fin], rtol=1e-12, atol=1e-13)


def test_identity_table_equals_contiguous_cache():
    rng = np.random.default_rng(5)
    B, Hq, Hkv, D, ps, mp = 2, 6, 3, 8, 4, 5
    k = rng.standard_normal((B, mp * ps, Hkv, D))
    v = rng.standard_normal((B, mp * ps, Hkv, D))
    q = rng.standard_normal((B, Hq, D))
    kp = k.reshape(B * mp, ps, Hkv, D)               # sequence b owns pages b*mp .. b*mp+mp-1
    vp = v.reshape(B * mp, ps, Hkv, D)
    bt = np.arange(B * mp).reshape(B, mp)
    lens = [17, 20]
    O, L = oracle.paged_decode_attention_ref(q, kp, vp, bt, lens, ps, 0.3)
    Oc, Lc = oracle.decode_attention_ref(q, k, v, lens, 0.3)
    np.testing.assert_allclose(O, Oc, rtol=1e-13, atol=1e-14)
    np.testing.assert_allclose(L, Lc, rtol=1e-13, atol=1e-14)


def test_page_ids_out_of_range_are_rejected():
    rng = np.random.default_rng(6)
    q, kp, vp, bt, _ = _case(rng, 1, 2, 1, 4, 2, 3, 4, [5])
    bt[0, 1] = 4
    with pytest.raises(ValueError):
        oracle.paged_decode_attention_ref(q, kp, vp, bt, [5], 2, 1.0)


def test_planted_page_offset_mistake_is_caught(monkeypatch):
    """A gather that reads row (j + 1) % page_size instead of j % page_size
    must disagree with the brute force."""
    rng = np.random.default_rng(7)
    q, kp, vp, bt, lens = _case(rng, 2, 2, 1, 4, 3, 4, 8, [10, 7])

    def bad_gather(pages, block_table, page_size, length, b):
        pages = np.asarray(pages, np.float64)
        out = np.zeros((length,) + pages.shape[2:])
        for j in range(length):
            out[j] = pages[int(block_table[b, j // page_size]), (j + 1) % page_size]
        return out

    monkeypatch.setattr(oa, "paged_gather_ref", bad_gather)
    O, _ = oa.paged_decode_attention_ref(q, kp, vp, bt, lens, 3, 0.5)
    Ob, _ = oracle.paged_attention_bruteforce(q.tolist(), kp.tolist(), vp.tolist(), bt.tolist(),
                                              lens, 3, 0.5)
    assert not np.allclose(O, np.array(Ob), atol=1e-6)
