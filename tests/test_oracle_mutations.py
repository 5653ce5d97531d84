"""Planted-mistake checks: each test swaps a plausible error into the oracle
(on the CPU, via monkeypatch) and asserts that at least one pin catches it.
A pin set that let one of these through would not pin the oracle."""

import numpy as np

import oracle
from oracle import attention as oa

import _pins


def _all_decode_pins(fn):
    return (_pins.golden_decode_ok(fn) and _pins.closed_forms_ok(fn)
            and _pins.bruteforce_ok(fn, oracle.attention_bruteforce))


def test_real_oracle_passes_every_pin():
    assert _all_decode_pins(oracle.decode_attention_ref)
    assert _pins.golden_combine_ok(oracle.lse_combine_ref)
    assert _pins.golden_bifurcated_ok(oracle.bifurcated_attention_ref)
    assert _pins.split_combine_ok(oracle.split_partials_ref, oracle.lse_combine_ref,
                                  oracle.decode_attention_ref)
    assert _pins.bifurcated_concat_ok(oracle.bifurcated_attention_ref,
                                      oracle.decode_attention_ref)


def _attend_variant(mistake):
    def attend(qg, kg, vg, scale):
        G, D = qg.shape
        n = kg.shape[0]
        if n == 0:
            return np.zeros((G, D)), np.full(G, -np.inf)
        sc = 1.0 if mistake == "drop_scale" else scale
        s = sc * (qg @ kg.T)
        m = s.max(axis=1)
        e = np.exp(s - m[:, None])
        l = e.sum(axis=1)
        if mistake == "no_normalise":
            o = e @ vg
        elif mistake == "transposed_v":
            o = (e @ vg[::-1]) / l[:, None]
        else:
            o = (e @ vg) / l[:, None]
        lse = np.log(l) if mistake == "lse_without_max" else m + np.log(l)
        if mistake == "log2_lse":
            lse = (m + np.log(l)) / np.log(2.0)
        return o, lse
    return attend


def test_planted_attend_mistakes_are_caught(monkeypatch):
    for mistake in ["drop_scale", "no_normalise", "transposed_v", "lse_without_max",
                    "log2_lse"]:
        monkeypatch.setattr(oa, "_attend", _attend_variant(mistake))
        assert not _all_decode_pins(oa.decode_attention_ref), mistake
    monkeypatch.undo()
    assert _all_decode_pins(oa.decode_attention_ref)


def test_planted_head_map_mistake_is_caught():
    def wrong_map(q, k, v, seqlens, scale):
        q = np.asarray(q, np.float64)
        k = np.asarray(k, np.float64)
        v = np.asarray(v, np.float64)
        B, Hq, D = q.shape
        Lcap, Hkv = k.shape[1], k.shape[2]
        lens = [Lcap] * B if seqlens is None else list(seqlens)
        O = np.zeros((B, Hq, D))
        L = np.full((B, Hq), -np.inf)
        for b in range(B):
            for h in range(Hq):
                g = h % Hkv                                   # planted: interleaved map
                o, l = oa._attend(q[b, h:h + 1], k[b, :lens[b], g], v[b, :lens[b], g], scale)
                O[b, h], L[b, h] = o[0], l[0]
        return O, L
    assert not _all_decode_pins(wrong_map)


def test_planted_length_off_by_one_is_caught():
    def off_by_one(q, k, v, seqlens, scale):
        if seqlens is not None:
            Lcap = np.asarray(k).shape[1]
            seqlens = [min(Lcap, int(x) + 1) for x in seqlens]
        return oracle.decode_attention_ref(q, k, v, seqlens, scale)
    assert not _all_decode_pins(off_by_one)


def test_planted_combine_mistakes_are_caught():
    def no_shift(o, lse):
        w = np.exp(np.asarray(lse))                       # planted: weights not / sum
        return (w[..., None] * o).sum(-2), np.log(w.sum(-1))
    assert not _pins.golden_combine_ok(no_shift)

    def plain_mean(o, lse):
        return np.asarray(o).mean(-2), np.asarray(lse).max(-1)
    assert not _pins.golden_combine_ok(plain_mean)


def test_planted_split_bounds_mistake_is_caught(monkeypatch):
    real = oa.split_bounds_ref

    def overlap(length, ns, i):
        lo, hi = real(length, ns, i)
        return max(0, lo - 1), hi                         # planted: one-token overlap
    monkeypatch.setattr(oa, "split_bounds_ref", overlap)
    assert not _pins.split_combine_ok(oa.split_partials_ref, oa.lse_combine_ref,
                                      oa.decode_attention_ref)


def test_planted_bifurcated_mistakes_are_caught():
    def ctx_only(q, kc, vc, kd, vd, lens, scale):
        n = np.asarray(q).shape[0]
        return oracle.bifurcated_attention_ref(q, kc, vc, kd, vd, [0] * n, scale)
    assert not _pins.golden_bifurcated_ok(ctx_only)
    assert not _pins.bifurcated_concat_ok(ctx_only, oracle.decode_attention_ref)

    def separate_softmax(q, kc, vc, kd, vd, lens, scale):
        # planted: normalise the two parts separately and average them
        n = np.asarray(q).shape[0]
        Oc, Lc = oracle.decode_attention_ref(q, np.repeat(np.asarray(kc)[None], n, 0),
                                             np.repeat(np.asarray(vc)[None], n, 0), None, scale)
        Od, Ld = oracle.decode_attention_ref(q, kd, vd, lens, scale)
        Od = np.where(np.isfinite(Ld)[..., None], Od, Oc)
        return 0.5 * (Oc + Od), np.logaddexp(Lc, Ld)
    assert not _pins.golden_bifurcated_ok(separate_softmax)
