"""Pins of the 8-bit-cache oracle (oracle/quant.py) on the CPU: the e4m3
decoding against an independent implementation and the format's landmark
values, brute force on tiny caches, and closed forms."""

import numpy as np

import oracle
from oracle import quant as oq

import _pins


def test_e4m3_decoding_matches_format():
    assert _pins.e4m3_table_ok(oracle.e4m3_to_f64)


def test_int8_codes_are_their_integers():
    codes = np.arange(-128, 128).astype(np.int8)
    assert np.array_equal(oracle.int8_to_f64(codes), np.arange(-128, 128, dtype=np.float64))


def test_dequantize_uses_each_heads_scale():
    codes = np.arange(-15, 15).astype(np.int8).reshape(2, 3, 5)        # [L, Hkv, D]
    scale = np.array([0.5, 2.0, -0.25], np.float32)
    out = oracle.dequantize_kv_ref(codes, scale, "int8")
    for j in range(2):
        for g in range(3):
            for d in range(5):
                assert out[j, g, d] == float(codes[j, g, d]) * float(scale[g])


def test_quant_oracle_against_bruteforce():
    assert _pins.quant_bruteforce_ok(oracle.quant_decode_attention_ref, oracle.attention_bruteforce)


def test_quant_oracle_closed_forms():
    assert _pins.quant_closed_forms_ok(oracle.quant_decode_attention_ref)


def test_quant_oracle_equals_plain_oracle_on_dequantised_values():
    rng = np.random.default_rng(3)
    q = rng.standard_normal((2, 8, 16))
    kc = rng.integers(-127, 128, (2, 40, 2, 16)).astype(np.int8)
    vc = rng.integers(-127, 128, (2, 40, 2, 16)).astype(np.int8)
    ks = np.array([0.02, 0.04], np.float32)
    vs = np.array([0.03, 0.01], np.float32)
    O, L = oracle.quant_decode_attention_ref(q, kc, vc, ks, vs, "int8", [40, 17], 0.25)
    k = kc.astype(np.float64) * ks.astype(np.float64)[:, None]
    v = vc.astype(np.float64) * vs.astype(np.float64)[:, None]
    O2, L2 = oracle.decode_attention_ref(q, k, v, [40, 17], 0.25)
    assert np.allclose(O, O2, rtol=0, atol=1e-13) and np.allclose(L, L2, rtol=0, atol=1e-13)


# ---------------------------------------------------------- planted mistakes

def _all_quant_pins():
    return (_pins.e4m3_table_ok(oq.e4m3_to_f64)
            and _pins.quant_bruteforce_ok(oq.quant_decode_attention_ref, oracle.attention_bruteforce)
            and _pins.quant_closed_forms_ok(oq.quant_decode_attention_ref))


def test_planted_quant_mistakes_are_caught(monkeypatch):
    real_e4m3 = oq.e4m3_to_f64
    real_deq = oq.dequantize_kv_ref

    def e4m3_bias8(codes):
        return real_e4m3(codes) / 2.0

    def e4m3_sub_wrong(codes):
        c = np.asarray(codes).astype(np.uint8)
        out = real_e4m3(c)
        sub = ((c >> 3) & 0xF) == 0
        return np.where(sub, out * 0.5, out)

    def deq_no_scale(codes, scale, kind):
        return real_deq(codes, np.ones_like(np.asarray(scale)), kind)

    def deq_unsigned_int8(codes, scale, kind):
        if kind == "int8":
            vals = np.asarray(codes).astype(np.uint8).astype(np.float64)
            return vals * np.asarray(scale, np.float64)[:, None]
        return real_deq(codes, scale, kind)

    def deq_scale_reversed(codes, scale, kind):
        return real_deq(codes, np.asarray(scale)[::-1].copy(), kind)

    for name, fn in [("e4m3_to_f64", e4m3_bias8), ("e4m3_to_f64", e4m3_sub_wrong),
                     ("dequantize_kv_ref", deq_no_scale),
                     ("dequantize_kv_ref", deq_unsigned_int8),
                     ("dequantize_kv_ref", deq_scale_reversed)]:
        monkeypatch.setattr(oq, name, fn)
        assert not _all_quant_pins(), fn.__name__
        monkeypatch.undo()
    assert _all_quant_pins()
