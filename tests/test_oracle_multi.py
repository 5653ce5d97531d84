"""Pins of the multi-token (speculative verification) decode oracle on the
CPU: hand-derived worked examples, a loop oracle with an explicit causal
mask, and the single-query special cases; plus planted mistakes."""

import numpy as np

import oracle
from oracle import attention as oa

import _pins


def test_multi_golden_examples():
    assert _pins.golden_multi_ok(oracle.multi_token_decode_ref)


def test_multi_against_bruteforce():
    assert _pins.multi_bruteforce_ok(oracle.multi_token_decode_ref, oracle.multi_token_bruteforce)


def test_multi_last_query_is_plain_decode():
    assert _pins.multi_last_query_is_plain_decode_ok(oracle.multi_token_decode_ref,
                                                     oracle.decode_attention_ref)


def test_causal_lengths():
    assert oracle.causal_lengths_ref(10, 3) == [8, 9, 10]
    assert oracle.causal_lengths_ref(1, 3) == [0, 0, 1]
    assert oracle.causal_lengths_ref(0, 2) == [0, 0]


def _all_multi_pins(fn):
    return (_pins.golden_multi_ok(fn)
            and _pins.multi_bruteforce_ok(fn, oracle.multi_token_bruteforce)
            and _pins.multi_last_query_is_plain_decode_ok(fn, oracle.decode_attention_ref))


def test_planted_multi_mistakes_are_caught(monkeypatch):
    real = oa.causal_lengths_ref
    mistakes = {
        "sees_own_position_excluded": lambda n, tq: [max(0, n - tq + t) for t in range(tq)],
        "not_causal": lambda n, tq: [n] * tq,
        "reversed_order": lambda n, tq: real(n, tq)[::-1],
    }
    for name, fn in mistakes.items():
        monkeypatch.setattr(oa, "causal_lengths_ref", fn)
        assert not _all_multi_pins(oa.multi_token_decode_ref), name
        monkeypatch.undo()
    assert _all_multi_pins(oa.multi_token_decode_ref)
