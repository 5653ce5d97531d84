"""Pin checks for the oracle, written as functions of the implementation under
test so that the same checks run against the real oracle (must pass) and
against oracles with a planted mistake (must fail, tests/test_oracle_mutations.py).

Every check compares against something other than the oracle itself: a
hand-derived worked example, a closed form, a brute-force loop oracle, or an
invariant the pages state.
"""

from __future__ import annotations

import json
import math
import os

import numpy as np

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "worked_examples.json")


def _val(x):
    if isinstance(x, str):
        if x == "-inf":
            return -math.inf
        if x.startswith("ln(") and x.endswith(")"):
            return math.log(float(x[3:-1]))
        raise ValueError(x)
    return float(x)


def _arr(nested):
    if isinstance(nested, list):
        return np.array([_arr(x) for x in nested], dtype=np.float64)
    return _val(nested)


def load_golden():
    with open(GOLDEN) as f:
        return json.load(f)


def _close(a, b, tol=1e-12):
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    if a.shape != b.shape:
        return False
    same_inf = (np.isinf(a) & np.isinf(b) & (np.sign(a) == np.sign(b)))
    fin = ~same_inf
    if np.any(np.isinf(a[fin])) or np.any(np.isinf(b[fin])):
        return False
    return bool(np.all(np.abs(a[fin] - b[fin]) <= tol * (1 + np.abs(b[fin]))))


def golden_decode_ok(decode_fn):
    for case in load_golden()["decode"]:
        O, L = decode_fn(_arr(case["q"]), _arr(case["k"]), _arr(case["v"]),
                         case["seqlens"], case["scale"])
        if not (_close(O, _arr(case["O"])) and _close(L, _arr(case["LSE"]))):
            return False
    return True


def golden_combine_ok(combine_fn):
    for case in load_golden()["combine"]:
        O, L = combine_fn(_arr(case["o_part"]), _arr(case["lse_part"]))
        if not (_close(O, _arr(case["O"])) and _close(L, _arr(case["LSE"]))):
            return False
    return True


def golden_bifurcated_ok(bif_fn):
    for case in load_golden()["bifurcated"]:
        O, L = bif_fn(_arr(case["q"]), _arr(case["k_ctx"]), _arr(case["v_ctx"]),
                      _arr(case["k_dec"]), _arr(case["v_dec"]), case["dec_lens"],
                      case["scale"])
        if not (_close(O, _arr(case["O"])) and _close(L, _arr(case["LSE"]))):
            return False
    return True


def closed_forms_ok(decode_fn, seed=0):
    """Single key -> its value and LSE = its score; identical keys -> mean of V
    and LSE = s + ln L; zero query -> mean of V and LSE = ln L."""
    rng = np.random.default_rng(seed)
    D, G, Hkv = 8, 3, 2
    Hq = G * Hkv
    q = rng.standard_normal((1, Hq, D))
    scale = 0.37
    # single key
    k = rng.standard_normal((1, 1, Hkv, D))
    v = rng.standard_normal((1, 1, Hkv, D))
    O, L = decode_fn(q, k, v, None, scale)
    for h in range(Hq):
        g = h // G
        if not _close(O[0, h], v[0, 0, g], 1e-12):
            return False
        if not _close(L[0, h], scale * float(q[0, h] @ k[0, 0, g]), 1e-12):
            return False
    # identical keys
    n = 7
    k1 = rng.standard_normal((1, 1, Hkv, D))
    k = np.repeat(k1, n, axis=1)
    v = rng.standard_normal((1, n, Hkv, D))
    O, L = decode_fn(q, k, v, None, scale)
    for h in range(Hq):
        g = h // G
        if not _close(O[0, h], v[0, :, g].mean(axis=0), 1e-12):
            return False
        if not _close(L[0, h], scale * float(q[0, h] @ k1[0, 0, g]) + math.log(n), 1e-12):
            return False
    # zero query
    k = rng.standard_normal((1, n, Hkv, D))
    O, L = decode_fn(np.zeros_like(q), k, v, None, scale)
    for h in range(Hq):
        g = h // G
        if not _close(O[0, h], v[0, :, g].mean(axis=0), 1e-12):
            return False
        if not _close(L[0, h], math.log(n), 1e-12):
            return False
    return True


def bruteforce_ok(decode_fn, brute_fn, trials=12, seed=1):
    """Vectorised oracle == pure-Python fsum oracle on tiny random shapes
    (GQA groups, ragged and empty lengths)."""
    rng = np.random.default_rng(seed)
    for t in range(trials):
        B = int(rng.integers(1, 3))
        Hkv = int(rng.integers(1, 3))
        G = int(rng.integers(1, 4))
        D = int(rng.integers(1, 9))
        Lcap = int(rng.integers(1, 17))
        q = rng.standard_normal((B, G * Hkv, D))
        k = rng.standard_normal((B, Lcap, Hkv, D))
        v = rng.standard_normal((B, Lcap, Hkv, D))
        seqlens = [int(rng.integers(0, Lcap + 1)) for _ in range(B)]
        if t % 3 == 0:
            seqlens = None
        scale = float(rng.uniform(0.1, 1.5))
        O, L = decode_fn(q, k, v, seqlens, scale)
        Ob, Lb = brute_fn(q.tolist(), k.tolist(), v.tolist(), seqlens, scale)
        if not (_close(O, np.array(Ob), 1e-12) and _close(L, np.array(Lb), 1e-12)):
            return False
    return True


def split_combine_ok(partials_fn, combine_fn, decode_fn, seed=2):
    """Combining the partials of any split count equals unsplit attention."""
    rng = np.random.default_rng(seed)
    B, Hkv, G, D, Lcap = 3, 2, 2, 5, 200
    q = rng.standard_normal((B, G * Hkv, D))
    k = rng.standard_normal((B, Lcap, Hkv, D))
    v = rng.standard_normal((B, Lcap, Hkv, D))
    seqlens = [200, 1, 137]
    O, L = decode_fn(q, k, v, seqlens, 0.6)
    for ns in [1, 2, 3, 4, 5, 6, 7, 8, 17, 200]:
        Op, Lp = partials_fn(q, k, v, seqlens, 0.6, ns)
        Oc, Lc = combine_fn(Op, Lp)
        if not (_close(Oc, O, 1e-12) and _close(Lc, L, 1e-12)):
            return False
    return True


def bifurcated_concat_ok(bif_fn, decode_fn, seed=3):
    """Bifurcated attention == plain attention over concat(context, decode)."""
    rng = np.random.default_rng(seed)
    n, Hkv, G, D, Lc, Ld = 4, 2, 3, 6, 11, 5
    q = rng.standard_normal((n, G * Hkv, D))
    kc = rng.standard_normal((Lc, Hkv, D))
    vc = rng.standard_normal((Lc, Hkv, D))
    kd = rng.standard_normal((n, Ld, Hkv, D))
    vd = rng.standard_normal((n, Ld, Hkv, D))
    lens = [5, 0, 3, 1]
    O, L = bif_fn(q, kc, vc, kd, vd, lens, 0.4)
    kcat = np.concatenate([np.repeat(kc[None], n, 0), kd], axis=1)
    vcat = np.concatenate([np.repeat(vc[None], n, 0), vd], axis=1)
    Or, Lr = decode_fn(q, kcat, vcat, [Lc + x for x in lens], 0.4)
    return _close(O, Or, 1e-12) and _close(L, Lr, 1e-12)
