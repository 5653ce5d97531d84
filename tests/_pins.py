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


# ------------------------------------------------------------ 8-bit caches

_E4M3_LANDMARKS = {
    0x00: 0.0, 0x01: 2.0 ** -9, 0x07: 7 / 8 * 2.0 ** -6, 0x08: 2.0 ** -6,
    0x38: 1.0, 0xB8: -1.0, 0x77: 240.0, 0x7E: 448.0, 0xFE: -448.0,
}


def e4m3_table_ok(e4m3_fn):
    """Every e4m3 code against PyTorch's float8_e4m3fn decoding (an
    independent implementation of the same format), plus landmark values of
    the format: 1.0, the largest finite 448, the smallest normal 2^-6 and
    subnormal 2^-9, and exactly two NaN codes (0x7F, 0xFF)."""
    import torch
    codes = np.arange(256, dtype=np.uint8)
    ours = np.asarray(e4m3_fn(codes), np.float64)
    lib = torch.from_numpy(codes.copy()).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    if not np.array_equal(np.isnan(ours), np.isnan(lib)):
        return False
    if sorted(np.flatnonzero(np.isnan(ours)).tolist()) != [0x7F, 0xFF]:
        return False
    fin = ~np.isnan(lib)
    if not np.array_equal(ours[fin], lib[fin]):
        return False
    return all(ours[c] == v for c, v in _E4M3_LANDMARKS.items())


def _code_value(kind, c):
    """Value of one code, by hand: the integer itself, or PyTorch's e4m3."""
    if kind == "int8":
        return float(int(c))
    import torch
    t = torch.tensor([int(c)], dtype=torch.uint8).view(torch.float8_e4m3fn)
    return float(t.to(torch.float64).item())


def _small_codes(rng, kind, shape):
    if kind == "int8":
        return rng.integers(-127, 128, shape).astype(np.int8)
    # e4m3 codes with |value| < 4 (exponent field <= 8), either sign
    mag = rng.integers(0, 0x48, shape)
    sign = rng.integers(0, 2, shape) << 7
    return (mag | sign).astype(np.uint8)


def quant_bruteforce_ok(quant_fn, bruteforce_fn):
    """Tiny int8 and e4m3 caches with ragged lengths and a distinct scale per
    kv head: the oracle against the loop oracle run on values dequantised by
    hand (code value x the scale of the code's own kv head)."""
    rng = np.random.default_rng(11)
    for kind, ks, vs in (("int8", [0.03, 0.05, 0.021], [0.04, 0.017, 0.033]),
                         ("e4m3", [0.7, 1.3, 0.9], [1.1, 0.6, 1.45])):
        B, Hkv, G, D, L = 2, 3, 2, 6, 5
        q = rng.standard_normal((B, Hkv * G, D))
        kc = _small_codes(rng, kind, (B, L, Hkv, D))
        vc = _small_codes(rng, kind, (B, L, Hkv, D))
        seqlens = [5, 3]
        scale = 0.4
        O, LSE = quant_fn(q, kc, vc, np.array(ks, np.float32), np.array(vs, np.float32), kind,
                          seqlens, scale)
        ksf = [float(np.float32(x)) for x in ks]
        vsf = [float(np.float32(x)) for x in vs]
        kd = [[[[_code_value(kind, kc[b, j, g, d]) * ksf[g] for d in range(D)] for g in range(Hkv)]
               for j in range(L)] for b in range(B)]
        vd = [[[[_code_value(kind, vc[b, j, g, d]) * vsf[g] for d in range(D)] for g in range(Hkv)]
               for j in range(L)] for b in range(B)]
        Ob, Lb = bruteforce_fn(q.tolist(), kd, vd, seqlens, scale)
        if not (_close(O, Ob, 1e-11) and _close(LSE, Lb, 1e-11)):
            return False
    return True


def quant_closed_forms_ok(quant_fn):
    """Closed forms on 8-bit caches:
    - V scale: O is linear in v_scale, LSE does not depend on it;
    - k_scale = 0: every score is 0, so O = mean of the dequantised V and
      LSE = ln len;
    - one cached token: O = v_scale[g] * v_code, LSE = scale * k_scale[g] *
      <q, k_code>;
    - codes past a sequence's length (NaN e4m3 codes included) are unused."""
    rng = np.random.default_rng(5)
    for kind in ("int8", "e4m3"):
        B, Hkv, G, D, L = 1, 2, 2, 4, 7
        q = rng.standard_normal((B, Hkv * G, D))
        kc = _small_codes(rng, kind, (B, L, Hkv, D))
        vc = _small_codes(rng, kind, (B, L, Hkv, D))
        ks = np.array([0.05, 0.08], np.float32) if kind == "int8" else np.array([0.9, 1.2], np.float32)
        vs = np.array([0.03, 0.06], np.float32) if kind == "int8" else np.array([0.5, 1.5], np.float32)
        val = np.vectorize(lambda c: _code_value(kind, c))
        O1, L1 = quant_fn(q, kc, vc, ks, vs, kind, None, 0.5)
        O2, L2 = quant_fn(q, kc, vc, ks, 4.0 * vs, kind, None, 0.5)    # x4: exact in fp32
        if not (_close(O2, 4.0 * O1) and _close(L2, L1)):
            return False
        O0, L0 = quant_fn(q, kc, vc, np.zeros(2, np.float32), vs, kind, [5], 0.5)
        for h in range(Hkv * G):
            g = h // G
            mean = val(vc[0, :5, g]).mean(axis=0) * float(vs[g])
            if not (_close(O0[0, h], mean) and _close(L0[0, h], math.log(5))):
                return False
        Os, Ls = quant_fn(q, kc, vc, ks, vs, kind, [1], 0.5)
        for h in range(Hkv * G):
            g = h // G
            s = 0.5 * float(ks[g]) * float(np.dot(q[0, h], val(kc[0, 0, g])))
            if not (_close(Os[0, h], val(vc[0, 0, g]) * float(vs[g])) and _close(Ls[0, h], s)):
                return False
        if kind == "e4m3":
            kn, vn = kc.copy(), vc.copy()
            kn[0, 4:] = 0x7F
            vn[0, 4:] = 0xFF
            Oa, La = quant_fn(q, kn, vn, ks, vs, kind, [4], 0.5)
            Ob, Lb = quant_fn(q, kc, vc, ks, vs, kind, [4], 0.5)
            if not (np.all(np.isfinite(Oa)) and _close(Oa, Ob) and _close(La, Lb)):
                return False
    return True


# ------------------------------------------------------- multi-token decode

def golden_multi_ok(multi_fn):
    """The hand-derived multi-token examples (tests/golden, "multi")."""
    for case in load_golden()["multi"]:
        O, L = multi_fn(_arr(case["q"]), _arr(case["k"]), _arr(case["v"]), case["seqlens"],
                        case["scale"])
        if not (_close(O, _arr(case["O"])) and _close(L, _arr(case["LSE"]))):
            return False
    return True


def multi_bruteforce_ok(multi_fn, brute_fn, trials=8, seed=3):
    """Vectorised multi-token oracle == the loop oracle with a per-key causal
    mask, on tiny shapes with GQA groups and histories shorter than, equal
    to and longer than the number of new positions."""
    rng = np.random.default_rng(seed)
    for _ in range(trials):
        B, Tq, Hkv, G, D, L = 2, int(rng.integers(1, 5)), 2, int(rng.integers(1, 3)), 4, 6
        q = rng.standard_normal((B, Tq, Hkv * G, D))
        k = rng.standard_normal((B, L, Hkv, D))
        v = rng.standard_normal((B, L, Hkv, D))
        seqlens = [int(rng.integers(0, L + 1)), L]
        O, LSE = multi_fn(q, k, v, seqlens, 0.7)
        Ob, Lb = brute_fn(q.tolist(), k.tolist(), v.tolist(), seqlens, 0.7)
        if not (_close(O, Ob, 1e-11) and _close(LSE, Lb, 1e-11)):
            return False
    return True


def multi_last_query_is_plain_decode_ok(multi_fn, decode_fn, seed=4):
    """The newest query position sees the whole history: its row equals
    single-query decode; with one new position the two definitions agree."""
    rng = np.random.default_rng(seed)
    q = rng.standard_normal((3, 4, 4, 8))
    k = rng.standard_normal((3, 20, 2, 8))
    v = rng.standard_normal((3, 20, 2, 8))
    lens = [20, 7, 2]
    O, L = multi_fn(q, k, v, lens, 0.3)
    O1, L1 = decode_fn(q[:, -1], k, v, lens, 0.3)
    if not (_close(O[:, -1], O1) and _close(L[:, -1], L1)):
        return False
    O2, L2 = multi_fn(q[:, :1], k, v, lens, 0.3)
    O3, L3 = decode_fn(q[:, 0], k, v, lens, 0.3)
    return _close(O2[:, 0], O3) and _close(L2[:, 0], L3)
