"""Second, loop-based oracle for tiny shapes.

TEST INFRASTRUCTURE ONLY (see the package docstring).

Pure Python: every dot product and sum is a ``math.fsum`` (exactly rounded
sum), and the softmax is written with no maximum subtraction,
p_j = e^(s_j) / sum_k e^(s_k), so it checks the vectorised oracle's max-shift
arithmetic instead of repeating it.  Valid only while every |s_j| is small
enough for e^(s_j) to stay finite (the tests keep |s| < 50).
"""

from __future__ import annotations

import math


def attention_bruteforce(q, k, v, seqlens, scale):
    """Exact single-query attention by definition.

    q: nested lists [B][Hq][D]; k, v: [B][Lcap][Hkv][D]; seqlens: list or None.
    Query head h reads kv head h // (Hq // Hkv).  Returns (O, LSE) as nested
    lists; an empty history gives O = 0 and LSE = -inf.
    """
    B = len(q)
    Hq = len(q[0])
    D = len(q[0][0])
    Lcap = len(k[0])
    Hkv = len(k[0][0])
    G = Hq // Hkv
    O = [[[0.0] * D for _ in range(Hq)] for _ in range(B)]
    LSE = [[-math.inf] * Hq for _ in range(B)]
    for b in range(B):
        n = Lcap if seqlens is None else int(seqlens[b])
        for h in range(Hq):
            g = h // G
            if n == 0:
                continue
            s = [scale * math.fsum(q[b][h][d] * k[b][j][g][d] for d in range(D))
                 for j in range(n)]
            e = [math.exp(x) for x in s]
            z = math.fsum(e)
            LSE[b][h] = math.log(z)
            for d in range(D):
                O[b][h][d] = math.fsum(e[j] * v[b][j][g][d] for j in range(n)) / z
    return O, LSE


def paged_attention_bruteforce(q, k_pages, v_pages, block_table, seqlens, page_size, scale):
    """Exact single-query attention over a paged cache, by definition: every
    key and value is fetched one token at a time through the block table
    (page block_table[b][j // page_size], row j % page_size).  Nested lists
    in, nested lists out, as attention_bruteforce."""
    B = len(q)
    Hq = len(q[0])
    D = len(q[0][0])
    Hkv = len(k_pages[0][0])
    G = Hq // Hkv
    O = [[[0.0] * D for _ in range(Hq)] for _ in range(B)]
    LSE = [[-math.inf] * Hq for _ in range(B)]
    for b in range(B):
        n = len(block_table[b]) * page_size if seqlens is None else int(seqlens[b])
        for h in range(Hq):
            g = h // G
            if n == 0:
                continue
            kk = [k_pages[block_table[b][j // page_size]][j % page_size][g] for j in range(n)]
            vv = [v_pages[block_table[b][j // page_size]][j % page_size][g] for j in range(n)]
            s = [scale * math.fsum(q[b][h][d] * kk[j][d] for d in range(D)) for j in range(n)]
            e = [math.exp(x) for x in s]
            z = math.fsum(e)
            LSE[b][h] = math.log(z)
            for d in range(D):
                O[b][h][d] = math.fsum(e[j] * vv[j][d] for j in range(n)) / z
    return O, LSE


def multi_token_bruteforce(q, k, v, seqlens, scale):
    """Multi-token decode by definition: q nested [B][Tq][Hq][D]; query t of
    sequence b attends over the keys at positions j <= len_b - Tq + t (a
    causal mask written out per key); k, v [B][Lcap][Hkv][D].  Returns
    (O [B][Tq][Hq][D], LSE [B][Tq][Hq])."""
    B = len(q)
    Tq = len(q[0])
    Lcap = len(k[0])
    O, LSE = [], []
    for b in range(B):
        n = Lcap if seqlens is None else int(seqlens[b])
        Ob, Lb = [], []
        for t in range(Tq):
            pos = n - Tq + t                       # this query's own position
            keys = [j for j in range(n) if j <= pos]
            kk = [[k[b][j] for j in keys]]
            vv = [[v[b][j] for j in keys]]
            o, l = attention_bruteforce([q[b][t]], kk, vv, [len(keys)], scale) if keys else (None, None)
            if o is None:
                Hq, D = len(q[b][t]), len(q[b][t][0])
                Ob.append([[0.0] * D for _ in range(Hq)])
                Lb.append([-math.inf] * Hq)
            else:
                Ob.append(o[0])
                Lb.append(l[0])
        O.append(Ob)
        LSE.append(Lb)
    return O, LSE
