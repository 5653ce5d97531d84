"""Vectorised fp64 oracle: exact single-query decode attention, its split /
log-sum-exp-combine decomposition, and bifurcated (context + decode) attention.

TEST INFRASTRUCTURE ONLY (see the package docstring).  Plain NumPy, float64,
no blocking or fusion beyond what each definition states.

Notation (shared by every function here):
  B batch, Hq query heads, Hkv key/value heads, G = Hq // Hkv query heads per
  key/value head, D head dimension, Lcap allocated cache length,
  len_b = seqlens[b] valid cached tokens of sequence b.
  Query head h reads key/value head g(h) = h // G (contiguous groups: the
  bifurcated-attention summary only says MQA/GQA compose with the method;
  contiguous grouping is the plain reading).
"""

from __future__ import annotations

import numpy as np

# Split partition granule (tokens).  A split's chunk is ceil(len / ns) rounded
# up to a multiple of SPLIT_ALIGN; the pages fix no partition, this is the
# reading adopted for the whole library.
SPLIT_ALIGN = 64
# Largest number of splits per (sequence, kv-head).
MAX_SPLITS = 256
# Shortest chunk the split heuristic will create (tokens): one 64-token tile
# of the split kernel (the split-count sweeps on B300 find the fastest call
# at 64-token chunks for histories of 512 to 2048 tokens).
MIN_CHUNK = 64
# Fixed cost of one wave of split CTAs in the heuristic's makespan model, in
# tokens of streaming (start-up latency of the first tiles plus the epilogue).
SPLIT_OVERHEAD_TOKENS = 256


def bf16_bits_to_f64(bits) -> np.ndarray:
    """Decode raw bfloat16 bit patterns (uint16) to float64 exactly.

    bfloat16 is the top 16 bits of an IEEE-754 binary32 value, so placing the
    pattern in the high half of a 32-bit word gives the binary32 value, which
    float64 represents exactly.
    """
    b = np.ascontiguousarray(np.asarray(bits, dtype=np.uint16))
    w = b.astype(np.uint32) << np.uint32(16)
    return w.view(np.float32).astype(np.float64)


def _softmax_stats(s: np.ndarray):
    """Row-wise max m, sum l = sum exp(s - m) and weights exp(s - m) / l.

    ``s`` is [rows, n] with n >= 1.  Definition of softmax with the maximum
    subtracted ("How does Flash Attention reduce memory traffic...", section
    on online softmax: ordinary softmax needs the whole row; the max shift
    only changes rounding).
    """
    m = s.max(axis=1)
    e = np.exp(s - m[:, None])
    l = e.sum(axis=1)
    return m, l, e


def _attend(qg: np.ndarray, kg: np.ndarray, vg: np.ndarray, scale: float):
    """Exact attention of G query rows over n keys (one key/value head).

    qg [G, D], kg [n, D], vg [n, D]  ->  O [G, D], LSE [G] (natural log of the
    sum of exp of the scaled scores).  n == 0 gives O = 0, LSE = -inf.
    """
    G, D = qg.shape
    n = kg.shape[0]
    if n == 0:
        return np.zeros((G, D)), np.full(G, -np.inf)
    s = scale * (qg @ kg.T)                       # [G, n]  scores
    m, l, e = _softmax_stats(s)
    o = (e @ vg) / l[:, None]                     # [G, D]  sum_j p_j v_j
    lse = m + np.log(l)
    return o, lse


def _check_shapes(q, k, v):
    B, Hq, D = q.shape
    Bk, Lcap, Hkv, Dk = k.shape
    if k.shape != v.shape or Bk != B or Dk != D or Hq % Hkv != 0:
        raise ValueError(f"bad shapes q{q.shape} k{k.shape} v{v.shape}")
    return B, Hq, D, Lcap, Hkv, Hq // Hkv


def _lens(seqlens, B, Lcap):
    if seqlens is None:
        return [Lcap] * B
    lens = [int(x) for x in np.asarray(seqlens).reshape(-1)]
    if len(lens) != B:
        raise ValueError("seqlens must have one entry per sequence")
    for x in lens:
        if x < 0 or x > Lcap:
            raise ValueError(f"seqlen {x} outside [0, {Lcap}]")
    return lens


def decode_attention_ref(q, k, v, seqlens, scale):
    """Exact single-query decode attention (the definition the method reaches).

    q [B, Hq, D]; k, v [B, Lcap, Hkv, D]; seqlens [B] or None (= Lcap).
    For each b and query head h, over keys j < len_b of kv head g = h // G:
        s_j = scale * <q[b,h], k[b,j,g]>,  m = max_j s_j,  l = sum_j e^(s_j-m)
        O[b,h] = sum_j e^(s_j-m) / l * v[b,j,g],   LSE[b,h] = m + ln l.
    Returns (O [B, Hq, D], LSE [B, Hq]) in float64.  len_b == 0 gives O = 0
    and LSE = -inf.

    One new query position per active sequence attends over its whole cached
    history ("What is Flash-Decoding...", section "Why decoding needs
    different scheduling"); the result is exact attention ("How does Flash
    Attention reduce memory traffic...", section "Flash Attention splits the
    problem into on-chip working sets").
    """
    q = np.asarray(q, np.float64)
    k = np.asarray(k, np.float64)
    v = np.asarray(v, np.float64)
    B, Hq, D, Lcap, Hkv, G = _check_shapes(q, k, v)
    lens = _lens(seqlens, B, Lcap)
    O = np.zeros((B, Hq, D))
    LSE = np.full((B, Hq), -np.inf)
    for b in range(B):
        n = lens[b]
        for g in range(Hkv):
            hs = slice(g * G, (g + 1) * G)
            O[b, hs], LSE[b, hs] = _attend(q[b, hs], k[b, :n, g], v[b, :n, g], scale)
    return O, LSE


def attention_weights_ref(q, k, seqlens, scale):
    """Softmax weights p[b, h, j] (zero for j >= len_b): the probabilities
    that decode_attention_ref averages V with.  Used by the sum-to-one pin."""
    q = np.asarray(q, np.float64)
    k = np.asarray(k, np.float64)
    B, Hq, D, Lcap, Hkv, G = _check_shapes(q, k, k)
    lens = _lens(seqlens, B, Lcap)
    P = np.zeros((B, Hq, Lcap))
    for b in range(B):
        n = lens[b]
        if n == 0:
            continue
        for g in range(Hkv):
            hs = slice(g * G, (g + 1) * G)
            s = scale * (q[b, hs] @ k[b, :n, g].T)
            _, l, e = _softmax_stats(s)
            P[b, hs, :n] = e / l[:, None]
    return P


def split_bounds_ref(length: int, ns: int, i: int):
    """Token range [begin, end) of split i when a history of ``length`` tokens
    is cut into ns splits.

    chunk = ceil(ceil(length / ns) / SPLIT_ALIGN) * SPLIT_ALIGN;
    begin = min(i * chunk, length); end = min((i + 1) * chunk, length).
    Splits that start at or past ``length`` are empty.  The Flash-Decoding
    page ("Why decoding needs different scheduling") only says the history is
    divided into parts; equal aligned chunks are the reading taken here.
    """
    if ns < 1 or i < 0 or i >= ns or length < 0:
        raise ValueError("bad split arguments")
    per = -(-length // ns)
    chunk = -(-per // SPLIT_ALIGN) * SPLIT_ALIGN
    begin = min(i * chunk, length)
    end = min((i + 1) * chunk, length)
    return begin, end


def choose_num_splits_ref(batch: int, kv_heads: int, max_len: int, num_sms: int) -> int:
    """Split-count heuristic (mirror of the library's host function).

    The Flash-Decoding page ("Why decoding needs different scheduling") gives
    only the direction: a small batch leaves too few independent blocks, so
    split the history; a short history or a large batch makes more splitting
    useless, and more splits are no guaranteed gain.  Reading adopted: a
    makespan model.  With ns splits of a max_len history, one CTA per
    (sequence, kv head, split) and two CTAs per SM at a time,
        chunk  = the split chunk of split_bounds_ref(max_len, ns, .)
        waves  = ceil(batch * kv_heads * nonempty_splits / (2 * num_sms))
        cost   = waves * (chunk + SPLIT_OVERHEAD_TOKENS)
    and the smallest ns in [1, min(MAX_SPLITS, ceil(max_len / MIN_CHUNK))]
    with the lowest cost wins.  SPLIT_OVERHEAD_TOKENS charges each wave the
    fixed start-up and epilogue time of a CTA, in tokens of streaming.
    """
    units = batch * kv_heads
    if units <= 0 or max_len <= 0 or num_sms <= 0:
        return 1
    cap = max(1, min(MAX_SPLITS, -(-max_len // MIN_CHUNK)))
    best_ns, best_cost = 1, None
    for ns in range(1, cap + 1):
        per = -(-max_len // ns)
        chunk = -(-per // SPLIT_ALIGN) * SPLIT_ALIGN
        used = -(-max_len // chunk)
        waves = -(-(units * used) // (2 * num_sms))
        cost = waves * (chunk + SPLIT_OVERHEAD_TOKENS)
        if best_cost is None or cost < best_cost:
            best_ns, best_cost = ns, cost
    return int(best_ns)


def split_partials_ref(q, k, v, seqlens, scale, ns):
    """Per-split partial results: for split i of sequence b, exact attention
    restricted to tokens [begin_i, end_i) (split_bounds_ref).

    Returns (O_part [B, Hq, ns, D], lse_part [B, Hq, ns]); an empty split has
    O = 0 and lse = -inf.  Each unit of work yields its own partial output
    together with a log-sum-exp value ("What is Flash-Decoding...", section
    "Why decoding needs different scheduling").
    """
    q = np.asarray(q, np.float64)
    k = np.asarray(k, np.float64)
    v = np.asarray(v, np.float64)
    B, Hq, D, Lcap, Hkv, G = _check_shapes(q, k, v)
    lens = _lens(seqlens, B, Lcap)
    O = np.zeros((B, Hq, ns, D))
    LSE = np.full((B, Hq, ns), -np.inf)
    for b in range(B):
        for i in range(ns):
            lo, hi = split_bounds_ref(lens[b], ns, i)
            for g in range(Hkv):
                hs = slice(g * G, (g + 1) * G)
                O[b, hs, i], LSE[b, hs, i] = _attend(
                    q[b, hs], k[b, lo:hi, g], v[b, lo:hi, g], scale)
    return O, LSE


def lse_combine_ref(o_part, lse_part):
    """Log-sum-exp reduction of partial results along the split axis (-2 for
    O, -1 for lse):
        LSE = ln sum_i e^(lse_i)   (evaluated as M + ln sum_i e^(lse_i - M),
                                    M = max_i lse_i)
        O   = sum_i e^(lse_i - LSE) * O_i
    All splits empty (every lse_i = -inf) gives O = 0, LSE = -inf.
    The Flash-Decoding page ("Why decoding needs different scheduling") has a
    final reduction merge the partials into exactly the full-history result.
    """
    o_part = np.asarray(o_part, np.float64)
    lse_part = np.asarray(lse_part, np.float64)
    M = lse_part.max(axis=-1)
    finite = np.isfinite(M)
    Ms = np.where(finite, M, 0.0)
    w_un = np.exp(lse_part - Ms[..., None])            # e^(lse_i - M), 0 for empty
    tot = w_un.sum(axis=-1)
    LSE = np.where(finite, Ms + np.log(np.where(finite, tot, 1.0)), -np.inf)
    w = np.where(finite[..., None], w_un / np.where(finite, tot, 1.0)[..., None], 0.0)
    O = (w[..., None] * o_part).sum(axis=-2)
    return O, LSE


def bifurcated_attention_ref(q, k_ctx, v_ctx, k_dec, v_dec, dec_lens, scale):
    """Bifurcated attention for single-context batch sampling.

    q [n, Hq, D]; k_ctx, v_ctx [Lc, Hkv, D] (one context shared by all n
    samples); k_dec, v_dec [n, Ld, Hkv, D]; dec_lens [n] or None (= Ld).
    Sample i attends over concat(context, its own first dec_lens[i] decode
    tokens).  Following the method's two-GEMM split ("Bifurcated Attention
    for Single-Context Large-Batch Sampling" summary, section "Tiivistelmä"):
      GEMM 1: S_ctx = scale * Q_g K_ctx[g]^T with the rows of Q_g being every
              (sample, query head of group g) pair -- the context keys are
              read once for all samples;
      GEMM 2: S_dec = scale * q_i K_dec[i, g]^T per sample;
    then one softmax over [S_ctx | S_dec] and O = P_ctx V_ctx + P_dec V_dec.
    Returns (O [n, Hq, D], LSE [n, Hq]) in float64.
    """
    q = np.asarray(q, np.float64)
    k_ctx = np.asarray(k_ctx, np.float64)
    v_ctx = np.asarray(v_ctx, np.float64)
    k_dec = np.asarray(k_dec, np.float64)
    v_dec = np.asarray(v_dec, np.float64)
    n, Hq, D = q.shape
    Lc, Hkv, Dc = k_ctx.shape
    n2, Ld, Hkv2, Dd = k_dec.shape
    if (n2 != n or Hkv2 != Hkv or Dc != D or Dd != D or Hq % Hkv
            or v_ctx.shape != k_ctx.shape or v_dec.shape != k_dec.shape):
        raise ValueError("bad bifurcated shapes")
    G = Hq // Hkv
    lens = _lens(dec_lens, n, Ld)
    O = np.zeros((n, Hq, D))
    LSE = np.full((n, Hq), -np.inf)
    for g in range(Hkv):
        hs = slice(g * G, (g + 1) * G)
        Qg = q[:, hs, :].reshape(n * G, D)                  # rows = (sample, head)
        S_ctx = (scale * (Qg @ k_ctx[:, g, :].T)).reshape(n, G, Lc)   # GEMM 1
        for i in range(n):
            kd = k_dec[i, :lens[i], g]
            vd = v_dec[i, :lens[i], g]
            S_dec = scale * (q[i, hs] @ kd.T)                # GEMM 2 (per sample)
            s = np.concatenate([S_ctx[i], S_dec], axis=1)    # [G, Lc + len_i]
            if s.shape[1] == 0:
                continue
            m, l, e = _softmax_stats(s)
            o = (e[:, :Lc] @ v_ctx[:, g, :] + e[:, Lc:] @ vd) / l[:, None]
            O[i, hs] = o
            LSE[i, hs] = m + np.log(l)
    return O, LSE


def causal_lengths_ref(length: int, tq: int):
    """Keys visible to each of the tq new query positions of a sequence whose
    cached history (the new positions included, at its end) is ``length``
    tokens long: query t sits at position length - tq + t and sees positions
    0 .. length - tq + t, i.e. max(0, length - tq + t + 1) keys."""
    return [max(0, int(length) - int(tq) + t + 1) for t in range(int(tq))]


def multi_token_decode_ref(q, k, v, seqlens, scale):
    """Decode attention with several new query positions per sequence
    (speculative verification): q [B, Tq, Hq, D]; k, v [B, Lcap, Hkv, D];
    seqlens [B] or None (= Lcap) counts the cached tokens including the Tq
    new ones.  Query t of sequence b is decode_attention_ref over the first
    causal_lengths_ref(len_b, Tq)[t] keys.  Returns (O [B, Tq, Hq, D],
    LSE [B, Tq, Hq]).

    The Flash-Decoding page contrasts prefill, which processes many query
    positions at once, with usual decoding, one new position per sequence
    (section "Why decoding needs different scheduling"); a verification step
    sits in between, and each new position attends causally to the history
    up to itself."""
    q = np.asarray(q, np.float64)
    k = np.asarray(k, np.float64)
    B, Tq, Hq, D = q.shape
    Lcap = k.shape[1]
    lens = _lens(seqlens, B, Lcap)
    O = np.zeros((B, Tq, Hq, D))
    LSE = np.full((B, Tq, Hq), -np.inf)
    for t in range(Tq):
        lt = [causal_lengths_ref(n, Tq)[t] for n in lens]
        O[:, t], LSE[:, t] = decode_attention_ref(q[:, t], k, v, lt, scale)
    return O, LSE


def paged_gather_ref(pages, block_table, page_size: int, length: int, b: int):
    """The first ``length`` cached tokens of sequence b from a paged cache.

    pages [num_pages, page_size, Hkv, D]; block_table [B, max_pages]: token j
    of sequence b is row j % page_size of page block_table[b, j // page_size]
    (the indirection table of paged KV storage in the memory-bound decoding
    explainer, section on the memory wall: fixed-size KV blocks mapped
    through a table).  Returns [length, Hkv, D]."""
    pages = np.asarray(pages, np.float64)
    bt = np.asarray(block_table)
    out = np.zeros((length,) + pages.shape[2:])
    for j in range(length):
        pid = int(bt[b, j // page_size])
        if pid < 0 or pid >= pages.shape[0]:
            raise ValueError(f"page id {pid} outside [0, {pages.shape[0]})")
        out[j] = pages[pid, j % page_size]
    return out


def paged_decode_attention_ref(q, k_pages, v_pages, block_table, seqlens, page_size, scale):
    """Decode attention over a paged KV cache: the same definition as
    decode_attention_ref with each sequence's keys and values read through
    its block table (paged_gather_ref).  seqlens None means every sequence
    fills its max_pages * page_size slots."""
    q = np.asarray(q, np.float64)
    bt = np.asarray(block_table)
    B, Hq, D = q.shape
    Hkv = np.asarray(k_pages).shape[2]
    G = Hq // Hkv
    cap = bt.shape[1] * page_size
    lens = _lens(seqlens, B, cap)
    O = np.zeros((B, Hq, D))
    LSE = np.full((B, Hq), -np.inf)
    for b in range(B):
        kb = paged_gather_ref(k_pages, bt, page_size, lens[b], b)
        vb = paged_gather_ref(v_pages, bt, page_size, lens[b], b)
        for g in range(Hkv):
            hs = slice(g * G, (g + 1) * G)
            O[b, hs], LSE[b, hs] = _attend(q[b, hs], kb[:, g], vb[:, g], scale)
    return O, LSE


def required_bytes_ref(elem_bytes_kv: int, elem_bytes_q: int, batch: int, hq: int,
                       hkv: int, d: int, lens) -> int:
    """Algorithmic bytes of one decode-attention call: K and V over
    [0, len_b) for every (b, kv head), the query read once, O (fp32) and LSE
    (fp32) written once.  Partial-result workspace and seqlens excluded."""
    kv = sum(int(x) for x in lens) * hkv * d * 2 * elem_bytes_kv
    return kv + batch * hq * d * elem_bytes_q + batch * hq * d * 4 + batch * hq * 4

