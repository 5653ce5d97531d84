"""fp64 CPU oracle for exact single-query decode attention.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path may import, call or
execute this package: only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` use it.  It
shares no code with the CUDA library (``decode_attention_20_b300``) and
imports nothing from it.

Sources (web pages, cited by title and section):

* "What is Flash-Decoding and when does it speed up LLMs?" (slavadubrov.com,
  Spanish edition), section "Why decoding needs different scheduling":
  split the cached history, each unit emits a partial result and a
  log-sum-exp value, a reduction recovers full-history attention.
* Summary of "Bifurcated Attention for Single-Context Large-Batch Sampling"
  (linnk.ai), sections "Tiivistelmä" (abstract) and "Tilastot" (statistics):
  attention during incremental decoding is split into two GEMMs, one over
  the prefill (context) KV and one over the decode KV; the result is exact.
* "How does Flash Attention reduce memory traffic during local inference?"
  (zimaspace.com, Italian edition), sections on tiling and online softmax:
  the family computes exact attention.

* "If you have ever watched an LLM generate a long response..." (gyaansetu.com,
  Kannada edition), section on fighting the memory wall: paged KV storage
  behind an indirection table, and 8-bit storage to halve the bytes moved
  (``quant.py``).

Every function works in float64 on the exact values of its inputs.  bf16
inputs are decoded from their raw 16-bit patterns by :func:`bf16_bits_to_f64`
(no torch conversion involved).

Parity pins (see ``tests/test_oracle_pins.py``): brute force on tiny shapes,
hand-derived worked examples (``tests/golden/``), closed forms (single key,
identical keys, zero query), split/combine == unsplit, bifurcated ==
concatenated, permutation invariance, SciPy/PyTorch library special cases.
Every function below is pinned; none is "parity unpinned".
"""

from .attention import (  # noqa: F401
    bf16_bits_to_f64,
    decode_attention_ref,
    attention_weights_ref,
    split_bounds_ref,
    choose_num_splits_ref,
    split_partials_ref,
    lse_combine_ref,
    bifurcated_attention_ref,
    paged_gather_ref,
    paged_decode_attention_ref,
    causal_lengths_ref,
    multi_token_decode_ref,
    required_bytes_ref,
    SPLIT_ALIGN,
    MAX_SPLITS,
    MIN_CHUNK,
    SPLIT_OVERHEAD_TOKENS,
)
from .bruteforce import attention_bruteforce, paged_attention_bruteforce, multi_token_bruteforce  # noqa: F401
from .quant import (  # noqa: F401
    e4m3_to_f64,
    int8_to_f64,
    dequantize_kv_ref,
    quant_decode_attention_ref,
)
