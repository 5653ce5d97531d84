"""Seeded synthetic workloads for decode attention.

This module only draws random inputs and lays them out; it holds none of the
attention arithmetic, so the CUDA library and the CPU oracle can both be fed
from it.  All values are N(0, 1) draws from ``torch.Generator`` objects:

* the bulk tensors (q, then k, then v; then the bifurcated decode k, v) come
  from one generator seeded with ``seed`` on the device they are built on
  (CPU draws for small cases, the device's own generator for the large ones,
  so multi-GiB caches are not pushed through host memory);
* the small integer extras (ragged ``seqlens``, the peaked key positions)
  come from a CPU generator seeded with ``seed + 1``, so they are identical
  whatever device holds the bulk tensors.

bf16 tensors are float32 draws rounded to nearest-even by ``Tensor.to``.

Workload shapes follow the pages' workloads: a CodeLlama-34B-shaped attention
layer at batch 1 (64 query heads, 8 kv heads, head dim 128) for the
Flash-Decoding sweep over 512..64K tokens, a ragged batch, single-context
batch sampling with MQA for bifurcated attention, and a long-context case
with a peaked softmax.
"""

from __future__ import annotations

import math
from dataclasses import dataclass, field
from typing import Optional

import torch

_CHUNK_ELEMS = 1 << 28  # draw at most 256 Mi float32 values at a time


def _randn(shape, dtype, gen, device):
    """N(0,1) float32 draws rounded to ``dtype``, drawn in row chunks so a
    multi-GiB bf16 tensor never needs its float32 image in one piece."""
    out = torch.empty(shape, dtype=dtype, device=device)
    flat = out.view(shape[0], -1)
    row = flat.shape[1]
    rows_per = max(1, _CHUNK_ELEMS // max(1, row))
    for r0 in range(0, shape[0], rows_per):
        r1 = min(shape[0], r0 + rows_per)
        x = torch.randn((r1 - r0, row), generator=gen, dtype=torch.float32, device=device)
        flat[r0:r1].copy_(x.to(dtype))
    return out


def _gen(seed, device):
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


@dataclass
class DecodeCase:
    """One decode-attention call: q [B,Hq,D], k/v cache [B,Lcap,Hkv,D],
    seqlens [B] int32 (CPU) or None for "every sequence is Lcap long"."""
    name: str
    q: torch.Tensor
    k: torch.Tensor
    v: torch.Tensor
    seqlens: Optional[torch.Tensor]
    scale: float
    num_splits: int = 0
    meta: dict = field(default_factory=dict)

    @property
    def lens(self):
        B, Lcap = self.k.shape[0], self.k.shape[1]
        if self.seqlens is None:
            return [Lcap] * B
        return [int(x) for x in self.seqlens.tolist()]


@dataclass
class BifurcatedCase:
    """Single-context batch sampling: q [n,Hq,D], shared context k/v
    [Lc,Hkv,D], per-sample decode k/v [n,Ld,Hkv,D], dec_lens [n] int32 (CPU)
    or None for "all Ld"."""
    name: str
    q: torch.Tensor
    k_ctx: torch.Tensor
    v_ctx: torch.Tensor
    k_dec: torch.Tensor
    v_dec: torch.Tensor
    dec_lens: Optional[torch.Tensor]
    scale: float
    meta: dict = field(default_factory=dict)

    @property
    def lens(self):
        n, Ld = self.k_dec.shape[0], self.k_dec.shape[1]
        if self.dec_lens is None:
            return [Ld] * n
        return [int(x) for x in self.dec_lens.tolist()]


@dataclass
class QuantCase:
    """Decode over an 8-bit cache: q [B,Hq,D]; k/v codes [B,Lcap,Hkv,D]
    (torch.int8, or torch.float8_e4m3fn for kind "e4m3"); k_scale, v_scale
    [Hkv] float32 (dequantised K = k_scale[g] * code); seqlens as DecodeCase."""
    name: str
    q: torch.Tensor
    k: torch.Tensor
    v: torch.Tensor
    k_scale: torch.Tensor
    v_scale: torch.Tensor
    seqlens: Optional[torch.Tensor]
    scale: float
    kind: str
    meta: dict = field(default_factory=dict)

    @property
    def lens(self):
        B, Lcap = self.k.shape[0], self.k.shape[1]
        if self.seqlens is None:
            return [Lcap] * B
        return [int(x) for x in self.seqlens.tolist()]


@dataclass
class MultiCase:
    """Several new query positions per sequence (speculative verification):
    q [B,Tq,Hq,D]; k/v cache [B,Lcap,Hkv,D] holding the history including the
    Tq new tokens; seqlens [B] int32 (CPU) or None for "all Lcap"."""
    name: str
    q: torch.Tensor
    k: torch.Tensor
    v: torch.Tensor
    seqlens: Optional[torch.Tensor]
    scale: float
    meta: dict = field(default_factory=dict)

    @property
    def lens(self):
        B, Lcap = self.k.shape[0], self.k.shape[1]
        if self.seqlens is None:
            return [Lcap] * B
        return [int(x) for x in self.seqlens.tolist()]


def multi_token_case(batch, tq, hq, hkv, d, lcap, dtype=torch.bfloat16, seed=0, seqlens=None,
                     ragged=None, q_dtype=None, device="cpu", scale=None, name="multi"):
    """Multi-token decode workload: like decode_case with Tq query positions
    per sequence (q drawn first, [B, Tq, Hq, D])."""
    q_dtype = dtype if q_dtype is None else q_dtype
    g = _gen(seed, device)
    q = _randn((batch, tq, hq, d), q_dtype, g, device)
    k = _randn((batch, lcap, hkv, d), dtype, g, device)
    v = _randn((batch, lcap, hkv, d), dtype, g, device)
    extra = _gen(seed + 1, "cpu")
    lens_t = None
    if ragged is not None:
        lo, hi = ragged
        lens_t = torch.randint(lo, hi + 1, (batch,), generator=extra, dtype=torch.int64).to(torch.int32)
    elif seqlens is not None:
        lens_t = torch.tensor(list(seqlens), dtype=torch.int32)
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    return MultiCase(name=name, q=q, k=k, v=v, seqlens=lens_t, scale=scale, meta={"seed": seed})


def _int8_codes(shape, sigma, gen, device):
    """Integer codes drawn from a normal of standard deviation ``sigma``,
    rounded and clipped to [-127, 127] (a symmetric 8-bit code range), in
    row chunks like _randn."""
    out = torch.empty(shape, dtype=torch.int8, device=device)
    flat = out.view(shape[0], -1)
    row = flat.shape[1]
    rows_per = max(1, _CHUNK_ELEMS // max(1, row))
    for r0 in range(0, shape[0], rows_per):
        r1 = min(shape[0], r0 + rows_per)
        x = torch.randn((r1 - r0, row), generator=gen, dtype=torch.float32, device=device)
        flat[r0:r1].copy_(torch.round(x * sigma).clamp_(-127, 127).to(torch.int8))
    return out


def quant_case(batch, hq, hkv, d, lcap, kind="int8", seed=0, seqlens=None, ragged=None,
               q_dtype=torch.bfloat16, device="cpu", scale=None, name="quant"):
    """Decode workload over an 8-bit cache.

    kind "int8": codes ~ round(N(0, 32^2)) clipped to [-127, 127], scales
    uniform in [0.5, 1.5] / 32 per kv head (dequantised values ~ N(0, 1)).
    kind "e4m3": N(0, 1) draws rounded to e4m3 by ``Tensor.to``, scales
    uniform in [0.5, 1.5] per kv head.  Scales come from the CPU generator
    seeded with ``seed + 1`` (after the ragged lengths)."""
    if kind not in ("int8", "e4m3"):
        raise ValueError(f"unknown 8-bit kind {kind!r}")
    g = _gen(seed, device)
    q = _randn((batch, hq, d), q_dtype, g, device)
    shape = (batch, lcap, hkv, d)
    if kind == "int8":
        k = _int8_codes(shape, 32.0, g, device)
        v = _int8_codes(shape, 32.0, g, device)
        base = 1.0 / 32.0
    else:
        k = _randn(shape, torch.float8_e4m3fn, g, device)
        v = _randn(shape, torch.float8_e4m3fn, g, device)
        base = 1.0
    extra = _gen(seed + 1, "cpu")
    lens_t = None
    if ragged is not None:
        lo, hi = ragged
        lens_t = torch.randint(lo, hi + 1, (batch,), generator=extra, dtype=torch.int64).to(torch.int32)
    elif seqlens is not None:
        lens_t = torch.tensor(list(seqlens), dtype=torch.int32)
    k_scale = ((0.5 + torch.rand(hkv, generator=extra, dtype=torch.float32)) * base).to(device)
    v_scale = ((0.5 + torch.rand(hkv, generator=extra, dtype=torch.float32)) * base).to(device)
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    return QuantCase(name=name, q=q, k=k, v=v, k_scale=k_scale, v_scale=v_scale, seqlens=lens_t,
                     scale=scale, kind=kind, meta={"seed": seed})


def decode_case(batch, hq, hkv, d, lcap, dtype=torch.bfloat16, seed=0,
                seqlens=None, ragged=None, peaked_frac=0.0, peak_factor=8.0,
                q_dtype=None, device="cpu", scale=None, name="decode"):
    """Generic decode workload.

    ``seqlens``: explicit list of lengths, or None.  ``ragged=(lo, hi)``
    draws each length uniformly from [lo, hi] (inclusive).  ``peaked_frac``
    multiplies the keys at a seeded fraction of each sequence's positions
    (all kv heads and dims of that position) by ``peak_factor``.
    """
    q_dtype = dtype if q_dtype is None else q_dtype
    g = _gen(seed, device)
    q = _randn((batch, hq, d), q_dtype, g, device)
    k = _randn((batch, lcap, hkv, d), dtype, g, device)
    v = _randn((batch, lcap, hkv, d), dtype, g, device)
    extra = _gen(seed + 1, "cpu")
    lens_t = None
    if ragged is not None:
        lo, hi = ragged
        lens_t = torch.randint(lo, hi + 1, (batch,), generator=extra, dtype=torch.int64)
        lens_t = lens_t.to(torch.int32)
    elif seqlens is not None:
        lens_t = torch.tensor(list(seqlens), dtype=torch.int32)
    peaks = None
    if peaked_frac > 0:
        npk = max(1, int(round(peaked_frac * lcap)))
        peaks = []
        for b in range(batch):
            pos = torch.randperm(lcap, generator=extra)[:npk].sort().values
            peaks.append(pos)
            idx = pos.to(device)
            k[b, idx] = k[b, idx] * peak_factor   # x8 is exact in bf16 / fp32
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    return DecodeCase(name=name, q=q, k=k, v=v, seqlens=lens_t, scale=scale,
                      meta={"peaks": peaks, "seed": seed})


# ---------------------------------------------------------------- named workloads

def tiny_mha(seed=0, device="cpu"):
    """Batch 1, one query token, MHA with 4 heads, head dim 64, 256 cached
    tokens, fp32 q/k/v, scale 1/sqrt(64).  Run with num_splits 1 and 4."""
    return decode_case(1, 4, 4, 64, 256, dtype=torch.float32, seed=seed,
                       device=device, name="tiny_mha_fp32_L256")


def flash_decoding_b1(L, seed=0, device="cpu"):
    """Batch 1, CodeLlama-34B-shaped layer: 64 query heads, 8 kv heads
    (GQA group 8), head dim 128, bf16 q/k/v, L cached tokens."""
    return decode_case(1, 64, 8, 128, L, dtype=torch.bfloat16, seed=seed,
                       device=device, name=f"b1_h64_kv8_d128_bf16_L{L}")


def ragged_batch(seed=0, device="cpu", batch=32, lcap=32768, lo=1024, hi=32768):
    """Batch 32, 32 query heads, 8 kv heads, head dim 128, bf16 padded cache
    [32, 32768, 8, 128]; lengths uniform in [1024, 32768]."""
    return decode_case(batch, 32, 8, 128, lcap, dtype=torch.bfloat16, seed=seed,
                       ragged=(lo, hi), device=device,
                       name=f"ragged_b{batch}_h32_kv8_d128_bf16_cap{lcap}")


def long_context_peaked(seed=0, device="cpu", batch=4, L=131072):
    """Batch 4, 131072 cached tokens, 32 query heads, 8 kv heads, head dim
    128, bf16; keys at a seeded 1% of positions scaled by 8 (peaked
    softmax)."""
    return decode_case(batch, 32, 8, 128, L, dtype=torch.bfloat16, seed=seed,
                       peaked_frac=0.01, device=device,
                       name=f"long_b{batch}_h32_kv8_d128_bf16_L{L}_peaked")


def bifurcated_case(n, hq, hkv, d, lc, ld, dtype=torch.bfloat16, seed=0,
                    dec_lens=None, ragged_dec=None, device="cpu", scale=None,
                    name="bifurcated"):
    """Single-context batch sampling workload (one shared context, n
    samples each with its own decode cache)."""
    g = _gen(seed, device)
    q = _randn((n, hq, d), dtype, g, device)
    k_ctx = _randn((lc, hkv, d), dtype, g, device)
    v_ctx = _randn((lc, hkv, d), dtype, g, device)
    k_dec = _randn((n, ld, hkv, d), dtype, g, device)
    v_dec = _randn((n, ld, hkv, d), dtype, g, device)
    extra = _gen(seed + 1, "cpu")
    lens_t = None
    if ragged_dec is not None:
        lo, hi = ragged_dec
        lens_t = torch.randint(lo, hi + 1, (n,), generator=extra, dtype=torch.int64).to(torch.int32)
    elif dec_lens is not None:
        lens_t = torch.tensor(list(dec_lens), dtype=torch.int32)
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    return BifurcatedCase(name=name, q=q, k_ctx=k_ctx, v_ctx=v_ctx, k_dec=k_dec,
                          v_dec=v_dec, dec_lens=lens_t, scale=scale, meta={"seed": seed})


def bifurcated_mqa(seed=0, device="cpu"):
    """MQA single-context sampling: shared context of 8192 tokens, n = 64
    samples each with 256 decode tokens, 32 query heads, 1 kv head, head dim
    128, bf16."""
    return bifurcated_case(64, 32, 1, 128, 8192, 256, seed=seed, device=device,
                           name="bifurcated_mqa_n64_h32_kv1_d128_ctx8192_dec256")


def replicate_context(case: BifurcatedCase):
    """The replicated-context comparison input: every sample gets its own
    copy of the context followed by its decode tokens, as one padded cache
    [n, Lc + Ld, Hkv, D], with seqlens = Lc + dec_len.  Pure data movement."""
    n, ld, hkv, d = case.k_dec.shape
    lc = case.k_ctx.shape[0]
    k = torch.empty((n, lc + ld, hkv, d), dtype=case.k_dec.dtype, device=case.k_dec.device)
    v = torch.empty_like(k)
    k[:, :lc] = case.k_ctx.unsqueeze(0)
    v[:, :lc] = case.v_ctx.unsqueeze(0)
    k[:, lc:] = case.k_dec
    v[:, lc:] = case.v_dec
    lens = torch.tensor([lc + x for x in case.lens], dtype=torch.int32)
    return DecodeCase(name=case.name + "_replicated", q=case.q, k=k, v=v,
                      seqlens=lens, scale=case.scale)


@dataclass
class PagedCase:
    """Decode attention over a paged cache: q [B,Hq,D], k/v pages
    [num_pages, page_size, Hkv, D], block_table [B, max_pages] int32 (CPU),
    seqlens [B] int32 (CPU) or None."""
    name: str
    q: torch.Tensor
    k_pages: torch.Tensor
    v_pages: torch.Tensor
    block_table: torch.Tensor
    seqlens: Optional[torch.Tensor]
    page_size: int
    scale: float
    meta: dict = field(default_factory=dict)

    @property
    def lens(self):
        B, mp = self.block_table.shape
        if self.seqlens is None:
            return [mp * self.page_size] * B
        return [int(x) for x in self.seqlens.tolist()]


def paged_case(batch, hq, hkv, d, page_size, max_pages, num_pages=None, dtype=torch.bfloat16,
               seed=0, seqlens=None, ragged=None, shared_prefix_pages=0, device="cpu",
               scale=None, name="paged"):
    """Paged workload: N(0,1) pages; each sequence's block table is a slice
    of one seeded permutation of the pages (sequences own distinct pages),
    except that the first ``shared_prefix_pages`` entries of every row
    point at sequence 0's first pages (a shared prefix)."""
    if num_pages is None:
        num_pages = batch * max_pages
    g = _gen(seed, device)
    q = _randn((batch, hq, d), dtype, g, device)
    k_pages = _randn((num_pages, page_size, hkv, d), dtype, g, device)
    v_pages = _randn((num_pages, page_size, hkv, d), dtype, g, device)
    extra = _gen(seed + 1, "cpu")
    perm = torch.randperm(num_pages, generator=extra)
    need = batch * max_pages
    if need > num_pages:
        raise ValueError("num_pages must cover batch * max_pages")
    bt = perm[:need].reshape(batch, max_pages).to(torch.int32)
    if shared_prefix_pages:
        bt[:, :shared_prefix_pages] = bt[0, :shared_prefix_pages]
    lens_t = None
    cap = max_pages * page_size
    if ragged is not None:
        lo, hi = ragged
        lens_t = torch.randint(lo, hi + 1, (batch,), generator=extra, dtype=torch.int64).to(torch.int32)
    elif seqlens is not None:
        lens_t = torch.tensor(list(seqlens), dtype=torch.int32)
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    return PagedCase(name=name, q=q, k_pages=k_pages, v_pages=v_pages, block_table=bt,
                     seqlens=lens_t, page_size=page_size, scale=scale,
                     meta={"seed": seed, "capacity": cap})


def paged_flash_decoding_b1(L=65536, page_size=64, seed=0, device="cpu"):
    """The batch-1 CodeLlama-34B-shaped layer (64 query heads, 8 kv heads,
    head dim 128, bf16) with its L-token history in pages of page_size
    tokens scattered by a seeded permutation."""
    return paged_case(1, 64, 8, 128, page_size, L // page_size, dtype=torch.bfloat16, seed=seed,
                      device=device, name=f"paged_b1_h64_kv8_d128_bf16_L{L}_p{page_size}")


def quant_flash_decoding_b1(L=65536, kind="int8", seed=0, device="cpu"):
    """The batch-1 CodeLlama-34B-shaped layer (64 query heads, 8 kv heads,
    head dim 128) over an 8-bit cache of L tokens."""
    return quant_case(1, 64, 8, 128, L, kind=kind, seed=seed, device=device,
                      name=f"b1_h64_kv8_d128_{kind}_L{L}")


def speculative_b1(L=65536, tq=4, seed=0, device="cpu"):
    """The batch-1 CodeLlama-34B-shaped layer (64 query heads, 8 kv heads,
    head dim 128, bf16) verifying tq new tokens against an L-token cache."""
    return multi_token_case(1, tq, 64, 8, 128, L, seed=seed, device=device,
                            name=f"verify{tq}_b1_h64_kv8_d128_bf16_L{L}")
