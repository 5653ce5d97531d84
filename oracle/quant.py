"""fp64 oracle for decode attention over an 8-bit key/value cache.

TEST INFRASTRUCTURE ONLY (see the package docstring).

Source: the memory-bound decoding explainer ("If you have ever watched an LLM
generate a long response...", gyaansetu.com, Kannada edition), section on
fighting the memory wall, paragraph on quantisation: values normally held as
16-bit floats are stored as 8-bit (or 4-bit) numbers, which cuts the bytes
crossing the memory bus by half or more, while keeping enough precision.
The page applies this to weights; decode attention streams the KV cache, so
the library applies the same storage step there.  Readings that the page
leaves open (listed with the library's design notes): the codes are signed
8-bit integers or 8-bit e4m3 floats, and each key/value head has one fp32
scale for K and one for V, so the cached value is

    K[b, j, g, :] = k_scale[g] * code_K[b, j, g, :]     (V likewise).

Attention is then the ordinary definition (decode_attention_ref) on these
dequantised values, computed exactly in float64.
"""

from __future__ import annotations

import numpy as np

from .attention import decode_attention_ref

KINDS = ("int8", "e4m3")


def e4m3_to_f64(codes) -> np.ndarray:
    """Value of each 8-bit e4m3 code (uint8 bit patterns), from the format:
    bit 7 sign s, bits 6..3 exponent E (bias 7), bits 2..0 mantissa M;
      E = 0:          (-1)^s * (M / 8) * 2^-6          (zero and subnormals)
      E = 1..15:      (-1)^s * (1 + M / 8) * 2^(E - 7)
      E = 15, M = 7:  NaN (the format has no infinities; largest finite 448).
    """
    c = np.asarray(codes).astype(np.uint8).astype(np.int64)
    sign = np.where((c >> 7) & 1, -1.0, 1.0)
    E = (c >> 3) & 0xF
    M = (c & 0x7).astype(np.float64)
    mag = np.where(E == 0, (M / 8.0) * 2.0 ** -6, (1.0 + M / 8.0) * np.exp2(E.astype(np.float64) - 7.0))
    out = sign * mag
    return np.where((E == 15) & (c & 0x7 == 7), np.nan, out)


def int8_to_f64(codes) -> np.ndarray:
    """Signed 8-bit integer codes as float64 (exact)."""
    return np.asarray(codes).astype(np.int8).astype(np.float64)


def dequantize_kv_ref(codes, scale, kind: str) -> np.ndarray:
    """codes [..., Hkv, D] -> float64 values scale[g] * value(code).

    ``codes``: int8 codes (kind "int8") or uint8 e4m3 bit patterns (kind
    "e4m3"); ``scale`` [Hkv]."""
    if kind == "int8":
        vals = int8_to_f64(codes)
    elif kind == "e4m3":
        vals = e4m3_to_f64(codes)
    else:
        raise ValueError(f"unknown 8-bit kind {kind!r}")
    sc = np.asarray(scale, np.float64).reshape(-1)
    if vals.shape[-2] != sc.shape[0]:
        raise ValueError(f"{sc.shape[0]} scales for {vals.shape[-2]} kv heads")
    return vals * sc[:, None]


def quant_decode_attention_ref(q, k_codes, v_codes, k_scale, v_scale, kind: str, seqlens, scale):
    """Decode attention over an 8-bit cache: decode_attention_ref on the
    dequantised K and V.  Returns (O [B, Hq, D], LSE [B, Hq]) in float64.
    Only the first len_b tokens of each sequence are dequantised (codes past
    a sequence's length, even NaN ones, never reach the result)."""
    kq = np.asarray(k_codes)
    vq = np.asarray(v_codes)
    B, Lcap = kq.shape[0], kq.shape[1]
    lens = [Lcap] * B if seqlens is None else [int(x) for x in np.asarray(seqlens).reshape(-1)]
    n = max(lens) if lens else 0
    if n > Lcap or min(lens, default=0) < 0:
        raise ValueError("seqlens outside [0, Lcap]")
    k = np.zeros(kq.shape, np.float64)
    v = np.zeros(vq.shape, np.float64)
    for b in range(B):
        k[b, :lens[b]] = dequantize_kv_ref(kq[b, :lens[b]], k_scale, kind)
        v[b, :lens[b]] = dequantize_kv_ref(vq[b, :lens[b]], v_scale, kind)
    return decode_attention_ref(q, k, v, lens, scale)
