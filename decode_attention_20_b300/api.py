"""Python binding of the C ABI (argument marshalling only).

Each function turns torch CUDA tensors into fd_tensor descriptors (pointer,
dtype, shape, strides), passes the current torch CUDA stream, and calls the
library entry point of the same name.  Every step of the computation runs in
the library's CUDA kernels; tensors that are not on a CUDA device are
rejected.
"""

from __future__ import annotations

import ctypes
import math
from typing import Optional

import torch

from . import _lib
from ._lib import FdError, FdTensor, check, lib  # noqa: F401

_DT = {torch.float32: _lib.FD_F32, torch.bfloat16: _lib.FD_BF16, torch.int32: _lib.FD_I32,
       torch.int8: _lib.FD_I8, torch.float8_e4m3fn: _lib.FD_E4M3}


# Descriptors by value: (pointer, dtype, shape, strides) -> fd_tensor.  A
# descriptor holds nothing but those values, so a cached one is the one that
# would be built; a decode loop that reuses its buffers builds each once.
_DESC_CACHE: dict = {}
_DESC_CACHE_MAX = 512


def _desc(t: Optional[torch.Tensor], name: str):
    if t is None:
        return None
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor (the library has no CPU path)")
    key = (t.data_ptr(), t.dtype, t.shape, t.stride())
    d = _DESC_CACHE.get(key)
    if d is not None:
        return d
    if t.dtype not in _DT:
        raise TypeError(f"{name}: unsupported dtype {t.dtype}")
    if t.dim() > 4:
        raise ValueError(f"{name}: at most 4 dims")
    d = _lib.raw_descriptor(key[0], _DT[t.dtype], list(key[2]), list(key[3]))
    if len(_DESC_CACHE) >= _DESC_CACHE_MAX:
        _DESC_CACHE.clear()
    _DESC_CACHE[key] = d
    return d


def _ref(d):
    return ctypes.byref(d) if d is not None else None


_raw_stream = getattr(torch._C, "_cuda_getCurrentRawStream", None)


def _stream(stream):
    if stream is None:
        if _raw_stream is not None:
            # The current stream's handle without building a Stream object.
            return ctypes.c_void_p(_raw_stream(torch.cuda.current_device()))
        return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    if isinstance(stream, torch.cuda.Stream):
        return ctypes.c_void_p(stream.cuda_stream)
    return ctypes.c_void_p(int(stream))


def decode_attention(q, k_cache, v_cache, seqlens=None, num_splits=0, scale=None,
                     out=None, lse=None, return_lse=True, stream=None):
    """Split-KV decode attention (fd_decode_attention).

    q [B, Hq, D]; k_cache, v_cache [B, Lcap, Hkv, D] (bf16 or fp32);
    seqlens [B] int32 CUDA tensor or None; returns (out [B,Hq,D] fp32,
    lse [B,Hq] fp32 or None)."""
    B, Hq, D = q.shape
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    if out is None:
        out = torch.empty((B, Hq, D), dtype=torch.float32, device=q.device)
    if lse is None and return_lse:
        lse = torch.empty((B, Hq), dtype=torch.float32, device=q.device)
    dq, dk, dv, ds = _desc(q, "q"), _desc(k_cache, "k_cache"), _desc(v_cache, "v_cache"), _desc(seqlens, "seqlens")
    do, dl = _desc(out, "out"), _desc(lse, "lse")
    check(lib().fd_decode_attention(_ref(dq), _ref(dk), _ref(dv), _ref(ds), int(num_splits),
                                    float(scale), _ref(do), _ref(dl), _stream(stream)))
    return out, lse


def decode_attention_multi(q, k_cache, v_cache, seqlens=None, num_splits=0, scale=None,
                           out=None, lse=None, return_lse=True, stream=None):
    """Multi-token decode attention (fd_decode_attention_multi): q [B, Tq,
    Hq, D]; the cache holds the history including the Tq new tokens; query t
    sees keys j < len_b - Tq + t + 1.  Returns (out [B, Tq, Hq, D] fp32,
    lse [B, Tq, Hq] fp32 or None)."""
    B, Tq, Hq, D = q.shape
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    if out is None:
        out = torch.empty((B, Tq, Hq, D), dtype=torch.float32, device=q.device)
    if lse is None and return_lse:
        lse = torch.empty((B, Tq, Hq), dtype=torch.float32, device=q.device)
    dq, dk, dv, ds = _desc(q, "q"), _desc(k_cache, "k_cache"), _desc(v_cache, "v_cache"), _desc(seqlens, "seqlens")
    do, dl = _desc(out, "out"), _desc(lse, "lse")
    check(lib().fd_decode_attention_multi(_ref(dq), _ref(dk), _ref(dv), _ref(ds), int(num_splits),
                                          float(scale), _ref(do), _ref(dl), _stream(stream)))
    return out, lse


def decode_attention_quant(q, k_cache, v_cache, k_scale, v_scale, seqlens=None, num_splits=0,
                           scale=None, out=None, lse=None, return_lse=True, stream=None):
    """Split-KV decode attention over an 8-bit cache (fd_decode_attention_quant).

    k_cache, v_cache [B, Lcap, Hkv, D] torch.int8 or torch.float8_e4m3fn
    codes; k_scale, v_scale [Hkv] fp32 CUDA tensors (K = k_scale[g] * codes,
    V likewise); the rest as decode_attention."""
    B, Hq, D = q.shape
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    if out is None:
        out = torch.empty((B, Hq, D), dtype=torch.float32, device=q.device)
    if lse is None and return_lse:
        lse = torch.empty((B, Hq), dtype=torch.float32, device=q.device)
    dq, dk, dv = _desc(q, "q"), _desc(k_cache, "k_cache"), _desc(v_cache, "v_cache")
    dks, dvs, ds = _desc(k_scale, "k_scale"), _desc(v_scale, "v_scale"), _desc(seqlens, "seqlens")
    do, dl = _desc(out, "out"), _desc(lse, "lse")
    check(lib().fd_decode_attention_quant(_ref(dq), _ref(dk), _ref(dv), _ref(dks), _ref(dvs),
                                          _ref(ds), int(num_splits), float(scale), _ref(do),
                                          _ref(dl), _stream(stream)))
    return out, lse


def decode_attention_paged(q, k_pages, v_pages, block_table, seqlens=None, num_splits=0,
                           scale=None, out=None, lse=None, return_lse=True, stream=None):
    """Split-KV decode attention over a paged cache
    (fd_decode_attention_paged): k_pages, v_pages [num_pages, page_size,
    Hkv, D]; block_table [B, max_pages] int32 CUDA tensor; seqlens [B] int32
    or None.  Returns (out [B,Hq,D] fp32, lse [B,Hq] fp32 or None)."""
    B, Hq, D = q.shape
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    if out is None:
        out = torch.empty((B, Hq, D), dtype=torch.float32, device=q.device)
    if lse is None and return_lse:
        lse = torch.empty((B, Hq), dtype=torch.float32, device=q.device)
    a = [_desc(q, "q"), _desc(k_pages, "k_pages"), _desc(v_pages, "v_pages"),
         _desc(block_table, "block_table"), _desc(seqlens, "seqlens")]
    do, dl = _desc(out, "out"), _desc(lse, "lse")
    check(lib().fd_decode_attention_paged(*[_ref(x) for x in a], int(num_splits), float(scale),
                                          _ref(do), _ref(dl), _stream(stream)))
    return out, lse


def decode_attention_partials(q, k_cache, v_cache, num_splits, seqlens=None, scale=None,
                              part_o=None, part_lse=None, stream=None):
    """The split stage alone (fd_decode_attention_partials): returns
    (part_o [B,Hq,ns,D], part_lse [B,Hq,ns]), fp32."""
    B, Hq, D = q.shape
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    if part_o is None:
        part_o = torch.empty((B, Hq, num_splits, D), dtype=torch.float32, device=q.device)
    if part_lse is None:
        part_lse = torch.empty((B, Hq, num_splits), dtype=torch.float32, device=q.device)
    args = [_desc(q, "q"), _desc(k_cache, "k_cache"), _desc(v_cache, "v_cache"), _desc(seqlens, "seqlens")]
    do, dl = _desc(part_o, "part_o"), _desc(part_lse, "part_lse")
    check(lib().fd_decode_attention_partials(*[_ref(a) for a in args], int(num_splits), float(scale),
                                             _ref(do), _ref(dl), _stream(stream)))
    return part_o, part_lse


def lse_combine(part_o, part_lse, out=None, lse=None, stream=None):
    """Log-sum-exp reduction (fd_lse_combine): part_o [R,S,D], part_lse [R,S]
    -> (out [R,D], lse [R])."""
    R, S, D = part_o.shape
    if out is None:
        out = torch.empty((R, D), dtype=torch.float32, device=part_o.device)
    if lse is None:
        lse = torch.empty((R,), dtype=torch.float32, device=part_o.device)
    a = [_desc(part_o, "part_o"), _desc(part_lse, "part_lse"), _desc(out, "out"), _desc(lse, "lse")]
    check(lib().fd_lse_combine(*[_ref(x) for x in a], _stream(stream)))
    return out, lse


def bifurcated_attention(q, k_ctx, v_ctx, k_dec, v_dec, dec_lens=None, scale=None, out=None,
                         lse=None, ctx_splits=0, return_lse=False, stream=None):
    """Bifurcated attention (fd_bifurcated_attention[_lse]): q [n,Hq,D],
    shared k_ctx/v_ctx [Lc,Hkv,D], per-sample k_dec/v_dec [n,Ld,Hkv,D],
    dec_lens [n] int32 or None.  Returns out [n,Hq,D] (and lse [n,Hq] when
    return_lse)."""
    n, Hq, D = q.shape
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    if out is None:
        out = torch.empty((n, Hq, D), dtype=torch.float32, device=q.device)
    if lse is None and return_lse:
        lse = torch.empty((n, Hq), dtype=torch.float32, device=q.device)
    a = [_desc(q, "q"), _desc(k_ctx, "k_ctx"), _desc(v_ctx, "v_ctx"), _desc(k_dec, "k_dec"),
         _desc(v_dec, "v_dec"), _desc(dec_lens, "dec_lens")]
    do, dl = _desc(out, "out"), _desc(lse, "lse")
    if lse is None and ctx_splits == 0:
        check(lib().fd_bifurcated_attention(*[_ref(x) for x in a], float(scale), _ref(do),
                                            _stream(stream)))
    else:
        check(lib().fd_bifurcated_attention_lse(*[_ref(x) for x in a], float(scale), int(ctx_splits),
                                                _ref(do), _ref(dl), _stream(stream)))
    return (out, lse) if return_lse else out


def choose_num_splits(batch, kv_heads, max_len, num_sms):
    return int(lib().fd_choose_num_splits(batch, kv_heads, max_len, num_sms))


def split_bounds(length, ns, i):
    b = ctypes.c_int64()
    e = ctypes.c_int64()
    check(lib().fd_split_bounds(length, ns, i, ctypes.byref(b), ctypes.byref(e)))
    return b.value, e.value


def workspace_bytes(batch, q_heads, head_dim, num_splits):
    return int(lib().fd_workspace_bytes(batch, q_heads, head_dim, num_splits))


def check_device_error(stream=None):
    """Synchronises the stream; raises FdError if the device clamped a
    length (FD_ERR_DEVICE_BOUNDS) or a bounded wait timed out."""
    check(lib().fd_check_device_error(_stream(stream)))


def profile_enable(on=True):
    check(lib().fd_profile_enable(1 if on else 0))


def profile_read(kind):
    """(launches, total_ms) of one kernel kind since the last enable."""
    n = ctypes.c_int64()
    ms = ctypes.c_double()
    check(lib().fd_profile_read(int(kind), ctypes.byref(n), ctypes.byref(ms)))
    return n.value, ms.value


def version():
    return lib().fd_version().decode()
