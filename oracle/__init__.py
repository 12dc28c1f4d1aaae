"""CPU oracle for paged decode attention -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  It never imports the CUDA library's
package and shares no code with it; it is a ctypes wrapper around
``oracle.c`` (plain fp64 C), whose header lists the passages it follows:

* "How does TensorRT-LLM work?", "The paged KV cache" -- block pool, per-request
  block table, decode reads every earlier token;
* "Introduction to TensorRT-LLM", "2. Paged KV Cache" -- fixed-size token
  blocks behind virtual-to-physical block tables;
* "TensorRT-LLM, in depth", "First principles: where the GPU memory goes" --
  the kv_bytes_per_token closed form and the Llama-3-8B geometry;
* "TensorRT-LLM, in depth", "Quantization: fewer bytes per weight and per
  cached token" -- FP8 KV cache.

Storage dtypes are named by strings: ``"f32"``, ``"bf16"``, ``"fp8"`` (OCP
E4M3).  Arrays crossing this boundary are numpy arrays holding the raw storage
bits (float32, uint16 for bf16, uint8 for E4M3); helpers accept torch CPU
tensors and convert them.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional, Tuple

import numpy as np

from . import build as _build

_DT = {"f32": 0, "bf16": 1, "fp8": 2}
_NP = {"f32": np.float32, "bf16": np.uint16, "fp8": np.uint8}
INT32_MAX = 2**31 - 1

_lib = None


def _load():
    global _lib
    if _lib is None:
        path = _build.build()
        lib = ctypes.CDLL(path)
        c = ctypes
        P = c.c_void_p
        lib.or_bf16_to_double.restype = c.c_double
        lib.or_bf16_to_double.argtypes = [c.c_uint16]
        lib.or_float_to_bf16.restype = c.c_uint16
        lib.or_float_to_bf16.argtypes = [c.c_float]
        lib.or_e4m3_to_double.restype = c.c_double
        lib.or_e4m3_to_double.argtypes = [c.c_uint8]
        lib.or_float_to_e4m3.restype = c.c_uint8
        lib.or_float_to_e4m3.argtypes = [c.c_float]
        lib.or_kv_bytes_per_token.restype = c.c_int64
        lib.or_kv_bytes_per_token.argtypes = [c.c_int64] * 4
        lib.or_slot_mapping.restype = c.c_int
        lib.or_slot_mapping.argtypes = [P, c.c_int, c.c_int, P, P, c.c_int, P]
        lib.or_kv_append.restype = c.c_int
        lib.or_kv_append.argtypes = [P, c.c_int, c.c_int, c.c_int, c.c_int, c.c_int, c.c_int,
                                     c.c_int, P, c.c_int, P, c.c_int, c.c_float]
        lib.or_paged_attention.restype = c.c_int
        lib.or_paged_attention.argtypes = [P, c.c_int, P, P, c.c_int, c.c_int, c.c_int, c.c_int,
                                           c.c_int, c.c_int, c.c_int, c.c_float, c.c_float, P,
                                           c.c_int, P, c.c_int, c.c_int, c.c_float, c.c_int,
                                           c.c_int, P, P, c.c_int, P]
        lib.or_paged_attention_mq.restype = c.c_int
        lib.or_paged_attention_mq.argtypes = [P, c.c_int, P, P, c.c_int, c.c_int, c.c_int, c.c_int,
                                              c.c_int, c.c_int, c.c_int, c.c_float, c.c_float, P,
                                              c.c_int, P, c.c_int, c.c_int, c.c_int, c.c_float, P, P,
                                              c.c_int, c.POINTER(c.c_int)]
        lib.or_lse_combine.restype = None
        lib.or_lse_combine.argtypes = [P, P, c.c_int, c.c_int, P, P]
        for name, t_in, t_out in (("or_e4m3_encode_array", P, P), ("or_e4m3_decode_array", P, P),
                                  ("or_bf16_encode_array", P, P), ("or_bf16_decode_array", P, P)):
            fn = getattr(lib, name)
            fn.restype = None
            fn.argtypes = [t_in, c.c_int64, t_out]
        _lib = lib
    return _lib


def _ptr(a: np.ndarray):
    assert a.flags["C_CONTIGUOUS"], "oracle arrays must be C-contiguous"
    return ctypes.c_void_p(a.ctypes.data)


def to_numpy_bits(x, dtype: str) -> np.ndarray:
    """Raw storage bits of a torch CPU tensor / numpy array as a numpy array."""
    try:
        import torch
        if isinstance(x, torch.Tensor):
            x = x.detach().cpu().contiguous()
            if dtype == "bf16":
                return x.view(torch.int16).numpy().view(np.uint16).copy()
            if dtype == "fp8":
                return x.view(torch.uint8).numpy().copy()
            return x.to(torch.float32).numpy().copy()
    except ImportError:  # pragma: no cover
        pass
    return np.ascontiguousarray(np.asarray(x).astype(_NP[dtype], copy=False))


# ------------------------------------------------------------------ formats

def e4m3_encode(x) -> np.ndarray:
    """binary32 -> OCP E4M3 codes (RN-even, saturating to +-448)."""
    x = np.ascontiguousarray(np.asarray(x, dtype=np.float32))
    out = np.empty(x.shape, dtype=np.uint8)
    _load().or_e4m3_encode_array(_ptr(x), x.size, _ptr(out))
    return out


def e4m3_decode(codes) -> np.ndarray:
    codes = np.ascontiguousarray(np.asarray(codes, dtype=np.uint8))
    out = np.empty(codes.shape, dtype=np.float64)
    _load().or_e4m3_decode_array(_ptr(codes), codes.size, _ptr(out))
    return out


def bf16_encode(x) -> np.ndarray:
    x = np.ascontiguousarray(np.asarray(x, dtype=np.float32))
    out = np.empty(x.shape, dtype=np.uint16)
    _load().or_bf16_encode_array(_ptr(x), x.size, _ptr(out))
    return out


def bf16_decode(bits) -> np.ndarray:
    bits = np.ascontiguousarray(np.asarray(bits, dtype=np.uint16))
    out = np.empty(bits.shape, dtype=np.float64)
    _load().or_bf16_decode_array(_ptr(bits), bits.size, _ptr(out))
    return out


def kv_bytes_per_token(layers: int, kv_heads: int, head_dim: int, bytes_per_elem: int) -> int:
    return int(_load().or_kv_bytes_per_token(layers, kv_heads, head_dim, bytes_per_elem))


# --------------------------------------------------------------- pool + ops

class OraclePool:
    """Host copy of a K pool and a V pool, [layers][blocks][kv_heads][bs][D]."""

    def __init__(self, num_layers: int, num_blocks: int, block_size: int, kv_heads: int,
                 head_dim: int, dtype: str, k_scale: float = 1.0, v_scale: float = 1.0,
                 fill: int = 0):
        self.num_layers, self.num_blocks, self.block_size = num_layers, num_blocks, block_size
        self.kv_heads, self.head_dim, self.dtype = kv_heads, head_dim, dtype
        self.k_scale, self.v_scale = float(k_scale), float(v_scale)
        shape = (num_layers, num_blocks, kv_heads, block_size, head_dim)
        nbytes = int(np.prod(shape)) * np.dtype(_NP[dtype]).itemsize
        self.k = np.full(nbytes, fill, dtype=np.uint8).view(_NP[dtype]).reshape(shape)
        self.v = np.full(nbytes, fill, dtype=np.uint8).view(_NP[dtype]).reshape(shape)


def slot_mapping(block_tables, block_size: int, seq_idx, pos) -> np.ndarray:
    bt = np.ascontiguousarray(np.asarray(block_tables, dtype=np.int32))
    si = np.ascontiguousarray(np.asarray(seq_idx, dtype=np.int32))
    ps = np.ascontiguousarray(np.asarray(pos, dtype=np.int32))
    out = np.empty(si.shape[0], dtype=np.int64)
    rc = _load().or_slot_mapping(_ptr(bt), bt.shape[1], block_size, _ptr(si), _ptr(ps),
                                 si.shape[0], _ptr(out))
    if rc != 0:
        raise IndexError("oracle slot_mapping: position outside the block table (rc=%d)" % rc)
    return out


def kv_append(pool: OraclePool, layer: int, k, v, in_dtype: str, slots) -> None:
    """Scatter k, v [T][kv_heads][D] (in_dtype "f32" or "bf16") into the pool."""
    kk = to_numpy_bits(k, in_dtype)
    vv = to_numpy_bits(v, in_dtype)
    sl = np.ascontiguousarray(np.asarray(slots, dtype=np.int64))
    T = sl.shape[0]
    assert kk.size == T * pool.kv_heads * pool.head_dim and vv.size == kk.size
    lib = _load()
    for src, dst, sc in ((kk, pool.k, pool.k_scale), (vv, pool.v, pool.v_scale)):
        rc = lib.or_kv_append(_ptr(dst), _DT[pool.dtype], pool.num_layers, pool.num_blocks,
                              pool.block_size, pool.kv_heads, pool.head_dim, layer, _ptr(src),
                              _DT[in_dtype], _ptr(sl), T, sc)
        if rc != 0:
            raise ValueError("oracle kv_append failed (rc=%d)" % rc)


def paged_attention(q, q_dtype: str, pool: OraclePool, layer: int, block_tables, seq_lens,
                    scale: float, window: Tuple[int, int] = (0, INT32_MAX), threads: int = 0,
                    return_threads: bool = False):
    """fp64 decode attention; returns (out [B][Hq][D] float64, lse [B][Hq] float64)."""
    qq = to_numpy_bits(q, q_dtype)
    B, Hq, D = qq.shape
    assert D == pool.head_dim
    bt = np.ascontiguousarray(np.asarray(block_tables, dtype=np.int32))
    sl = np.ascontiguousarray(np.asarray(seq_lens, dtype=np.int32))
    out = np.zeros((B, Hq, D), dtype=np.float64)
    lse = np.zeros((B, Hq), dtype=np.float64)
    used = ctypes.c_int(0)
    rc = _load().or_paged_attention(
        _ptr(qq), _DT[q_dtype], _ptr(pool.k), _ptr(pool.v), _DT[pool.dtype], pool.num_layers,
        pool.num_blocks, pool.block_size, pool.kv_heads, pool.head_dim, layer, pool.k_scale,
        pool.v_scale, _ptr(bt), bt.shape[1], _ptr(sl), B, Hq, scale, int(window[0]),
        int(window[1]), _ptr(out), _ptr(lse), int(threads), ctypes.byref(used))
    if rc != 0:
        raise IndexError("oracle paged_attention: bad block table or length (rc=%d)" % rc)
    if return_threads:
        return out, lse, used.value
    return out, lse


def paged_attention_mq(q, q_dtype: str, pool: OraclePool, layer: int, block_tables, seq_lens,
                       scale: float, threads: int = 0, return_threads: bool = False):
    """fp64 multi-query attention: q [B][C][Hq][D], query c of sequence b at
    position L_b - C + c attends causally to tokens 0..L_b - C + c.
    Returns (out [B][C][Hq][D], lse [B][C][Hq]) (+ the thread count used)."""
    qq = to_numpy_bits(q, q_dtype)
    B, C, Hq, D = qq.shape
    assert D == pool.head_dim
    bt = np.ascontiguousarray(np.asarray(block_tables, dtype=np.int32))
    sl = np.ascontiguousarray(np.asarray(seq_lens, dtype=np.int32))
    out = np.zeros((B, C, Hq, D), dtype=np.float64)
    lse = np.zeros((B, C, Hq), dtype=np.float64)
    used = ctypes.c_int(0)
    rc = _load().or_paged_attention_mq(
        _ptr(qq), _DT[q_dtype], _ptr(pool.k), _ptr(pool.v), _DT[pool.dtype], pool.num_layers,
        pool.num_blocks, pool.block_size, pool.kv_heads, pool.head_dim, layer, pool.k_scale,
        pool.v_scale, _ptr(bt), bt.shape[1], _ptr(sl), B, C, Hq, scale, _ptr(out), _ptr(lse), int(threads),
        ctypes.byref(used))
    if rc != 0:
        raise IndexError("oracle paged_attention_mq: bad block table or length (rc=%d)" % rc)
    if return_threads:
        return out, lse, used.value
    return out, lse


def lse_combine(o_parts, lse_parts) -> Tuple[np.ndarray, float]:
    """Combine per-window (o_s, lse_s), o_parts [S][D] -> (out [D], lse)."""
    o = np.ascontiguousarray(np.asarray(o_parts, dtype=np.float64))
    l = np.ascontiguousarray(np.asarray(lse_parts, dtype=np.float64))
    S, D = o.shape
    out = np.empty(D, dtype=np.float64)
    lse = np.empty(1, dtype=np.float64)
    _load().or_lse_combine(_ptr(o), _ptr(l), S, D, _ptr(out), _ptr(lse))
    return out, float(lse[0])


def dequantized_pool_rows(pool: OraclePool, which: str) -> np.ndarray:
    """The pool's K or V values as float64 (E4M3 codes times their scale)."""
    arr = pool.k if which == "k" else pool.v
    if pool.dtype == "f32":
        return arr.astype(np.float64)
    if pool.dtype == "bf16":
        return bf16_decode(arr)
    sc = pool.k_scale if which == "k" else pool.v_scale
    return e4m3_decode(arr) * sc
