"""ctypes front end of the fp64 CPU oracle (test infrastructure only).

The shared library is compiled from ``pa_oracle.c`` with the system C compiler
on first use (or by the package build step).  Nothing here imports the CUDA
package; inputs arrive as numpy arrays (bf16 as uint16 bit patterns).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from typing import Optional, Sequence

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "pa_oracle.c")
_LIB = os.path.join(_HERE, "libpa_oracle.so")
_lib = None

_DTYPE_CODE = {"f32": 0, "bf16": 1}


def library_path() -> str:
    return _LIB


def build_oracle(force: bool = False) -> str:
    """Compile pa_oracle.c into libpa_oracle.so (plain C, -O2, pthreads)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-o", tmp, _SRC, "-lm", "-lpthread"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is None:
        build_oracle()
        lib = ctypes.CDLL(_LIB)
        P, I, L, D = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_double
        lib.oracle_reshape_and_cache.restype = I
        lib.oracle_reshape_and_cache.argtypes = [P, P, L, P, P, P, L, I, I, I, L, I]
        lib.oracle_paged_attention.restype = I
        lib.oracle_paged_attention.argtypes = [P, P, L, P, P, P, I, P, P, P, I, I, I, I, I, I, L,
                                               D, P, I, I]
        lib.oracle_split_partials.restype = I
        lib.oracle_split_partials.argtypes = [P, P, P, I, I, P, P, P, I, P, P, P, I, I, I, I, I,
                                              I, L, D]
        lib.oracle_split_combine.restype = I
        lib.oracle_split_combine.argtypes = [P, P, P, P, I, I, I, P, P, I, I, I, P]
        lib.oracle_paged_attention_kv.restype = I
        lib.oracle_paged_attention_kv.argtypes = [P, P, L, P, P, P, I, I, P, P, P, I, I, I, I, I,
                                                  I, L, D, P, I, I]
        lib.oracle_e4m3_value.restype = D
        lib.oracle_e4m3_value.argtypes = [I]
        lib.oracle_e4m3_encode.restype = I
        lib.oracle_e4m3_encode.argtypes = [ctypes.c_float]
        lib.oracle_quantize_kv_fp8.restype = I
        lib.oracle_quantize_kv_fp8.argtypes = [P, P, L, P, P, P, P, P, L, I, I, I, L, I]
        _lib = lib
    return _lib


def _ptr(a: Optional[np.ndarray]):
    return None if a is None else ctypes.c_void_p(a.ctypes.data)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def reshape_and_cache(new_k, new_v, key_cache, value_cache, slot_mapping, block_size: int):
    """Scatter new_k/new_v [T, H_kv, D] into copies of the pools; returns them."""
    lib = _load()
    kc = np.array(key_cache, copy=True, order="C")
    vc = np.array(value_cache, copy=True, order="C")
    nk = np.ascontiguousarray(new_k)
    nv = np.ascontiguousarray(new_v)
    sm = _c(slot_mapping, np.int64)
    T, Hkv, D = nk.shape
    rc = lib.oracle_reshape_and_cache(_ptr(nk), _ptr(nv), Hkv * D, _ptr(kc), _ptr(vc), _ptr(sm),
                                      T, Hkv, D, block_size, kc.shape[0], nk.itemsize)
    if rc:
        raise ValueError(f"oracle_reshape_and_cache: slot outside the pool (rc={rc})")
    return kc, vc


def paged_attention(q, key_cache, value_cache, cu_seqlens_q, seq_lens_k, block_tables, *,
                    dtype: str, num_q_heads: int, num_kv_heads: int, head_dim: int,
                    block_size: int, scale: float, causal: bool, sinks=None,
                    rows: Optional[Sequence[int]] = None, nthreads: Optional[int] = None):
    """fp64 attention for the query rows in ``rows`` (default: all).

    Returns an array [len(rows), H_q, D] of float64."""
    lib = _load()
    q = np.ascontiguousarray(q)
    total_q = q.shape[0]
    rows = np.arange(total_q, dtype=np.int64) if rows is None else _c(rows, np.int64)
    out = np.zeros((len(rows), num_q_heads, head_dim), dtype=np.float64)
    cu = _c(cu_seqlens_q, np.int32)
    sl = _c(seq_lens_k, np.int32)
    bt = _c(block_tables, np.int32)
    kc = np.ascontiguousarray(key_cache)
    vc = np.ascontiguousarray(value_cache)
    sk = None if sinks is None else _c(sinks, np.float64)
    nthreads = nthreads or os.cpu_count() or 1
    rc = lib.oracle_paged_attention(_ptr(out), _ptr(rows), len(rows), _ptr(q), _ptr(kc), _ptr(vc),
                                    _DTYPE_CODE[dtype], _ptr(cu), _ptr(sl), _ptr(bt), bt.shape[1],
                                    len(sl), num_q_heads, num_kv_heads, head_dim, block_size,
                                    kc.shape[0], float(scale), _ptr(sk), int(bool(causal)),
                                    int(nthreads))
    if rc:
        raise ValueError(f"oracle_paged_attention failed (rc={rc})")
    return out


def attention_of(w, rows=None, *, key_cache=None, value_cache=None, nthreads=None, **over):
    """Oracle attention for a Workload (pool after this step's scatter unless
    explicit pools are given)."""
    if key_cache is None:
        key_cache, value_cache = w.pool_with_new_tokens()
    args = dict(dtype=w.dtype, num_q_heads=w.num_q_heads, num_kv_heads=w.num_kv_heads,
                head_dim=w.head_dim, block_size=w.block_size, scale=w.scale, causal=w.causal,
                sinks=w.sinks)
    args.update(over)
    return paged_attention(w.q, key_cache, value_cache, w.cu_seqlens_q, w.seq_lens_k,
                           w.block_tables, rows=rows, nthreads=nthreads, **args)


def split_partials(q, key_cache, value_cache, cu_seqlens_q, seq_lens_k, block_tables, *,
                   dtype: str, num_q_heads: int, num_kv_heads: int, head_dim: int,
                   block_size: int, scale: float, partition_size: int, max_parts: int):
    """Split-KV partials (o, m, l) for the single-query requests, float64."""
    lib = _load()
    S = len(seq_lens_k)
    part_o = np.zeros((S, max_parts, num_q_heads, head_dim), dtype=np.float64)
    part_m = np.full((S, max_parts, num_q_heads), -np.inf, dtype=np.float64)
    part_l = np.zeros((S, max_parts, num_q_heads), dtype=np.float64)
    q = np.ascontiguousarray(q)
    kc = np.ascontiguousarray(key_cache)
    vc = np.ascontiguousarray(value_cache)
    bt = _c(block_tables, np.int32)
    rc = lib.oracle_split_partials(_ptr(part_o), _ptr(part_m), _ptr(part_l), max_parts,
                                   partition_size, _ptr(q), _ptr(kc), _ptr(vc),
                                   _DTYPE_CODE[dtype], _ptr(_c(cu_seqlens_q, np.int32)),
                                   _ptr(_c(seq_lens_k, np.int32)), _ptr(bt), bt.shape[1], S,
                                   num_q_heads, num_kv_heads, head_dim, block_size, kc.shape[0],
                                   float(scale))
    if rc:
        raise ValueError(f"oracle_split_partials failed (rc={rc})")
    return part_o, part_m, part_l


def split_combine(part_o, part_m, part_l, cu_seqlens_q, seq_lens_k, *, partition_size: int,
                  sinks=None):
    """The shared reduce over partials (float32 or float64 arrays).

    Returns [S, H_q, D] float64 (zeros for requests that are not single-query)."""
    lib = _load()
    f32 = part_o.dtype == np.float32
    dt = np.float32 if f32 else np.float64
    po = _c(part_o, dt)
    pm = _c(part_m, dt)
    pl = _c(part_l, dt)
    S, max_parts, Hq, D = po.shape
    out = np.zeros((S, Hq, D), dtype=np.float64)
    sk = None if sinks is None else _c(sinks, np.float64)
    rc = lib.oracle_split_combine(_ptr(out), _ptr(po), _ptr(pm), _ptr(pl), int(f32), max_parts,
                                  partition_size, _ptr(_c(cu_seqlens_q, np.int32)),
                                  _ptr(_c(seq_lens_k, np.int32)), S, Hq, D, _ptr(sk))
    if rc:
        raise ValueError(f"oracle_split_combine failed (rc={rc})")
    return out


# ---------------------------------------------------------------- quantised KV cache
def e4m3_values() -> np.ndarray:
    """The number each of the 256 E4M3 codes stands for (float64; NaN codes NaN)."""
    lib = _load()
    return np.array([lib.oracle_e4m3_value(c) for c in range(256)], dtype=np.float64)


def e4m3_encode(values) -> np.ndarray:
    """E4M3 codes of float32 values (nearest, ties to even, saturated at 448)."""
    lib = _load()
    v = np.asarray(values, dtype=np.float32).ravel()
    return np.array([lib.oracle_e4m3_encode(float(x)) for x in v], dtype=np.uint8)


def quantize_kv_fp8(new_k, new_v, key_codes, value_codes, key_scales, value_scales,
                    slot_mapping, block_size: int, dtype: str):
    """Scatter new_k/new_v [T, H_kv, D] (bf16 bits or float32) into copies of the
    quantised pools (codes [num_blocks, bs, H_kv, D] uint8, scales
    [num_blocks, bs, H_kv] float32); returns the four new arrays."""
    lib = _load()
    kc = np.array(key_codes, dtype=np.uint8, copy=True, order="C")
    vc = np.array(value_codes, dtype=np.uint8, copy=True, order="C")
    ks = np.array(key_scales, dtype=np.float32, copy=True, order="C")
    vs = np.array(value_scales, dtype=np.float32, copy=True, order="C")
    nk = np.ascontiguousarray(new_k)
    nv = np.ascontiguousarray(new_v)
    sm = _c(slot_mapping, np.int64)
    T, Hkv, D = nk.shape
    rc = lib.oracle_quantize_kv_fp8(_ptr(nk), _ptr(nv), Hkv * D, _ptr(kc), _ptr(vc), _ptr(ks),
                                    _ptr(vs), _ptr(sm), T, Hkv, D, block_size, kc.shape[0],
                                    _DTYPE_CODE[dtype])
    if rc:
        raise ValueError(f"oracle_quantize_kv_fp8: slot outside the pool (rc={rc})")
    return kc, vc, ks, vs


def dequantize_kv_fp8(codes, scales) -> np.ndarray:
    """value(code) * scale for a quantised pool, exactly (float64)."""
    table = e4m3_values()
    return table[np.asarray(codes, dtype=np.uint8)] * np.asarray(scales, np.float64)[..., None]


def paged_attention_kv(q, key_cache_f64, value_cache_f64, cu_seqlens_q, seq_lens_k,
                       block_tables, *, q_dtype: str, num_q_heads: int, num_kv_heads: int,
                       head_dim: int, block_size: int, scale: float, causal: bool, sinks=None,
                       rows: Optional[Sequence[int]] = None, nthreads: Optional[int] = None):
    """fp64 attention of q (bf16 bits or float32) over float64 pools (a
    dequantised cache), for the query rows in ``rows`` (default: all)."""
    lib = _load()
    q = np.ascontiguousarray(q)
    rows = np.arange(q.shape[0], dtype=np.int64) if rows is None else _c(rows, np.int64)
    out = np.zeros((len(rows), num_q_heads, head_dim), dtype=np.float64)
    cu = _c(cu_seqlens_q, np.int32)
    sl = _c(seq_lens_k, np.int32)
    bt = _c(block_tables, np.int32)
    kc = _c(key_cache_f64, np.float64)
    vc = _c(value_cache_f64, np.float64)
    sk = None if sinks is None else _c(sinks, np.float64)
    nthreads = nthreads or os.cpu_count() or 1
    rc = lib.oracle_paged_attention_kv(_ptr(out), _ptr(rows), len(rows), _ptr(q), _ptr(kc),
                                       _ptr(vc), _DTYPE_CODE[q_dtype], 2, _ptr(cu), _ptr(sl),
                                       _ptr(bt), bt.shape[1], len(sl), num_q_heads, num_kv_heads,
                                       head_dim, block_size, kc.shape[0], float(scale), _ptr(sk),
                                       int(bool(causal)), int(nthreads))
    if rc:
        raise ValueError(f"oracle_paged_attention_kv failed (rc={rc})")
    return out
