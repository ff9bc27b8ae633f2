"""Thin Python binding of libpa.so (ctypes): argument marshalling only.

Each function has the name of the C entry point it calls and takes torch
tensors that already live on the current CUDA device; it passes their data
pointers, sizes and the current CUDA stream, and raises ``PAError`` on a
non-zero status.  Every step of the computation runs in the library's CUDA
kernels; if ``libpa.so`` is missing this module raises instead of computing
anything itself.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libpa.so")

PA_F32, PA_BF16 = 0, 1
_DTYPES = {torch.float32: PA_F32, torch.bfloat16: PA_BF16}

_lib = None


class PAError(RuntimeError):
    pass


def load_library(path: Optional[str] = None) -> ctypes.CDLL:
    """Load libpa.so (built by paged_kv_varlen_gb300.build); raise if absent."""
    global _lib
    if _lib is not None:
        return _lib
    path = path or LIB_PATH
    if not os.path.exists(path):
        raise PAError(f"{path} is missing: build it with `python -m paged_kv_varlen_gb300.build` "
                      "(there is no CPU fallback)")
    lib = ctypes.CDLL(path)
    P, I, L, F, S = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_float, ctypes.c_size_t
    lib.pa_status_string.restype = ctypes.c_char_p
    lib.pa_status_string.argtypes = [I]
    lib.pa_last_error_string.restype = ctypes.c_char_p
    lib.pa_last_error_string.argtypes = []
    lib.pa_build_info.restype = ctypes.c_char_p
    lib.pa_build_info.argtypes = []
    lib.pa_describe_plan.restype = I
    lib.pa_describe_plan.argtypes = [I, L, I, I, I, I, I, I, I, I, I, ctypes.c_char_p, S]
    lib.pa_last_plan.restype = ctypes.c_char_p
    lib.pa_last_plan.argtypes = []
    lib.pa_reshape_and_cache.restype = I
    lib.pa_reshape_and_cache.argtypes = [P, P, L, P, P, P, L, I, I, I, L, I, P]
    lib.pa_varlen_attention.restype = I
    lib.pa_varlen_attention.argtypes = [P, P, P, P, P, P, P, I, I, L, I, I, I, I, I, I, L, F, P,
                                        I, I, P, S, I, P]
    lib.pa_varlen_attention_workspace_size.restype = S
    lib.pa_varlen_attention_workspace_size.argtypes = [I, I, I, I, I]
    lib.pa_choose_partition_size.restype = I
    lib.pa_choose_partition_size.argtypes = [I, I, I, I, I]
    lib.pa_scatter_and_attend.restype = I
    lib.pa_scatter_and_attend.argtypes = [P, P, L, P, L, P, P, P, P, P, P, P, I, I, L, I, I, I, I,
                                          I, I, L, F, P, I, I, P, S, I, P]
    lib.pa_split_kv_reduce.restype = I
    lib.pa_split_kv_reduce.argtypes = [P, P, P, P, P, P, I, I, I, I, I, P, I, P]
    lib.pa_device_error.restype = I
    lib.pa_device_error.argtypes = [ctypes.POINTER(ctypes.c_int)]
    lib.pa_test_expire_next_wait.restype = None
    lib.pa_test_expire_next_wait.argtypes = []
    lib.pa_reshape_and_cache_fp8.restype = I
    lib.pa_reshape_and_cache_fp8.argtypes = [P, P, L, P, P, P, P, P, L, I, I, I, L, I, P]
    lib.pa_varlen_attention_fp8kv.restype = I
    lib.pa_varlen_attention_fp8kv.argtypes = [P, P, P, P, P, P, P, P, P, I, I, L, I, I, I, I, I,
                                              I, L, F, P, I, I, P, S, I, P]
    _lib = lib
    return lib


def _check(status: int, what: str):
    if status != 0:
        lib = load_library()
        raise PAError(f"{what}: {lib.pa_status_string(status).decode()} "
                      f"({lib.pa_last_error_string().decode()})")


def _ptr(t: Optional[torch.Tensor]):
    if t is None:
        return None
    if not t.is_cuda:
        raise PAError("tensors must live on a CUDA device")
    if not t.is_contiguous():
        raise PAError("tensors must be contiguous")
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream) -> ctypes.c_void_p:
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _dtype(t: torch.Tensor) -> int:
    try:
        return _DTYPES[t.dtype]
    except KeyError:
        raise PAError(f"unsupported dtype {t.dtype}: float32 or bfloat16") from None


def build_info() -> str:
    return load_library().pa_build_info().decode()


def pa_reshape_and_cache(key: torch.Tensor, value: torch.Tensor, key_cache: torch.Tensor,
                         value_cache: torch.Tensor, slot_mapping: torch.Tensor, *, stream=None):
    """key/value [T, H_kv, D] (rows may be strided, e.g. slices of a fused QKV),
    caches [num_blocks, block_size, H_kv, D], slot_mapping [T] int64."""
    lib = load_library()
    T, Hkv, D = key.shape
    nb, bs = key_cache.shape[0], key_cache.shape[1]
    if key.stride() != value.stride() or key.stride(2) != 1 or key.stride(1) != D:
        raise PAError("key/value rows must be [H_kv, D]-contiguous with equal strides")
    if slot_mapping.dtype != torch.int64:
        raise PAError("slot_mapping must be int64")
    st = lib.pa_reshape_and_cache(ctypes.c_void_p(key.data_ptr()), ctypes.c_void_p(value.data_ptr()),
                                  key.stride(0), _ptr(key_cache), _ptr(value_cache),
                                  _ptr(slot_mapping), T, Hkv, D, bs, nb, _dtype(key_cache),
                                  _stream(stream))
    _check(st, "pa_reshape_and_cache")


def pa_varlen_attention_workspace_size(num_seqs: int, max_seqlen_k: int, num_q_heads: int,
                                       head_dim: int, partition_size: int = 0) -> int:
    return int(load_library().pa_varlen_attention_workspace_size(
        num_seqs, max_seqlen_k, num_q_heads, head_dim, partition_size))


def _parse_plan(line: str) -> dict:
    return dict(kv.split("=", 1) for kv in line.split())


def pa_describe_plan(num_seqs: int, total_q: int, max_seqlen_q: int, max_seqlen_k: int,
                     num_q_heads: int, num_kv_heads: int, head_dim: int, partition_size: int,
                     dtype, sm_count: int, quantised: bool = False) -> dict:
    """The launches an attention call with these sizes makes (host only), as a
    dict of the library's key=value plan line.  dtype: "bf16", "f32" or a
    torch dtype."""
    buf = ctypes.create_string_buffer(512)
    st = load_library().pa_describe_plan(num_seqs, total_q, max_seqlen_q, max_seqlen_k,
                                         num_q_heads, num_kv_heads, head_dim, partition_size,
                                         {"bf16": PA_BF16, "f32": PA_F32}.get(dtype, None)
                                         if isinstance(dtype, str) else _DTYPES[dtype],
                                         int(bool(quantised)), sm_count, buf, 512)
    _check(st, "pa_describe_plan")
    return _parse_plan(buf.value.decode())


def pa_last_plan() -> dict:
    """The plan of the last attention call this thread launched ({} before any)."""
    line = load_library().pa_last_plan().decode()
    return {} if line == "none" else _parse_plan(line)


def pa_choose_partition_size(num_seqs: int, num_kv_heads: int, max_seqlen_k: int,
                             partition_size: int, sm_count: int) -> int:
    return int(load_library().pa_choose_partition_size(num_seqs, num_kv_heads, max_seqlen_k,
                                                        partition_size, sm_count))


def pa_varlen_attention(out: torch.Tensor, q: torch.Tensor, key_cache: torch.Tensor,
                        value_cache: torch.Tensor, cu_seqlens_q: torch.Tensor,
                        seq_lens_k: torch.Tensor, block_tables: torch.Tensor, *,
                        max_seqlen_q: int, max_seqlen_k: int, scale: float,
                        sinks: Optional[torch.Tensor] = None, causal: bool = True,
                        partition_size: int = 0, workspace: Optional[torch.Tensor] = None,
                        stream=None) -> torch.Tensor:
    """q/out [total_q, H_q, D]; caches [num_blocks, block_size, H_kv, D];
    cu_seqlens_q [S+1], seq_lens_k [S], block_tables [S, max_blocks] int32.
    ``workspace`` (uint8, device) is allocated here when not given."""
    lib = load_library()
    total_q, Hq, D = q.shape
    nb, bs, Hkv, _ = key_cache.shape
    S = seq_lens_k.shape[0]
    for name, t in (("cu_seqlens_q", cu_seqlens_q), ("seq_lens_k", seq_lens_k),
                    ("block_tables", block_tables)):
        if t.dtype != torch.int32:
            raise PAError(f"{name} must be int32")
    if sinks is not None and sinks.dtype != torch.float32:
        raise PAError("sinks must be float32")
    if workspace is None:
        nbytes = pa_varlen_attention_workspace_size(S, max_seqlen_k, Hq, D, partition_size)
        workspace = torch.empty(max(nbytes, 1), dtype=torch.uint8, device=q.device)
    st = lib.pa_varlen_attention(_ptr(out), _ptr(q), _ptr(key_cache), _ptr(value_cache),
                                 _ptr(cu_seqlens_q), _ptr(seq_lens_k), _ptr(block_tables),
                                 block_tables.shape[1], S, total_q, int(max_seqlen_q),
                                 int(max_seqlen_k), Hq, Hkv, D, bs, nb, float(scale),
                                 _ptr(sinks), int(bool(causal)), int(partition_size),
                                 _ptr(workspace), workspace.numel(), _dtype(q), _stream(stream))
    _check(st, "pa_varlen_attention")
    return out


def pa_scatter_and_attend(new_k: torch.Tensor, new_v: torch.Tensor, slot_mapping: torch.Tensor,
                          out: torch.Tensor, q: torch.Tensor, key_cache: torch.Tensor,
                          value_cache: torch.Tensor, cu_seqlens_q: torch.Tensor,
                          seq_lens_k: torch.Tensor, block_tables: torch.Tensor, *,
                          max_seqlen_q: int, max_seqlen_k: int, scale: float,
                          sinks: Optional[torch.Tensor] = None, causal: bool = True,
                          partition_size: int = 0, workspace: Optional[torch.Tensor] = None,
                          stream=None) -> torch.Tensor:
    """pa_reshape_and_cache(new_k, new_v, ...) then pa_varlen_attention(...) as one
    call; new_k/new_v [total_q, H_kv, D] (rows may be strided), slot_mapping int64."""
    lib = load_library()
    total_q, Hq, D = q.shape
    nb, bs, Hkv, _ = key_cache.shape
    S = seq_lens_k.shape[0]
    if new_k.stride() != new_v.stride() or new_k.stride(2) != 1 or new_k.stride(1) != D:
        raise PAError("new_k/new_v rows must be [H_kv, D]-contiguous with equal strides")
    if slot_mapping.dtype != torch.int64:
        raise PAError("slot_mapping must be int64")
    for name, t in (("cu_seqlens_q", cu_seqlens_q), ("seq_lens_k", seq_lens_k),
                    ("block_tables", block_tables)):
        if t.dtype != torch.int32:
            raise PAError(f"{name} must be int32")
    if sinks is not None and sinks.dtype != torch.float32:
        raise PAError("sinks must be float32")
    if workspace is None:
        nbytes = pa_varlen_attention_workspace_size(S, max_seqlen_k, Hq, D, partition_size)
        workspace = torch.empty(max(nbytes, 1), dtype=torch.uint8, device=q.device)
    st = lib.pa_scatter_and_attend(
        ctypes.c_void_p(new_k.data_ptr()), ctypes.c_void_p(new_v.data_ptr()), new_k.stride(0),
        _ptr(slot_mapping), new_k.shape[0], _ptr(out), _ptr(q), _ptr(key_cache),
        _ptr(value_cache), _ptr(cu_seqlens_q), _ptr(seq_lens_k), _ptr(block_tables),
        block_tables.shape[1], S, total_q, int(max_seqlen_q), int(max_seqlen_k), Hq, Hkv, D, bs,
        nb, float(scale), _ptr(sinks), int(bool(causal)), int(partition_size), _ptr(workspace),
        workspace.numel(), _dtype(q), _stream(stream))
    _check(st, "pa_scatter_and_attend")
    return out


def pa_split_kv_reduce(out: torch.Tensor, part_out: torch.Tensor, part_max: torch.Tensor,
                       part_sum: torch.Tensor, cu_seqlens_q: torch.Tensor,
                       seq_lens_k: torch.Tensor, *, partition_size: int,
                       sinks: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """part_out [S, max_parts, H_q, D], part_max/part_sum [S, max_parts, H_q] float32."""
    lib = load_library()
    S, max_parts, Hq, D = part_out.shape
    st = lib.pa_split_kv_reduce(_ptr(out), _ptr(part_out), _ptr(part_max), _ptr(part_sum),
                                _ptr(cu_seqlens_q), _ptr(seq_lens_k), S, max_parts,
                                int(partition_size), Hq, D, _ptr(sinks), _dtype(out),
                                _stream(stream))
    _check(st, "pa_split_kv_reduce")
    return out


def pa_device_error() -> int:
    """Read and clear the library's device error word (synchronises)."""
    code = ctypes.c_int(0)
    _check(load_library().pa_device_error(ctypes.byref(code)), "pa_device_error")
    return code.value


def pa_test_expire_next_wait() -> None:
    """Test hook: the next multi-query launch skips one K tile per CTA, so a
    bounded wait runs out and sets the device error word (no fault)."""
    load_library().pa_test_expire_next_wait()


def pa_varlen_attention_static_scratch(out: torch.Tensor, q: torch.Tensor,
                                       key_cache: torch.Tensor, value_cache: torch.Tensor,
                                       cu_seqlens_q: torch.Tensor, seq_lens_k: torch.Tensor,
                                       block_tables: torch.Tensor, *, max_seqlen_q: int,
                                       max_seqlen_k: int, scale: float,
                                       sinks: Optional[torch.Tensor] = None, causal: bool = True,
                                       partition_size: int = 0, stream=None) -> torch.Tensor:
    """pa_varlen_attention without a workspace, for callers that must not
    allocate device memory: the split-KV partials go to the library's fixed
    16 MiB device scratch (shared by all calls; order overlapping calls on one
    stream).  Raises PAError (PA_ERR_WORKSPACE) when a call needs more."""
    lib = load_library()
    fn = lib.pa_varlen_attention_static_scratch
    if fn.argtypes is None:
        P, I, L, F = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_float
        fn.restype = I
        fn.argtypes = [P, P, P, P, P, P, P, I, I, L, I, I, I, I, I, I, L, F, P, I, I, I, P]
    total_q, Hq, D = q.shape
    nb, bs, Hkv, _ = key_cache.shape
    st = fn(_ptr(out), _ptr(q), _ptr(key_cache), _ptr(value_cache), _ptr(cu_seqlens_q),
            _ptr(seq_lens_k), _ptr(block_tables), block_tables.shape[1], seq_lens_k.shape[0],
            total_q, int(max_seqlen_q), int(max_seqlen_k), Hq, Hkv, D, bs, nb, float(scale),
            _ptr(sinks), int(bool(causal)), int(partition_size), _dtype(q), _stream(stream))
    _check(st, "pa_varlen_attention_static_scratch")
    return out


# ---------------------------------------------------------------- quantised KV cache
def pa_reshape_and_cache_fp8(key: torch.Tensor, value: torch.Tensor, key_codes: torch.Tensor,
                             value_codes: torch.Tensor, key_scales: torch.Tensor,
                             value_scales: torch.Tensor, slot_mapping: torch.Tensor, *,
                             stream=None):
    """key/value [T, H_kv, D] (bf16 or float32; rows may be strided), codes
    [num_blocks, block_size, H_kv, D] uint8, scales [num_blocks, block_size,
    H_kv] float32, slot_mapping [T] int64."""
    lib = load_library()
    T, Hkv, D = key.shape
    nb, bs = key_codes.shape[0], key_codes.shape[1]
    if key.stride() != value.stride() or key.stride(2) != 1 or key.stride(1) != D:
        raise PAError("key/value rows must be [H_kv, D]-contiguous with equal strides")
    if slot_mapping.dtype != torch.int64:
        raise PAError("slot_mapping must be int64")
    if key_codes.dtype != torch.uint8 or key_scales.dtype != torch.float32:
        raise PAError("codes must be uint8 and scales float32")
    st = lib.pa_reshape_and_cache_fp8(ctypes.c_void_p(key.data_ptr()),
                                      ctypes.c_void_p(value.data_ptr()), key.stride(0),
                                      _ptr(key_codes), _ptr(value_codes), _ptr(key_scales),
                                      _ptr(value_scales), _ptr(slot_mapping), T, Hkv, D, bs, nb,
                                      _dtype(key), _stream(stream))
    _check(st, "pa_reshape_and_cache_fp8")


def pa_varlen_attention_fp8kv(out: torch.Tensor, q: torch.Tensor, key_codes: torch.Tensor,
                              value_codes: torch.Tensor, key_scales: torch.Tensor,
                              value_scales: torch.Tensor, cu_seqlens_q: torch.Tensor,
                              seq_lens_k: torch.Tensor, block_tables: torch.Tensor, *,
                              max_seqlen_q: int, max_seqlen_k: int, scale: float,
                              sinks: Optional[torch.Tensor] = None, causal: bool = True,
                              partition_size: int = 0, workspace: Optional[torch.Tensor] = None,
                              stream=None) -> torch.Tensor:
    """pa_varlen_attention over the quantised cache (codes uint8 [num_blocks,
    block_size, H_kv, D], scales float32 [num_blocks, block_size, H_kv]); q/out
    bf16."""
    lib = load_library()
    total_q, Hq, D = q.shape
    nb, bs, Hkv, _ = key_codes.shape
    S = seq_lens_k.shape[0]
    for name, t in (("cu_seqlens_q", cu_seqlens_q), ("seq_lens_k", seq_lens_k),
                    ("block_tables", block_tables)):
        if t.dtype != torch.int32:
            raise PAError(f"{name} must be int32")
    if sinks is not None and sinks.dtype != torch.float32:
        raise PAError("sinks must be float32")
    if workspace is None:
        nbytes = pa_varlen_attention_workspace_size(S, max_seqlen_k, Hq, D, partition_size)
        workspace = torch.empty(max(nbytes, 1), dtype=torch.uint8, device=q.device)
    st = lib.pa_varlen_attention_fp8kv(
        _ptr(out), _ptr(q), _ptr(key_codes), _ptr(value_codes), _ptr(key_scales),
        _ptr(value_scales), _ptr(cu_seqlens_q), _ptr(seq_lens_k), _ptr(block_tables),
        block_tables.shape[1], S, total_q, int(max_seqlen_q), int(max_seqlen_k), Hq, Hkv, D, bs,
        nb, float(scale), _ptr(sinks), int(bool(causal)), int(partition_size), _ptr(workspace),
        workspace.numel(), _dtype(q), _stream(stream))
    _check(st, "pa_varlen_attention_fp8kv")
    return out
