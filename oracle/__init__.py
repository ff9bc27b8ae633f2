"""CPU oracle for paged varlen attention -- TEST INFRASTRUCTURE, NOT THE PRODUCT.

A plain fp64 C implementation (``pa_oracle.c``) of what the hot path computes,
loaded through ctypes.  Only the tests, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline / reference leg may import this package; the CUDA
library and its Python binding never do.

Functions mirror the library's calls but take numpy arrays and return float64:
  reshape_and_cache(...)        byte-exact scatter (returns new pool arrays)
  paged_attention(w, rows=...)  fp64 attention for selected query rows
  split_partials / split_combine  the split-KV partials and shared reduce
  quantize_kv_fp8 / dequantize_kv_fp8 / paged_attention_kv  the quantised KV
                                cache (8-bit E4M3 codes, a scale per token and head)
  e4m3_values / e4m3_encode     the 8-bit float format itself
"""
from .oracle import (  # noqa: F401
    build_oracle,
    attention_of,
    paged_attention,
    reshape_and_cache,
    split_combine,
    split_partials,
    library_path,
    e4m3_encode,
    e4m3_values,
    quantize_kv_fp8,
    dequantize_kv_fp8,
    paged_attention_kv,
)
