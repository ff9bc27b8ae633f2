"""Unified paged variable-length attention for GB300 (sm_103a).

The compute lives in a C-ABI shared library (``libpa.so``) built from the
CUDA sources in ``csrc/``; ``binding`` marshals torch tensors into its calls:

  pa_reshape_and_cache   scatter this step's K/V rows into the page pool
  pa_varlen_attention    attention over packed query rows and paged K/V
  pa_split_kv_reduce     merge split-KV partials (log2-space max / exp-sum)

``staging`` packs a step's input arrays into one pinned host buffer (one
host-to-device copy per step).  Importing the package does not load the library; the first call does, and it
raises if the library is missing -- there is no CPU fallback.
"""

__all__ = ["binding", "staging", "workloads"]
