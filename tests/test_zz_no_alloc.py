"""pa_varlen_attention_static_scratch: attention for callers that cannot
allocate device memory (a host framework that owns every allocation, a
serving loop that must not stall on cudaMalloc/cudaFree, a plugin without an
allocator).  Its split-KV partials live in the library's fixed 16 MiB device
array instead of a caller workspace.

Checked through the C ABI against pa_varlen_attention with a workspace, on two
calls in a row (the array keeps the previous call's contents), and a call
that needs more scratch than the array holds must be refused.  This file is
collected last on purpose; it also passes when run alone in a fresh process.
"""
import numpy as np
import pytest
import torch

from harness import DeviceWorkload, assert_close, from_dev
from paged_kv_varlen_gb300 import binding as pa
from paged_kv_varlen_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


def _static_call(dw, out, partition_size):
    w = dw.w
    return pa.pa_varlen_attention_static_scratch(
        out, dw.q, dw.key_cache, dw.value_cache, dw.cu_seqlens_q, dw.seq_lens_k,
        dw.block_tables, max_seqlen_q=w.max_seqlen_q, max_seqlen_k=w.max_seqlen_k,
        scale=w.scale, sinks=dw.sinks, causal=w.causal, partition_size=partition_size)


@pytest.mark.parametrize("dtype", [wl.BF16, wl.F32])
def test_static_scratch_matches_workspace_call_twice(dtype):
    # decode rows long enough to split into several 256-key partitions, plus
    # multi-query rows in the same call
    w = wl.random_small(4242, dtype=dtype, num_seqs=7, num_q_heads=8, num_kv_heads=2,
                        head_dim=128, block_size=16, max_prior=3000, max_q=3, with_sinks=True)
    w2 = wl.random_small(4243, dtype=dtype, num_seqs=5, num_q_heads=8, num_kv_heads=2,
                         head_dim=128, block_size=16, max_prior=1800, max_q=1)
    for i, case in enumerate((w, w2)):       # two calls in a row, different shapes
        dw = DeviceWorkload(case)
        dw.scatter()
        ref = dw.attention(partition_size=256, out=torch.empty_like(dw.q))
        out = torch.full_like(dw.q, float("nan"))
        torch.cuda.synchronize()
        free_before = torch.cuda.mem_get_info()[0]
        torch_before = torch.cuda.memory_allocated()
        _static_call(dw, out, 256)
        torch.cuda.synchronize()
        if i == 1:
            # after the first call has looked up the array's address (which may
            # load the library's module holding it), a call changes neither the
            # device's free memory nor torch's allocations
            assert torch.cuda.mem_get_info()[0] == free_before
            assert torch.cuda.memory_allocated() == torch_before
        assert_close(from_dev(out), from_dev(ref), case.dtype, f"static scratch {case.name}")
        assert pa.pa_device_error() == 0


def test_static_scratch_refuses_calls_that_need_more():
    # 64 decode rows with 64k contexts split into 256-key partitions need
    # 64 * 256 * 32 * (128 + 2) * 4 bytes of partials: far above 16 MiB
    q = torch.zeros(64, 32, 128, dtype=torch.bfloat16, device="cuda")
    kc = torch.zeros(8, 16, 8, 128, dtype=torch.bfloat16, device="cuda")
    cu = torch.arange(65, dtype=torch.int32, device="cuda")
    sl = torch.full((64,), 16, dtype=torch.int32, device="cuda")
    bt = torch.zeros(64, 4096, dtype=torch.int32, device="cuda")
    out = torch.zeros_like(q)
    with pytest.raises(pa.PAError, match="WORKSPACE.*needs [0-9]+ bytes"):
        pa.pa_varlen_attention_static_scratch(out, q, kc, kc, cu, sl, bt, max_seqlen_q=1,
                                              max_seqlen_k=65536, scale=0.1,
                                              partition_size=256)
    assert torch.count_nonzero(out) == 0     # nothing was launched
