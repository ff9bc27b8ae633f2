"""Shared helpers of the GPU parity tests: move a seeded workload to the GPU,
run the library's calls through the binding, compare with the fp64 oracle.

Tolerances (float outputs against the fp64 oracle):
  float32 inputs:  max |err| <= 1e-5
  bf16 inputs:     max |err| <= 2e-2 and mean |err| <= 2e-3
The scatter is compared bit for bit.
"""
from __future__ import annotations

import numpy as np
import torch

from oracle.oracle import attention_of
from oracle import oracle as orc
from paged_kv_varlen_gb300 import binding as pa
from paged_kv_varlen_gb300 import workloads as wl

TOL_F32_MAX = 1e-5
TOL_BF16_MAX = 2e-2
TOL_BF16_MEAN = 2e-3


def to_dev(a: np.ndarray, dtype: str, device="cuda") -> torch.Tensor:
    """Stored array (float32, or bf16 bits in uint16) -> device tensor."""
    if dtype == wl.BF16:
        t = torch.from_numpy(np.ascontiguousarray(a).view(np.int16))
        return t.to(device).view(torch.bfloat16)
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(device)


def from_dev(t: torch.Tensor) -> np.ndarray:
    """Device tensor -> float64 numpy (exact widening)."""
    return t.float().cpu().numpy().astype(np.float64)


def dev_bits(t: torch.Tensor) -> np.ndarray:
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).cpu().numpy().view(np.uint16)
    return t.view(torch.int32).cpu().numpy().view(np.uint32)


class DeviceWorkload:
    """A workload's tensors on the GPU (pool *before* this step's scatter)."""

    def __init__(self, w: wl.Workload, device="cuda"):
        self.w = w
        self.q = to_dev(w.q, w.dtype, device)
        self.key_cache = to_dev(w.key_cache, w.dtype, device)
        self.value_cache = to_dev(w.value_cache, w.dtype, device)
        self.new_k = to_dev(w.new_k, w.dtype, device)
        self.new_v = to_dev(w.new_v, w.dtype, device)
        self.slot_mapping = torch.from_numpy(w.slot_mapping).to(device)
        self.cu_seqlens_q = torch.from_numpy(w.cu_seqlens_q).to(device)
        self.seq_lens_k = torch.from_numpy(w.seq_lens_k).to(device)
        self.block_tables = torch.from_numpy(w.block_tables).to(device)
        self.sinks = (torch.from_numpy(w.sinks.astype(np.float32)).to(device)
                      if w.sinks is not None else None)
        self.out = torch.empty_like(self.q)

    def scatter(self):
        pa.pa_reshape_and_cache(self.new_k, self.new_v, self.key_cache, self.value_cache,
                                self.slot_mapping)

    def poisoned_workspace(self, partition_size):
        """A workspace of the size the call needs, every byte 0xFF (NaN as fp32):
        its contents need no initialisation, so no result may depend on them."""
        w = self.w
        n = pa.pa_varlen_attention_workspace_size(w.num_seqs, w.max_seqlen_k, w.num_q_heads,
                                                  w.head_dim, partition_size)
        return torch.full((max(n, 16),), 0xFF, dtype=torch.uint8, device="cuda")

    def attention(self, partition_size=None, workspace=None, sinks="default", out=None):
        w = self.w
        out = self.out if out is None else out
        P = w.partition_size if partition_size is None else partition_size
        if workspace is None:
            workspace = self.poisoned_workspace(P)
        pa.pa_varlen_attention(
            out, self.q, self.key_cache, self.value_cache, self.cu_seqlens_q, self.seq_lens_k,
            self.block_tables, max_seqlen_q=w.max_seqlen_q, max_seqlen_k=w.max_seqlen_k,
            scale=w.scale, sinks=self.sinks if sinks == "default" else sinks, causal=w.causal,
            partition_size=P, workspace=workspace)
        return out

    def step(self, **kw):
        self.scatter()
        return self.attention(**kw)

    def fused_step(self, partition_size=None, out=None):
        """The same step through pa_scatter_and_attend (one call)."""
        w = self.w
        out = self.out if out is None else out
        P = w.partition_size if partition_size is None else partition_size
        pa.pa_scatter_and_attend(
            self.new_k, self.new_v, self.slot_mapping, out, self.q, self.key_cache,
            self.value_cache, self.cu_seqlens_q, self.seq_lens_k, self.block_tables,
            max_seqlen_q=w.max_seqlen_q, max_seqlen_k=w.max_seqlen_k, scale=w.scale,
            sinks=self.sinks, causal=w.causal, partition_size=P,
            workspace=self.poisoned_workspace(P))
        return out


def assert_close(got: np.ndarray, ref: np.ndarray, dtype: str, what: str = ""):
    err = np.abs(got - ref)
    assert np.isfinite(got).all(), f"{what}: non-finite output"
    mx, mean = float(err.max()) if err.size else 0.0, float(err.mean()) if err.size else 0.0
    if dtype == wl.F32:
        assert mx <= TOL_F32_MAX, f"{what}: max abs err {mx:.3e} > {TOL_F32_MAX}"
    else:
        assert mx <= TOL_BF16_MAX, f"{what}: max abs err {mx:.3e} > {TOL_BF16_MAX}"
        assert mean <= TOL_BF16_MEAN, f"{what}: mean abs err {mean:.3e} > {TOL_BF16_MEAN}"
    return mx, mean


def check_scatter(dw: "DeviceWorkload", slot_mapping=None):
    """Runs the GPU scatter and checks the WHOLE pool: the pages this step
    touches bit for bit against the oracle's scatter, every other page bit for
    bit against its bytes before the step (compared on the device, so a large
    pool costs no host copy).  Slots past the pool are skipped like negative
    ones (reading R5), so the oracle gets -1 for them.  Returns the oracle's
    pools."""
    w = dw.w
    sm = w.slot_mapping if slot_mapping is None else np.asarray(slot_mapping, np.int64)
    nslots = w.num_blocks * w.block_size
    kc_before = dev_bits_t(dw.key_cache).clone()
    vc_before = dev_bits_t(dw.value_cache).clone()
    pa.pa_reshape_and_cache(dw.new_k, dw.new_v, dw.key_cache, dw.value_cache,
                            torch.from_numpy(sm).to(dw.key_cache.device))
    sm_oracle = np.where((sm >= 0) & (sm < nslots), sm, -1)
    kc_ref, vc_ref = orc.reshape_and_cache(w.new_k, w.new_v, w.key_cache, w.value_cache,
                                           sm_oracle, w.block_size)
    pages = np.unique(sm_oracle[sm_oracle >= 0] // w.block_size)
    view = np.uint16 if w.dtype == wl.BF16 else np.uint32
    pidx = torch.from_numpy(pages).to(dw.key_cache.device)
    assert np.array_equal(dev_bits(dw.key_cache[pidx]), kc_ref[pages].view(view)), \
        "key cache scatter differs"
    assert np.array_equal(dev_bits(dw.value_cache[pidx]), vc_ref[pages].view(view)), \
        "value cache scatter differs"
    untouched = torch.ones(w.num_blocks, dtype=torch.bool, device=dw.key_cache.device)
    untouched[pidx] = False
    assert torch.equal(dev_bits_t(dw.key_cache)[untouched], kc_before[untouched]), \
        "the scatter wrote a page no token maps to (key cache)"
    assert torch.equal(dev_bits_t(dw.value_cache)[untouched], vc_before[untouched]), \
        "the scatter wrote a page no token maps to (value cache)"
    return kc_ref, vc_ref


def dev_bits_t(t: torch.Tensor) -> torch.Tensor:
    """Bit view of a device tensor (NaN payloads compare equal)."""
    return t.view(torch.int16) if t.dtype == torch.bfloat16 else t.view(torch.int32)


def check_step(w: wl.Workload, rows=None, partition_size=None, nthreads=None):
    """Scatter + attention on the GPU vs the oracle (bit-exact whole pool after
    the scatter, tolerance on the sampled output rows).  Returns (max err,
    mean err)."""
    dw = DeviceWorkload(w)
    kc_ref, vc_ref = check_scatter(dw)
    dw.attention(partition_size=partition_size)
    torch.cuda.synchronize()
    assert pa.pa_device_error() == 0
    out = from_dev(dw.out)
    sel = np.arange(w.total_q) if rows is None else np.asarray(rows, dtype=np.int64)
    ref = attention_of(w, rows=sel, key_cache=kc_ref, value_cache=vc_ref, nthreads=nthreads)
    return assert_close(out[sel], ref, w.dtype, w.name)
