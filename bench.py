"""Benchmark of the paged varlen attention hot path on GB300.

One step = one pass of the whole hot path over one batch: the KV scatter of
this step's tokens, then attention over the packed query rows and paged K/V
(the split-KV decode kernel and its shared reduce for single-query rows, the
tcgen05 kernel for multi-query rows) -- one pa_scatter_and_attend call
(``--step two-call``: pa_reshape_and_cache then pa_varlen_attention).

Headline workload (``value``): the GQA decode batch -- 32 requests with
contexts U[512, 8192], (H_q, H_kv, D) = (32, 8, 128), bf16, block size 16,
40k-page shuffled pool, split-KV partition 512.  Metric: decode KV GB/s =
algorithmic bytes per step / step time.  The default run also times the other
three workloads of the metric, each in a sub-record of the same JSON line
(``workloads``: 2 varlen causal prefill -> TFLOP/s; 3 mixed packed step ->
tokens/s; 4 long-context decode with sinks -> GB/s), each with its own
roofline, end-to-end figure and CPU baseline; then the padded layout of the
prefill batch and the two decode workloads over the quantised KV cache
(``1_fp8kv``, ``4_fp8kv``: E4M3 codes with a float32 scale per (token, KV
head) row, bytes counted as read).  ``--workload N`` times only N;
``--kv-cache fp8 --workload N`` only N over the quantised cache.

Algorithmic work per step: every visible (query row, key) pair costs
4 * D flops per query head (QK^T and PV); bytes are each context token's K and
V rows once per KV head, the queries and outputs, the block tables and the
scatter's reads and writes.  The accessed KV exceeds the 126 MB L2 on the decode
workloads, so no flush is needed between steps.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload 1..4] [--no-cpu-baseline] [--layout packed|padded]
                    [--step two-call|fused] [--only-primary] [--kv-cache bf16|fp8]

Under torchrun (N > 1) every rank runs its own independent batch (requests are
independent units: weak scaling, no collective on the data path); timing is
the max over ranks.  ``--impl reference`` times the fp64 CPU oracle on the host
cores (rank 0 only) on a bounded per-step sample of the same workload.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "decode paged-attn KV GB/s (% HBM peak); varlen prefill TFLOP/s; tokens/s"
DEFAULT_WORKLOAD = 1
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0

# DRAM bytes (dram__bytes_read.sum + dram__bytes_write.sum) of one
# paged_decode_tc_kernel launch on workload 1, from an ncu capture (summary and
# command in profiles/paged_decode_tc_kernel__gqa_decode_bf16.md) of the
# kernel sources whose hash is recorded beside it: the files that define that
# kernel.  Reported as null once they change, until a new capture is taken.
NCU_TRAFFIC = {"sources_sha256": "79bb8d8ff887ab01c86416183e78737d3549c5267180b728c53ea436b1267083",
               "bytes_per_launch": 526288384 + 4950528, "workload": 1,
               "kernel": "paged_decode_tc_kernel"}
TRAFFIC_SOURCES = ("decode_tc.cuh", "decode_tc_d128.cu", "pa_common.cuh", "tc_common.cuh")


def kernel_sources_hash() -> str:
    """sha256 over the sources of the kernel whose traffic NCU_TRAFFIC holds."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "paged_kv_varlen_gb300", "csrc")
    for f in TRAFFIC_SOURCES:
        with open(os.path.join(csrc, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()


def dist_env():
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")),
            int(os.environ.get("LOCAL_RANK", "0")))


def max_over_ranks(value: float, world: int, device=None) -> float:
    """Max of a float over all ranks (identity when world == 1)."""
    if world <= 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ------------------------------------------------------------------ algorithmic work
def visible_keys(w) -> np.ndarray:
    """Keys each packed query row sees (bottom-right causal alignment)."""
    vis = np.empty(w.total_q, dtype=np.int64)
    for r in range(w.num_seqs):
        n, N = int(w.q_lens[r]), int(w.seq_lens[r])
        c0 = int(w.cu_seqlens_q[r])
        i = np.arange(n)
        vis[c0:c0 + n] = np.clip(N - n + i + 1, 0, N) if w.causal else N
    return vis


def algorithmic_work(w) -> dict:
    e = 2 if w.dtype == "bf16" else 4
    kv = w.kv_bytes_read()
    qo = 2 * w.total_q * w.num_q_heads * w.head_dim * e
    pages = int(((w.seq_lens + w.block_size - 1) // w.block_size).sum())
    meta = 4 * pages + 4 * (w.num_seqs * 2 + 1)
    scatter = 2 * 2 * w.total_q * w.num_kv_heads * w.head_dim * e + 8 * w.total_q
    flops = 4.0 * w.head_dim * w.num_q_heads * float(visible_keys(w).sum())
    return {"kv": kv, "attention_bytes": kv + qo + meta, "step_bytes": kv + qo + meta + scatter,
            "flops": flops, "tokens": w.total_q}


def workload_kind(w) -> str:
    if w.max_seqlen_q <= 1:
        return "decode"
    if int((w.q_lens == 1).sum()) == 0:
        return "prefill"
    return "mixed"


def metric_value(kind: str, work: dict, seconds: float, world: int):
    if kind == "decode":
        return world * work["step_bytes"] / seconds / 1e9, "GB/s"
    if kind == "prefill":
        return world * work["flops"] / seconds / 1e12, "TFLOP/s"
    return world * work["tokens"] / seconds, "tokens/s"


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), float(p["bf16_tflops"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, FALLBACK_BF16_TFLOPS, "fallback"


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons while running."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str):
        self.gpu_id = gpu_id
        self.proc = None
        self.lines = []
        self.t_on = self.t_off = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "50", "-i", self.gpu_id], stdout=subprocess.PIPE,
                stderr=subprocess.DEVNULL, text=True)
            threading.Thread(target=self._read, daemon=True).start()
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def mark_on(self):
        self.t_on = time.time()

    def mark_off(self):
        self.t_off = time.time()

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.1)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for t, line in self.lines:
            if self.t_on is None or not (self.t_on <= t <= self.t_off + 0.05):
                continue
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx = float(parts[2])
            except ValueError:
                continue
            for name, val in zip(names, parts[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(sm)}


def gpu_id_for(torch, device) -> str:
    try:
        u = str(torch.cuda.get_device_properties(device).uuid)
        return u if u.startswith("GPU-") else "GPU-" + u
    except Exception:
        vis = os.environ.get("CUDA_VISIBLE_DEVICES", "")
        return vis.split(",")[device] if vis else str(device)


# ------------------------------------------------------------------ CPU oracle
def prepare_oracle_pool(w):
    from oracle import oracle as orc
    w._kc_ref, w._vc_ref = orc.reshape_and_cache(w.new_k, w.new_v, w.key_cache, w.value_cache,
                                                 w.slot_mapping, w.block_size)
    w._vis = visible_keys(w)


def time_oracle(w, rows, nthreads):
    """Wall time of the fp64 oracle on the given query rows (pool holding this
    step's tokens)."""
    from oracle import oracle as orc
    t0 = time.perf_counter()
    orc.paged_attention(w.q, w._kc_ref, w._vc_ref, w.cu_seqlens_q, w.seq_lens_k, w.block_tables,
                        dtype=w.dtype, num_q_heads=w.num_q_heads, num_kv_heads=w.num_kv_heads,
                        head_dim=w.head_dim, block_size=w.block_size, scale=w.scale,
                        causal=w.causal, sinks=w.sinks, rows=rows, nthreads=nthreads)
    return time.perf_counter() - t0


def rows_work(w, rows) -> dict:
    """Work the oracle does for these rows, in the units of the GPU metric."""
    e = 2 if w.dtype == "bf16" else 4
    vis = w._vis[np.asarray(rows)]
    return {"step_bytes": float(vis.sum()) * w.num_kv_heads * w.head_dim * e * 2
                          + len(rows) * 2 * w.num_q_heads * w.head_dim * e,
            "flops": 4.0 * w.head_dim * w.num_q_heads * float(vis.sum()),
            "tokens": len(rows)}


def sample_rows(w, target_flops: float, seed: int = 0):
    """Rows whose oracle work is about `target_flops` (all rows if less)."""
    total = 4.0 * w.head_dim * w.num_q_heads * float(w._vis.sum())
    if total <= target_flops:
        return np.arange(w.total_q)
    rng = np.random.default_rng(seed)
    k = max(1, int(w.total_q * target_flops / total))
    return np.sort(rng.choice(w.total_q, size=k, replace=False))


def cpu_baseline(w, kind, budget_s=8.0, budget_1core_s=4.0):
    """The oracle as it stands, on samples of the workload's rows: on all host
    cores until about `budget_s` of wall time, and on one core until about
    `budget_1core_s`."""
    nthreads = os.cpu_count() or 1
    prepare_oracle_pool(w)

    def timed(target_flops, threads, budget):
        rows = sample_rows(w, target_flops)
        t, n = 0.0, 0
        while t < budget and n < 1000:
            t += time_oracle(w, rows, threads)
            n += 1
        work = {k: v * n for k, v in rows_work(w, rows).items()}
        value, unit = metric_value(kind, work, t, 1)
        return value, unit, (f"{n} pass(es) over {len(rows)} of {w.total_q} query rows "
                             f"(all heads), fp64 C oracle, {t:.1f} s wall")

    value, unit, sample = timed(4e9, nthreads, budget_s)
    v1, _, sample1 = timed(4e9 / max(1, nthreads), 1, budget_1core_s)
    return {"value": round(value, 6), "unit": unit, "cores": nthreads, "kind": "oracle",
            "sample": sample,
            "single_core": {"value": round(v1, 6), "unit": unit, "cores": 1, "sample": sample1}}


L2_BYTES = 126e6          # GB300 L2 (the device reports ~126 MB)
FLUSH_BYTES = 256 << 20   # written between timed steps when a step's data fits in L2


def needs_l2_flush(w, work) -> bool:
    """A step whose K/V, queries and outputs fit in L2 twice over would find
    them resident from the step before: such steps are timed with an L2 flush
    between them."""
    e = 2 if w.dtype == "bf16" else 4
    return work["kv"] + 2 * w.total_q * w.num_q_heads * w.head_dim * e < 2 * L2_BYTES


def workload_config(w, widx, P_used, layout, step, world, work, flushed=None):
    if flushed is None:
        flushed = needs_l2_flush(w, work)
    return {"workload": WORKLOAD_NAMES_CACHE[widx], "num_seqs": w.num_seqs,
            "total_q": w.total_q, "total_kv_tokens": int(w.seq_lens.sum()),
            "partition_size": P_used,
            "l2": (f"flushed between timed steps ({FLUSH_BYTES >> 20} MB write, outside the "
                   "per-step events)") if flushed
                  else "no flush: the data a step reads exceeds twice the 126 MB L2",
            "parallelism": f"independent batch per GPU x{world}",
            "layout": layout, "step": step}


WORKLOAD_NAMES_CACHE = {}


def run_reference(args, rank, world):
    if rank != 0:
        return 0
    from paged_kv_varlen_gb300 import workloads as wl
    WORKLOAD_NAMES_CACHE.update(wl.WORKLOAD_NAMES)
    widx = args.workload or DEFAULT_WORKLOAD
    w = wl.workload(widx)
    kind = workload_kind(w)
    prepare_oracle_pool(w)
    nthreads = os.cpu_count() or 1
    # per-step sample: one query row (all heads), cycling over the batch
    order = np.random.default_rng(1).permutation(w.total_q)
    pick = lambda i: order[i % len(order):i % len(order) + 1]  # noqa: E731
    for i in range(args.warmup):
        time_oracle(w, pick(i), nthreads)
    t_total = 0.0
    work = {"step_bytes": 0.0, "flops": 0.0, "tokens": 0}
    for i in range(args.steps):
        rows = pick(i)
        t_total += time_oracle(w, rows, nthreads)
        for k, v in rows_work(w, rows).items():
            work[k] += v
    value, unit = metric_value(kind, work, t_total, 1)
    sample = "one query row (all heads) per step, cycling over the batch; fp64 C oracle"
    P_used = w.partition_size
    fused = args.step == "fused"
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 6), "unit": unit,
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(1e3 * t_total / args.steps, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": workload_config(w, widx, P_used, args.layout,
                                  "pa_scatter_and_attend" if fused
                                  else "pa_reshape_and_cache + pa_varlen_attention", world,
                                  algorithmic_work(w)),
        "cpu_baseline": {"value": round(value, 6), "unit": unit, "cores": nthreads,
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": round(value, 6), "unit": unit, "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# ------------------------------------------------------------------ GPU arm
def measure(args, widx, rank, world, local, with_cpu_baseline):
    """Times one workload on this rank's GPU: the device-resident step, the
    end-to-end step through host buffers, the roofline of the attention call.
    Returns the record (the JSON line's fields)."""
    import torch
    from paged_kv_varlen_gb300 import binding as pa
    from paged_kv_varlen_gb300 import workloads as wl

    device = torch.device("cuda", local)
    w = wl.workload(widx)
    kind = workload_kind(w)
    work = algorithmic_work(w)
    w_useful = w
    if args.layout == "padded":
        # time the padded layout of the same batch; the work counted stays the
        # packed batch's useful work, so the metric is the effective rate
        w = wl.padded(w)

    def dev(a):
        if w.dtype == "bf16":
            return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(device).view(
                torch.bfloat16)
        return torch.from_numpy(np.ascontiguousarray(a)).to(device)

    q, kc, vc = dev(w.q), dev(w.key_cache), dev(w.value_cache)
    nk, nv = dev(w.new_k), dev(w.new_v)
    sm = torch.from_numpy(w.slot_mapping).to(device)
    cu = torch.from_numpy(w.cu_seqlens_q).to(device)
    sl = torch.from_numpy(w.seq_lens_k).to(device)
    bt = torch.from_numpy(w.block_tables).to(device)
    sk = torch.from_numpy(w.sinks).to(device) if w.sinks is not None else None
    out = torch.empty_like(q)
    P = w.partition_size
    ws_bytes = pa.pa_varlen_attention_workspace_size(w.num_seqs, w.max_seqlen_k, w.num_q_heads,
                                                     w.head_dim, P)
    ws = torch.empty(max(ws_bytes, 16), dtype=torch.uint8, device=device)
    stream = torch.cuda.current_stream(device)
    sms = torch.cuda.get_device_properties(device).multi_processor_count
    P_used = pa.pa_choose_partition_size(w.num_seqs, w.num_kv_heads, w.max_seqlen_k, P, sms)
    tc_decode = w.dtype == "bf16" and w.head_dim in (128, 256)
    # fused: one pa_scatter_and_attend call (the decode kernel overlaps the scatter)
    fused = args.step == "fused"
    launches_per_step = 1 + 1 + (1 if w.max_seqlen_q > 1 else 0) + (1 if P_used > 0 else 0)

    def scatter(k_in=nk, v_in=nv, s_in=sm):
        if not fused:
            pa.pa_reshape_and_cache(k_in, v_in, kc, vc, s_in, stream=stream)

    def attend(q_in=q, cu_in=cu, sl_in=sl, bt_in=bt, o=out, k_in=nk, v_in=nv, s_in=sm):
        if fused:
            pa.pa_scatter_and_attend(k_in, v_in, s_in, o, q_in, kc, vc, cu_in, sl_in, bt_in,
                                     max_seqlen_q=w.max_seqlen_q, max_seqlen_k=w.max_seqlen_k,
                                     scale=w.scale, sinks=sk, causal=w.causal, partition_size=P,
                                     workspace=ws, stream=stream)
            return
        pa.pa_varlen_attention(o, q_in, kc, vc, cu_in, sl_in, bt_in,
                               max_seqlen_q=w.max_seqlen_q, max_seqlen_k=w.max_seqlen_k,
                               scale=w.scale, sinks=sk, causal=w.causal, partition_size=P,
                               workspace=ws, stream=stream)

    def barrier():
        if world > 1:
            import torch.distributed as dist
            dist.barrier()

    steps = args.steps
    flush = needs_l2_flush(w, work)
    flush_buf = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=device) if flush else None
    # ---------------- device-resident timing
    for _ in range(args.warmup):
        scatter()
        attend()
    torch.cuda.synchronize()
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(steps)]
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    clocks = ClockSampler(gpu_id_for(torch, local))
    clocks.start()
    time.sleep(0.3)
    barrier()
    torch.cuda.synchronize()
    clocks.mark_on()
    start.record(stream)
    for i in range(steps):
        if flush:
            flush_buf.fill_(i & 255)   # evicts the previous step's data from L2
        ev[i][0].record(stream)
        scatter()
        ev[i][1].record(stream)
        attend()
        ev[i][2].record(stream)
    end.record(stream)
    end.synchronize()
    clocks.mark_off()
    barrier()
    torch.cuda.synchronize()
    clk = clocks.stop()
    assert pa.pa_device_error() == 0, "device error word set during the benchmark"
    if flush:   # the steps alone: from each step's first event to its last
        elapsed_s = max_over_ranks(sum(ev[i][0].elapsed_time(ev[i][2]) for i in range(steps))
                                   / 1e3, world, device)
    else:
        elapsed_s = max_over_ranks(start.elapsed_time(end) / 1e3, world, device)
    attn_ms = [ev[i][1].elapsed_time(ev[i][2]) for i in range(steps)]
    attn_avg_s = max_over_ranks(sum(attn_ms) / len(attn_ms) / 1e3, world, device)
    step_s = elapsed_s / steps
    value, unit = metric_value(kind, work, step_s, world)

    # ---------------- end to end through the public API with host buffers: the
    # step's inputs packed in one pinned staging buffer (one host-to-device
    # copy), the output read back
    from paged_kv_varlen_gb300.staging import StepStaging
    stage = StepStaging({"q": q, "new_k": nk, "new_v": nv, "slot_mapping": sm,
                         "cu_seqlens_q": cu, "seq_lens_k": sl, "block_tables": bt}, device)
    for name, t in (("q", q), ("new_k", nk), ("new_v", nv), ("slot_mapping", sm),
                    ("cu_seqlens_q", cu), ("seq_lens_k", sl), ("block_tables", bt)):
        stage.host[name].copy_(t.cpu())
    dv = stage.dev
    h_out = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    h2d = stage.nbytes
    d2h = h_out.numel() * h_out.element_size()

    def e2e_step():
        stage.upload()
        scatter(dv["new_k"], dv["new_v"], dv["slot_mapping"])
        attend(dv["q"], dv["cu_seqlens_q"], dv["seq_lens_k"], dv["block_tables"],
               k_in=dv["new_k"], v_in=dv["new_v"], s_in=dv["slot_mapping"])
        h_out.copy_(out, non_blocking=True)

    for _ in range(args.warmup):
        e2e_step()
    torch.cuda.synchronize()
    barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(steps):
        e2e_step()
    e1.record(stream)
    e1.synchronize()
    barrier()
    assert pa.pa_device_error() == 0, "device error word set during the end-to-end steps"
    e2e_s = max_over_ranks(e0.elapsed_time(e1) / 1e3, world, device) / steps
    e2e_value, _ = metric_value(kind, work, e2e_s, world)

    # ---------------- roofline of the dominant launch (the attention call; with
    # the fused step it also moves the scatter's bytes)
    hbm, bf16, peak_kind = measured_peaks()
    call_bytes = work["step_bytes"] if fused else work["attention_bytes"]
    t_bw = call_bytes / (hbm * 1e9)
    t_fl = work["flops"] / (bf16 * 1e12)
    traffic = (NCU_TRAFFIC["bytes_per_launch"]
               if NCU_TRAFFIC["sources_sha256"] == kernel_sources_hash()
               and NCU_TRAFFIC.get("workload") == widx else None)
    if kind == "decode" or (kind == "mixed" and t_bw >= t_fl):
        roof = {"bound": "hbm", "achieved": round(call_bytes / attn_avg_s / 1e9, 2),
                "peak": hbm, "unit": "GB/s"}
    else:
        roof = {"bound": "tensor", "achieved": round(work["flops"] / attn_avg_s / 1e12, 2),
                "peak": bf16, "unit": "TFLOP/s"}
    roof["frac"] = round(roof["achieved"] / roof["peak"], 4)
    roof["traffic"] = traffic
    if traffic is not None:
        roof["traffic_kernel"] = NCU_TRAFFIC["kernel"]
    dec = "paged_decode_tc_kernel" if tc_decode else "paged_decode_kernel"
    if fused:
        dec = "scatter_rows_kernel + " + dec
    roof["kernel"] = {"decode": f"{dec} + split_reduce_kernel",
                      "prefill": "paged_prefill_tc_kernel",
                      "mixed": f"{dec} + paged_prefill_tc_kernel + split_reduce_kernel"
                      }[kind] + (" (one pa_scatter_and_attend call)" if fused
                                 else " (one attention call)")
    roof["peak_source"] = (f"{peak_kind} (MEASURED_PEAKS.json "
                           f"{'hbm_gbs' if roof['bound'] == 'hbm' else 'bf16_tflops'})"
                           if peak_kind == "measured" else "fallback")
    roof["avg_launch_us"] = round(attn_avg_s * 1e6, 3)
    if kind == "mixed":
        # the step needs both HBM (decode and verify rows) and the tensor cores
        # (prefill chunks): its roofline time is the larger of the two
        roof["roofline_time_us"] = round(1e6 * max(t_bw, t_fl), 2)
        roof["t_bw_us"] = round(1e6 * t_bw, 2)
        roof["t_flop_us"] = round(1e6 * t_fl, 2)
        roof["frac_of_max_roofline"] = round(max(t_bw, t_fl) / attn_avg_s, 4)

    rec = {
        "metric": METRIC, "value": round(value, 3), "unit": unit, "n_gpus": world,
        "steps": steps, "warmup": args.warmup, "ms_per_step": round(1e3 * step_s, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": w.dtype,
        "data": "synthetic (seeded N(0,1) Q/K/V)",
        "config": workload_config(w_useful, widx, P_used, args.layout,
                                  "pa_scatter_and_attend" if fused
                                  else "pa_reshape_and_cache + pa_varlen_attention", world, work,
                                  flushed=flush),
        "kv_gbs": round(world * work["step_bytes"] / step_s / 1e9, 2),
        "tflops": round(world * work["flops"] / step_s / 1e12, 3),
        "tokens_per_s": round(world * w_useful.total_q / step_s, 1),
        "roofline": roof,
        "e2e": {"value": round(e2e_value, 3), "unit": unit, "h2d_bytes_per_step": int(h2d),
                "d2h_bytes_per_step": int(d2h), "ms_per_step": round(1e3 * e2e_s, 5)},
        "gpu_launches": int(launches_per_step * steps),
        "clocks": clk,
    }
    if rank == 0 and world == 1 and with_cpu_baseline:
        rec["cpu_baseline"] = cpu_baseline(w_useful, kind)
    del q, kc, vc, nk, nv, out, ws, stage, flush_buf
    torch.cuda.empty_cache()
    return rec


def fp8kv_work(w) -> dict:
    """Algorithmic work of a step over the quantised cache: every context
    token's K and V rows once per KV head as D one-byte codes plus a float32
    scale; bf16 queries and outputs; the quantising scatter reads the new bf16
    rows and writes their codes and scales."""
    Hkv, D = w.num_kv_heads, w.head_dim
    kv = int(w.seq_lens.sum()) * Hkv * (D + 4) * 2
    qo = 2 * w.total_q * w.num_q_heads * D * 2
    pages = int(((w.seq_lens + w.block_size - 1) // w.block_size).sum())
    meta = 4 * pages + 4 * (w.num_seqs * 2 + 1)
    scatter = 2 * w.total_q * Hkv * (2 * D + D + 4) + 8 * w.total_q
    flops = 4.0 * D * w.num_q_heads * float(visible_keys(w).sum())
    return {"kv": kv, "attention_bytes": kv + qo + meta, "step_bytes": kv + qo + meta + scatter,
            "flops": flops, "tokens": w.total_q}


def measure_fp8kv(args, widx, rank, world, local):
    """Times a decode workload over the quantised KV cache (E4M3 codes with a
    float32 scale per (token, KV head) row): one step = the quantising scatter
    of the step's new rows, then attention over the quantised pool.  The pool
    is quantised once, untimed, from the workload's bf16 pool."""
    import torch
    from paged_kv_varlen_gb300 import binding as pa
    from paged_kv_varlen_gb300 import workloads as wl

    device = torch.device("cuda", local)
    w = wl.workload(widx)
    assert workload_kind(w) == "decode" and w.dtype == "bf16"
    work = fp8kv_work(w)
    nb, bs, Hkv, D = w.num_blocks, w.block_size, w.num_kv_heads, w.head_dim

    def dev(a):
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(device).view(
            torch.bfloat16)

    q, nk, nv = dev(w.q), dev(w.new_k), dev(w.new_v)
    kcodes = torch.empty((nb, bs, Hkv, D), dtype=torch.uint8, device=device)
    vcodes = torch.empty_like(kcodes)
    kscales = torch.empty((nb, bs, Hkv), dtype=torch.float32, device=device)
    vscales = torch.empty_like(kscales)
    all_slots = torch.arange(nb * bs, dtype=torch.int64, device=device)
    stream = torch.cuda.current_stream(device)
    kc = dev(w.key_cache).view(nb * bs, Hkv, D)
    vc = dev(w.value_cache).view(nb * bs, Hkv, D)
    pa.pa_reshape_and_cache_fp8(kc, vc, kcodes, vcodes, kscales, vscales, all_slots,
                                stream=stream)
    del kc, vc, all_slots
    sm = torch.from_numpy(w.slot_mapping).to(device)
    cu = torch.from_numpy(w.cu_seqlens_q).to(device)
    sl = torch.from_numpy(w.seq_lens_k).to(device)
    bt = torch.from_numpy(w.block_tables).to(device)
    sk = torch.from_numpy(w.sinks).to(device) if w.sinks is not None else None
    out = torch.empty_like(q)
    P = w.partition_size
    ws_bytes = pa.pa_varlen_attention_workspace_size(w.num_seqs, w.max_seqlen_k, w.num_q_heads,
                                                     D, P)
    ws = torch.empty(max(ws_bytes, 16), dtype=torch.uint8, device=device)
    sms = torch.cuda.get_device_properties(device).multi_processor_count
    P_used = pa.pa_choose_partition_size(w.num_seqs, Hkv, w.max_seqlen_k, P, sms)
    launches_per_step = 2 + (1 if P_used > 0 else 0)

    def step(q_in=q, k_in=nk, v_in=nv, s_in=sm, cu_in=cu, sl_in=sl, bt_in=bt, events=None):
        pa.pa_reshape_and_cache_fp8(k_in, v_in, kcodes, vcodes, kscales, vscales, s_in,
                                    stream=stream)
        if events is not None:
            events[0].record(stream)
        pa.pa_varlen_attention_fp8kv(out, q_in, kcodes, vcodes, kscales, vscales, cu_in, sl_in,
                                     bt_in, max_seqlen_q=w.max_seqlen_q,
                                     max_seqlen_k=w.max_seqlen_k, scale=w.scale, sinks=sk,
                                     causal=w.causal, partition_size=P, workspace=ws,
                                     stream=stream)
        if events is not None:
            events[1].record(stream)

    def barrier():
        if world > 1:
            import torch.distributed as dist
            dist.barrier()

    steps = args.steps
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(steps)]
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    clocks = ClockSampler(gpu_id_for(torch, local))
    clocks.start()
    time.sleep(0.3)
    barrier()
    torch.cuda.synchronize()
    clocks.mark_on()
    start.record(stream)
    for i in range(steps):
        step(events=ev[i])
    end.record(stream)
    end.synchronize()
    clocks.mark_off()
    barrier()
    torch.cuda.synchronize()
    clk = clocks.stop()
    assert pa.pa_device_error() == 0, "device error word set during the benchmark"
    step_s = max_over_ranks(start.elapsed_time(end) / 1e3, world, device) / steps
    attn_s = max_over_ranks(sum(e[0].elapsed_time(e[1]) for e in ev) / steps / 1e3, world,
                            device)
    value, unit = metric_value("decode", work, step_s, world)

    from paged_kv_varlen_gb300.staging import StepStaging
    stage = StepStaging({"q": q, "new_k": nk, "new_v": nv, "slot_mapping": sm,
                         "cu_seqlens_q": cu, "seq_lens_k": sl, "block_tables": bt}, device)
    for name, t in (("q", q), ("new_k", nk), ("new_v", nv), ("slot_mapping", sm),
                    ("cu_seqlens_q", cu), ("seq_lens_k", sl), ("block_tables", bt)):
        stage.host[name].copy_(t.cpu())
    dv = stage.dev
    h_out = torch.empty(out.shape, dtype=out.dtype).pin_memory()

    def e2e_step():
        stage.upload()
        step(dv["q"], dv["new_k"], dv["new_v"], dv["slot_mapping"], dv["cu_seqlens_q"],
             dv["seq_lens_k"], dv["block_tables"])
        h_out.copy_(out, non_blocking=True)

    for _ in range(args.warmup):
        e2e_step()
    torch.cuda.synchronize()
    barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(steps):
        e2e_step()
    e1.record(stream)
    e1.synchronize()
    barrier()
    assert pa.pa_device_error() == 0, "device error word set during the end-to-end steps"
    e2e_s = max_over_ranks(e0.elapsed_time(e1) / 1e3, world, device) / steps
    e2e_value, _ = metric_value("decode", work, e2e_s, world)

    hbm, _, peak_kind = measured_peaks()
    achieved = work["attention_bytes"] / attn_s / 1e9
    roof = {"bound": "hbm", "achieved": round(achieved, 2), "peak": hbm, "unit": "GB/s",
            "frac": round(achieved / hbm, 4), "traffic": None,
            "kernel": "paged_decode_tc_fp8_kernel + split_reduce_kernel (one attention call)",
            "peak_source": (f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs)"
                            if peak_kind == "measured" else "fallback"),
            "avg_launch_us": round(attn_s * 1e6, 3)}
    cfg = workload_config(w, widx, P_used, "packed",
                          "pa_reshape_and_cache_fp8 + pa_varlen_attention_fp8kv", world, work,
                          flushed=False)
    cfg["kv_cache"] = "E4M3 codes + float32 scale per (token, KV head) row"
    rec = {"value": round(value, 3), "unit": unit, "ms_per_step": round(1e3 * step_s, 5),
           "dtype": "bf16 q/out, e4m3 K/V codes, f32 accumulation", "config": cfg,
           "kv_gbs": round(world * work["step_bytes"] / step_s / 1e9, 2),
           "tokens_per_s": round(world * w.total_q / step_s, 1), "roofline": roof,
           "e2e": {"value": round(e2e_value, 3), "unit": unit,
                   "h2d_bytes_per_step": int(stage.nbytes),
                   "d2h_bytes_per_step": int(h_out.numel() * h_out.element_size()),
                   "ms_per_step": round(1e3 * e2e_s, 5)},
           "gpu_launches": int(launches_per_step * steps), "clocks": clk}
    del q, nk, nv, kcodes, vcodes, kscales, vscales, out, ws, stage
    torch.cuda.empty_cache()
    return rec


def run_ours(args, rank, world, local):
    import torch
    from paged_kv_varlen_gb300 import workloads as wl

    WORKLOAD_NAMES_CACHE.update(wl.WORKLOAD_NAMES)
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=device)

    primary = args.workload or DEFAULT_WORKLOAD
    with_cpu = not args.no_cpu_baseline
    if args.kv_cache == "fp8":
        rec = measure_fp8kv(args, primary, rank, world, local)
        rec.update({"metric": METRIC, "n_gpus": world, "steps": args.steps,
                    "warmup": args.warmup, "higher_is_better": True, "scaling": "weak",
                    "vs_baseline": None, "data": "synthetic (seeded N(0,1) Q/K/V)"})
        if rank == 0:
            print(json.dumps(rec), flush=True)
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()
        return 0
    line = measure(args, primary, rank, world, local, with_cpu)
    if args.workload is None and not args.only_primary:
        subs = {}
        keep = ("value", "unit", "ms_per_step", "dtype", "config", "kv_gbs", "tflops",
                "tokens_per_s", "roofline", "e2e", "gpu_launches", "clocks", "cpu_baseline")
        for widx in (2, 3, 4):
            rec = measure(args, widx, rank, world, local, with_cpu)
            subs[str(widx)] = {k: rec[k] for k in keep if k in rec}
        # the prefill batch laid out padded ([B, T_max]: every request padded to
        # the longest), useful work counted: what packing is worth on this mix
        padded_args = argparse.Namespace(**vars(args))
        padded_args.layout = "padded"
        padded_args.steps = min(args.steps, 500)
        rec = measure(padded_args, 2, rank, world, local, False)
        subs["2_padded"] = {k: rec[k] for k in keep if k in rec}
        # the decode batches over the quantised KV cache
        for widx in (1, 4):
            subs[f"{widx}_fp8kv"] = measure_fp8kv(args, widx, rank, world, local)
        line["workloads"] = subs
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=5000)
    ap.add_argument("--warmup", type=int, default=50)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", type=int, choices=[1, 2, 3, 4], default=None,
                    help="time only this workload (default: 1 as the headline, plus 2-4 "
                         "as sub-records)")
    ap.add_argument("--only-primary", action="store_true",
                    help="time only the headline workload")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--layout", choices=["packed", "padded"], default="packed",
                    help="padded: the same batch padded to [B, T_max] (useful work counted)")
    ap.add_argument("--step", choices=["fused", "two-call"], default="fused",
                    help="fused: one pa_scatter_and_attend call per step; two-call: "
                         "pa_reshape_and_cache then pa_varlen_attention")
    ap.add_argument("--kv-cache", choices=["bf16", "fp8"], default="bf16",
                    help="fp8: time only the decode workload (1 or 4) over the quantised "
                         "cache (E4M3 codes + a float32 scale per row)")
    args = ap.parse_args(argv)
    if args.kv_cache == "fp8" and (args.workload or DEFAULT_WORKLOAD) not in (1, 4):
        ap.error("--kv-cache fp8 times the decode workloads 1 and 4 only")
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    rank, world, local = dist_env()
    if args.impl == "reference":
        return run_reference(args, rank, world)
    from paged_kv_varlen_gb300 import build
    build.build_library()
    return run_ours(args, rank, world, local)


if __name__ == "__main__":
    sys.exit(main())
