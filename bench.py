"""Benchmark of the paged varlen attention hot path on GB300.

One step = one pass of the whole hot path over one batch: the KV scatter of
this step's tokens (pa_reshape_and_cache), then attention over the packed
query rows and paged K/V (pa_varlen_attention: split-KV decode kernel + the
shared reduce).  Default workload: the GQA decode batch -- 32 requests with
contexts U[512, 8192], (H_q, H_kv, D) = (32, 8, 128), bf16, block size 16,
40k-page shuffled pool, split-KV partition 512.

Metric: decode KV GB/s = algorithmic bytes per step (each context token's K
and V rows once per KV head, queries, outputs, block tables, the scatter's
reads and writes) / step time.  The accessed KV (~570 MB) exceeds the 126 MB
L2, so no flush is needed between steps.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Under torchrun (N > 1) every rank runs its own independent batch (requests are
independent units: weak scaling, no collective on the data path); timing is
the max over ranks.  ``--impl reference`` times the fp64 CPU oracle on the
host cores (rank 0 only) on a bounded per-step sample of the same workload.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
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
WORKLOAD_INDEX = 1
FALLBACK_HBM_GBS = 6800.0

# dram__bytes_read.sum + dram__bytes_write.sum per attention call (decode kernel
# + reduce) from an ncu capture, valid only for the kernel sources whose hash
# is recorded beside it; null otherwise.
NCU_TRAFFIC = {"sources_sha256": None, "bytes_per_launch": None}


def kernel_sources_hash() -> str:
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "paged_kv_varlen_gb300", "csrc")
    for f in ("decode_kernel.cuh", "pa_common.cuh", "reduce.cu"):
        with open(os.path.join(csrc, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def max_over_ranks(value: float, world: int, device=None) -> float:
    """Max of a float over all ranks (identity when world == 1)."""
    if world <= 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def algorithmic_bytes(w) -> dict:
    """Bytes one step must move at minimum (per the layouts of the ABI)."""
    e = 2 if w.dtype == "bf16" else 4
    kv = w.kv_bytes_read()
    qo = 2 * w.total_q * w.num_q_heads * w.head_dim * e
    pages = int(((w.seq_lens + w.block_size - 1) // w.block_size).sum())
    meta = 4 * pages + 4 * (w.num_seqs * 2 + 1)
    scatter = 2 * 2 * w.total_q * w.num_kv_heads * w.head_dim * e + 8 * w.total_q
    return {"kv": kv, "attention": kv + qo + meta, "step": kv + qo + meta + scatter}


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


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
            self.reader = threading.Thread(target=self._read, daemon=True)
            self.reader.start()
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
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": mx, "reasons": sorted(reasons), "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


def gpu_id_for(torch, device) -> str:
    try:
        u = str(torch.cuda.get_device_properties(device).uuid)
        return u if u.startswith("GPU-") else "GPU-" + u
    except Exception:
        vis = os.environ.get("CUDA_VISIBLE_DEVICES", "")
        return vis.split(",")[device] if vis else str(device)


# ------------------------------------------------------------------ CPU oracle
def time_oracle(w, rows, nthreads):
    """Wall time of the fp64 oracle on the given decode rows (pool already
    holding this step's tokens)."""
    from oracle import oracle as orc
    t0 = time.perf_counter()
    orc.paged_attention(w.q, w._kc_ref, w._vc_ref, w.cu_seqlens_q, w.seq_lens_k, w.block_tables,
                        dtype=w.dtype, num_q_heads=w.num_q_heads, num_kv_heads=w.num_kv_heads,
                        head_dim=w.head_dim, block_size=w.block_size, scale=w.scale,
                        causal=w.causal, sinks=w.sinks, rows=rows, nthreads=nthreads)
    return time.perf_counter() - t0


def row_bytes(w, rows):
    e = 2 if w.dtype == "bf16" else 4
    total = 0
    for row in rows:
        r = int(np.searchsorted(w.cu_seqlens_q, row, side="right") - 1)
        total += int(w.seq_lens_k[r]) * w.num_kv_heads * w.head_dim * e * 2
        total += 2 * w.num_q_heads * w.head_dim * e
    return total


def prepare_oracle_pool(w):
    from oracle import oracle as orc
    w._kc_ref, w._vc_ref = orc.reshape_and_cache(w.new_k, w.new_v, w.key_cache, w.value_cache,
                                                 w.slot_mapping, w.block_size)


def cpu_baseline(w, budget_s=12.0):
    """The oracle as it stands on all host cores, on whole batches of the
    workload until about `budget_s` of CPU work."""
    nthreads = os.cpu_count() or 1
    prepare_oracle_pool(w)
    rows = np.arange(w.total_q)
    t, n = 0.0, 0
    while t < budget_s and n < 1000:
        t += time_oracle(w, rows, nthreads)
        n += 1
    gbs = n * row_bytes(w, rows) / t / 1e9
    return {"value": round(gbs, 4), "unit": "GB/s", "cores": nthreads, "kind": "oracle",
            "sample": f"{n} full batch(es) of the workload ({w.total_q} decode rows, all heads), "
                      f"fp64 C oracle, {t:.1f} s wall"}


def run_reference(args, rank, world):
    if rank != 0:
        return 0
    from paged_kv_varlen_gb300 import workloads as wl
    w = wl.workload(WORKLOAD_INDEX)
    prepare_oracle_pool(w)
    nthreads = os.cpu_count() or 1
    # per-step sample: one decode row (all heads), cycling over the batch
    order = np.arange(w.total_q)
    for i in range(args.warmup):
        time_oracle(w, order[i % len(order):i % len(order) + 1], nthreads)
    t_total, b_total = 0.0, 0
    for i in range(args.steps):
        rows = order[i % len(order):i % len(order) + 1]
        t_total += time_oracle(w, rows, nthreads)
        b_total += row_bytes(w, rows)
    value = b_total / t_total / 1e9
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(1e3 * t_total / args.steps, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": wl.WORKLOAD_NAMES[WORKLOAD_INDEX],
                   "sample": "one decode row (all 32 query heads) per step"},
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": nthreads,
                         "kind": "oracle",
                         "sample": "one decode row (all heads) per step, cycling over the "
                                   "32-row batch; fp64 C oracle"},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# ------------------------------------------------------------------ GPU arm
def run_ours(args, rank, world, local):
    import torch
    from paged_kv_varlen_gb300 import binding as pa
    from paged_kv_varlen_gb300 import workloads as wl

    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=device)

    w = wl.workload(WORKLOAD_INDEX)
    nbytes = algorithmic_bytes(w)

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
    out = torch.empty_like(q)
    P = w.partition_size
    ws_bytes = pa.pa_varlen_attention_workspace_size(w.num_seqs, w.max_seqlen_k, w.num_q_heads,
                                                     w.head_dim, P)
    ws = torch.empty(max(ws_bytes, 16), dtype=torch.uint8, device=device)
    stream = torch.cuda.current_stream(device)
    sms = torch.cuda.get_device_properties(device).multi_processor_count
    P_used = pa.pa_choose_partition_size(w.num_seqs, w.num_kv_heads, w.max_seqlen_k, P, sms)
    launches_per_step = 1 + 1 + (1 if w.max_seqlen_q > 1 else 0) + (1 if P_used > 0 else 0)

    def scatter(k_in=nk, v_in=nv, s_in=sm):
        pa.pa_reshape_and_cache(k_in, v_in, kc, vc, s_in, stream=stream)

    def attend(q_in=q, cu_in=cu, sl_in=sl, bt_in=bt, o=out):
        pa.pa_varlen_attention(o, q_in, kc, vc, cu_in, sl_in, bt_in,
                               max_seqlen_q=w.max_seqlen_q, max_seqlen_k=w.max_seqlen_k,
                               scale=w.scale, sinks=None, causal=w.causal, partition_size=P,
                               workspace=ws, stream=stream)

    def barrier():
        if world > 1:
            import torch.distributed as dist
            dist.barrier()

    # ---------------- device-resident timing
    for _ in range(args.warmup):
        scatter()
        attend()
    torch.cuda.synchronize()
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    clocks = ClockSampler(gpu_id_for(torch, local))
    clocks.start()
    time.sleep(0.3)
    barrier()
    torch.cuda.synchronize()
    clocks.mark_on()
    start.record(stream)
    for i in range(args.steps):
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
    elapsed_s = max_over_ranks(start.elapsed_time(end) / 1e3, world, device)
    attn_ms = [ev[i][1].elapsed_time(ev[i][2]) for i in range(args.steps)]
    attn_avg_s = max_over_ranks(sum(attn_ms) / len(attn_ms) / 1e3, world, device)
    step_s = elapsed_s / args.steps
    value = world * nbytes["step"] / step_s / 1e9

    # ---------------- end to end through the public API with host buffers
    pin = lambda t: t.cpu().pin_memory()  # noqa: E731
    h_q, h_nk, h_nv, h_sm = pin(q), pin(nk), pin(nv), pin(sm)
    h_cu, h_sl, h_bt = pin(cu), pin(sl), pin(bt)
    h_out = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    d_q, d_nk, d_nv, d_sm = (torch.empty_like(t) for t in (q, nk, nv, sm))
    d_cu, d_sl, d_bt = (torch.empty_like(t) for t in (cu, sl, bt))
    h2d = sum(t.numel() * t.element_size() for t in (h_q, h_nk, h_nv, h_sm, h_cu, h_sl, h_bt))
    d2h = h_out.numel() * h_out.element_size()

    def e2e_step():
        for d, h in ((d_q, h_q), (d_nk, h_nk), (d_nv, h_nv), (d_sm, h_sm), (d_cu, h_cu),
                     (d_sl, h_sl), (d_bt, h_bt)):
            d.copy_(h, non_blocking=True)
        scatter(d_nk, d_nv, d_sm)
        attend(d_q, d_cu, d_sl, d_bt)
        h_out.copy_(out, non_blocking=True)

    for _ in range(args.warmup):
        e2e_step()
    torch.cuda.synchronize()
    barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.steps):
        e2e_step()
    e1.record(stream)
    e1.synchronize()
    barrier()
    e2e_s = max_over_ranks(e0.elapsed_time(e1) / 1e3, world, device) / args.steps
    e2e_value = world * nbytes["step"] / e2e_s / 1e9

    # ---------------- roofline of the dominant launch (decode kernel + reduce)
    peak, peak_kind = measured_peaks()
    achieved = nbytes["attention"] / attn_avg_s / 1e9
    traffic = None
    if NCU_TRAFFIC["sources_sha256"] == kernel_sources_hash():
        traffic = NCU_TRAFFIC["bytes_per_launch"]

    line = {
        "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(1e3 * step_s, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded N(0,1) Q/K/V, bf16)",
        "config": {"workload": wl.WORKLOAD_NAMES[WORKLOAD_INDEX], "num_seqs": w.num_seqs,
                   "total_kv_tokens": int(w.seq_lens.sum()), "partition_size": P_used,
                   "l2": "inputs larger than L2 (~570 MB of KV per step vs 126 MB L2); no flush",
                   "parallelism": f"independent batch per GPU x{world}"},
        "tokens_per_s": round(world * w.total_q / step_s, 1),
        "roofline": {"bound": "hbm", "achieved": round(achieved, 2), "peak": peak,
                     "unit": "GB/s", "frac": round(achieved / peak, 4), "traffic": traffic,
                     "kernel": "paged_decode_kernel + split_reduce_kernel (one attention call)",
                     "peak_source": f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs)"
                                    if peak_kind == "measured" else "fallback 6.8 TB/s",
                     "avg_launch_us": round(attn_avg_s * 1e6, 3)},
        "e2e": {"value": round(e2e_value, 2), "unit": "GB/s", "h2d_bytes_per_step": int(h2d),
                "d2h_bytes_per_step": int(d2h), "ms_per_step": round(1e3 * e2e_s, 5)},
        "gpu_launches": int(launches_per_step * args.steps),
        "clocks": clk,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(w)
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
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args(argv)
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
