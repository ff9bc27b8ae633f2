"""GPU parity on the edges of the method: padding and out-of-pool slots in the
scatter, non-causal multi-query rows and rows that see no key on the
tensor-core kernel, and the one-call step against the oracle.

Tolerances as everywhere: fp32 max abs 1e-5; bf16 max abs 2e-2, mean 2e-3;
the scatter bit for bit over the whole pool.
"""
import numpy as np
import pytest
import torch

from harness import DeviceWorkload, assert_close, check_scatter, check_step, dev_bits_t, from_dev
from oracle import oracle as orc
from oracle.oracle import attention_of
from paged_kv_varlen_gb300 import binding as pa
from paged_kv_varlen_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


# ---------------------------------------------------------------- scatter
@pytest.mark.parametrize("dtype", [wl.F32, wl.BF16])
@pytest.mark.parametrize("D", [64, 128, 256])
def test_scatter_skips_padding_and_out_of_pool_slots(dtype, D):
    """Negative slots are padding tokens and slots at or past num_blocks *
    block_size lie outside the pool: both are skipped, and no other slot of the
    pool changes (reading R5; pptc.cn section 3: memory no token maps to is
    never touched)."""
    w = wl.random_small(120 + D, dtype=dtype, num_seqs=6, num_q_heads=8, num_kv_heads=2,
                        head_dim=D, max_prior=60, max_q=9)
    sm = w.slot_mapping.copy()
    nslots = w.num_blocks * w.block_size
    T = len(sm)
    assert T >= 8
    sm[0] = -1
    sm[T // 3] = -7
    sm[T // 2] = nslots                  # first slot past the pool
    sm[T - 2] = nslots + 12345
    sm[T - 1] = 1 << 40
    dw = DeviceWorkload(w)
    check_scatter(dw, slot_mapping=sm)
    torch.cuda.synchronize()
    assert pa.pa_device_error() == 0


def test_scatter_full_pool_on_every_full_size_workload():
    """The whole pool after the scatter, for the workloads whose steps write
    many pages (the prefill's 6,000 tokens, the mixed step's 4,000)."""
    for widx in (2, 3):
        dw = DeviceWorkload(wl.workload(widx))
        check_scatter(dw)
    torch.cuda.synchronize()
    assert pa.pa_device_error() == 0


# ---------------------------------------------------------------- tensor-core rows
NONCAUSAL = [(D, Hq, Hkv) for D in (64, 128, 256) for (Hq, Hkv) in ((8, 2), (8, 1), (3, 3))]


@pytest.mark.parametrize("D,Hq,Hkv", NONCAUSAL, ids=[f"D{d}-{a}x{b}" for d, a, b in NONCAUSAL])
def test_non_causal_multi_query_rows_bf16(D, Hq, Hkv):
    """causal = 0 on the tcgen05 multi-query kernel: every row sees all N keys
    (reading R7), verify windows and chunks up to 40 rows spanning several
    query blocks, with a ragged last key tile."""
    w = wl.random_small(140 + D + Hq, dtype=wl.BF16, num_seqs=5, num_q_heads=Hq,
                        num_kv_heads=Hkv, head_dim=D, max_prior=300, max_q=40, causal=False,
                        with_sinks=(Hkv == 2))
    check_step(w)


@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("D", [64, 128, 256])
def test_more_query_rows_than_keys_bf16(D, causal):
    """Requests with n query rows but only N < n keys.  Causal row i sees keys
    j <= N - n + i, so the first n - N rows see none and are zeros (reading
    R6); a request with N = 0 is all zeros; non-causal rows see all N."""
    w = wl.random_small(160 + D, dtype=wl.BF16, num_seqs=5, num_q_heads=8, num_kv_heads=2,
                        head_dim=D, max_prior=0, max_q=70, causal=causal, with_sinks=True)
    N = w.seq_lens_k.copy()
    n = w.q_lens
    N[0] = 0
    for r in range(1, w.num_seqs):
        N[r] = max(0, int(n[r]) - 1 - 7 * r) if n[r] > 1 else N[r]
    dw = DeviceWorkload(w)
    kc_ref, vc_ref = check_scatter(dw)
    dw.seq_lens_k.copy_(torch.from_numpy(N.astype(np.int32)))
    dw.attention()
    torch.cuda.synchronize()
    assert pa.pa_device_error() == 0
    w.seq_lens_k = N.astype(np.int32)
    ref = attention_of(w, key_cache=kc_ref, value_cache=vc_ref)
    got = from_dev(dw.out)
    assert_close(got, ref, w.dtype, f"n > N, causal={causal}")
    if causal:
        for r in range(w.num_seqs):
            c0 = int(w.cu_seqlens_q[r])
            blind = int(n[r]) - int(N[r])
            if blind > 0:
                assert torch.count_nonzero(dw.out[c0:c0 + blind]) == 0


# ---------------------------------------------------------------- one-call step vs the oracle
ONECALL = [
    ("decode-bf16-D128", lambda: wl.random_small(91, dtype=wl.BF16, num_seqs=6, head_dim=128,
                                                  num_q_heads=8, num_kv_heads=2, max_prior=1400,
                                                  max_q=1, with_sinks=True)),
    ("mixed-bf16-D128", lambda: wl.random_small(92, dtype=wl.BF16, num_seqs=7, head_dim=128,
                                                 num_q_heads=8, num_kv_heads=2, max_prior=900,
                                                 max_q=40)),
    ("mixed-bf16-D256", lambda: wl.random_small(93, dtype=wl.BF16, num_seqs=5, head_dim=256,
                                                 num_q_heads=6, num_kv_heads=1, max_prior=700,
                                                 max_q=20, block_size=32)),
    ("decode-f32-D128", lambda: wl.random_small(94, dtype=wl.F32, num_seqs=4, head_dim=128,
                                                 max_prior=500, max_q=1)),
    ("mixed-bf16-D64", lambda: wl.random_small(95, dtype=wl.BF16, num_seqs=4, head_dim=64,
                                                max_prior=300, max_q=9)),
]


def _fused_vs_oracle(w, rows=None, partition_size=None):
    dw = DeviceWorkload(w)
    kc_before = dev_bits_t(dw.key_cache).clone()
    dw.fused_step(partition_size=partition_size)
    torch.cuda.synchronize()
    assert pa.pa_device_error() == 0
    kc_ref, vc_ref = orc.reshape_and_cache(w.new_k, w.new_v, w.key_cache, w.value_cache,
                                           w.slot_mapping, w.block_size)
    pages = np.unique(w.slot_mapping[w.slot_mapping >= 0] // w.block_size)
    view = np.uint16 if w.dtype == wl.BF16 else np.uint32
    pidx = torch.from_numpy(pages).cuda()
    assert np.array_equal(dev_bits_t(dw.key_cache[pidx]).cpu().numpy().view(view),
                          kc_ref[pages].view(view))
    assert np.array_equal(dev_bits_t(dw.value_cache[pidx]).cpu().numpy().view(view),
                          vc_ref[pages].view(view))
    untouched = torch.ones(w.num_blocks, dtype=torch.bool, device="cuda")
    untouched[pidx] = False
    assert torch.equal(dev_bits_t(dw.key_cache)[untouched], kc_before[untouched])
    sel = np.arange(w.total_q) if rows is None else np.asarray(rows, np.int64)
    ref = attention_of(w, rows=sel, key_cache=kc_ref, value_cache=vc_ref)
    return assert_close(from_dev(dw.out)[sel], ref, w.dtype, w.name)


@pytest.mark.parametrize("P", [0, -1, 32])
@pytest.mark.parametrize("name,make", ONECALL, ids=[f[0] for f in ONECALL])
def test_scatter_and_attend_matches_oracle(name, make, P):
    """pa_scatter_and_attend against the oracle's scatter and attention
    (kwkr.cn kernel table: reshape_and_cache, then attention)."""
    _fused_vs_oracle(make(), partition_size=P)


@pytest.mark.parametrize("widx", [1, 3])
def test_scatter_and_attend_full_size_matches_oracle(widx):
    """The one-call step on the full-size decode and mixed workloads against
    the oracle (decode rows: all; multi-query requests: first, last and two
    random rows)."""
    w = wl.workload(widx)
    rng = np.random.default_rng(7)
    rows = []
    for r in range(w.num_seqs):
        c0, c1 = int(w.cu_seqlens_q[r]), int(w.cu_seqlens_q[r + 1])
        rows.extend(range(c0, c1) if c1 - c0 <= 5 else [c0, c1 - 1] + rng.integers(c0, c1, 2).tolist())
    _fused_vs_oracle(w, rows=sorted(set(rows)))


# ---------------------------------------------------------------- padded layout
@pytest.mark.parametrize("D,Hq,Hkv", [(256, 16, 2), (128, 8, 2), (64, 4, 4)])
def test_padded_layout_matches_oracle(D, Hq, Hkv):
    """The same ragged batch laid out padded ([B, T_max]: every request gets
    the longest request's query rows and keys, the layout a padded attention
    computes on; aisignalhub.me, "packed queries and paged KV", batch A vs B)
    runs through the same call and matches the oracle on every row."""
    small = wl.random_small(180 + D, dtype=wl.BF16, num_seqs=5, num_q_heads=Hq,
                            num_kv_heads=Hkv, head_dim=D, max_prior=0, max_q=90)
    w = wl.padded(small)
    assert len(set(w.q_lens.tolist())) == 1 and w.total_q == w.num_seqs * int(w.q_lens[0])
    check_step(w)


@pytest.mark.parametrize("D,dtype", [(128, wl.BF16), (64, wl.F32)])
def test_launch_plan_recorded_and_logged(D, dtype):
    """A real call records the plan pa_describe_plan gives for its sizes on
    this GPU, and with PA_DEBUG=1 prints it to stderr (a child process, so
    the variable is read at its first call)."""
    import os
    import subprocess
    import sys
    w = wl.random_small(515 + D, dtype=dtype, num_seqs=6, num_q_heads=8, num_kv_heads=2,
                        head_dim=D, max_prior=700, max_q=7)
    dw = DeviceWorkload(w)
    dw.scatter()
    dw.attention(partition_size=256)
    torch.cuda.synchronize()
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    want = pa.pa_describe_plan(w.num_seqs, w.total_q, w.max_seqlen_q, w.max_seqlen_k,
                               w.num_q_heads, w.num_kv_heads, D, 256, dtype, sms)
    assert pa.pa_last_plan() == want
    assert want["mq_kernel"] == ("paged_prefill_tc" if dtype == wl.BF16 else "paged_decode_rows")
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    code = ("import sys; sys.path.insert(0, %r); sys.path.insert(0, %r)\n"
            "from harness import DeviceWorkload\n"
            "from paged_kv_varlen_gb300 import workloads as wl\n"
            "w = wl.random_small(%d, dtype=%r, num_seqs=6, num_q_heads=8, num_kv_heads=2,"
            " head_dim=%d, max_prior=700, max_q=7)\n"
            "dw = DeviceWorkload(w); dw.scatter(); dw.attention(partition_size=256)\n"
            "import torch; torch.cuda.synchronize()\n"
            % (root, os.path.join(root, "tests"), 515 + D, dtype, D))
    r = subprocess.run([sys.executable, "-c", code], env=dict(os.environ, PA_DEBUG="1"),
                       capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l[4:] for l in r.stderr.splitlines() if l.startswith("pa: ")]
    assert lines and dict(kv.split("=", 1) for kv in lines[-1].split()) == want
