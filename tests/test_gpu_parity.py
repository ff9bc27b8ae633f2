"""GPU parity: the CUDA path (through the C ABI) against the fp64 oracle.

Small ragged cases span several tiles, partitions and a ragged tail; the
five named workloads run at full size in the launch configuration the
benchmark times, compared on sampled rows (all rows where the oracle is
quick).  Tolerances: fp32 max abs 1e-5; bf16 max abs 2e-2 and mean 2e-3.
"""
import math
import zlib

import numpy as np

import pytest
import torch

from harness import DeviceWorkload, assert_close, check_step, from_dev
from oracle.oracle import attention_of
from paged_kv_varlen_gb300 import binding as pa
from paged_kv_varlen_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


# ---------------------------------------------------------------- small cases
SMALL = []
for dtype in (wl.F32, wl.BF16):
    for D in (64, 128, 256):
        for (Hq, Hkv) in ((4, 2), (8, 1), (6, 6), (12, 2)):
            SMALL.append(dict(dtype=dtype, head_dim=D, num_q_heads=Hq, num_kv_heads=Hkv))


@pytest.mark.parametrize("case", SMALL, ids=lambda c: "{dtype}-D{head_dim}-{num_q_heads}x{num_kv_heads}".format(**c))
@pytest.mark.parametrize("bs", [8, 16, 32])
def test_small_ragged_mixed(case, bs):
    seed = zlib.crc32(repr((case["dtype"], case["head_dim"], case["num_q_heads"], bs)).encode()) % 10000
    w = wl.random_small(seed, num_seqs=5, block_size=bs, max_prior=300, max_q=6,
                        with_sinks=(bs == 16), **case)
    check_step(w)


@pytest.mark.parametrize("P", [-1, 0, 32, 256, 512])
@pytest.mark.parametrize("dtype", [wl.F32, wl.BF16])
def test_decode_partitions(P, dtype):
    """Single-query rows with contexts spanning many partitions and a ragged tail."""
    w = wl.random_small(77, dtype=dtype, num_seqs=6, num_q_heads=8, num_kv_heads=2,
                        head_dim=128, block_size=16, max_prior=2100, max_q=1,
                        with_sinks=True, partition_size=P)
    check_step(w)


@pytest.mark.parametrize("with_sinks", [False, True])
def test_decode_item_split_across_many_ctas(with_sinks):
    """One 65536-key partition next to 100 one-tile requests: the decode grid
    balances tiles, so that partition is cut between dozens of CTAs, whose
    partials the reduce merges (kwkr.cn trick 4: split partials + one reduce)."""
    prior = np.array([65535] + [127] * 100, dtype=np.int64)
    w = wl.build("split_across_ctas", wl.BF16, 4, 1, 128, 16, prior, np.ones(101, np.int64),
                 seed=101, partition_size=65536, with_sinks=with_sinks, pool_slack=1.2)
    check_step(w)


def test_split_merge_is_bit_reproducible():
    """A partition cut across dozens of CTAs leaves many extra partials per
    head; the reduce merges them in a fixed (cut-table) order, so two runs
    give identical bits."""
    prior = np.array([65535] + [127] * 100, dtype=np.int64)
    w = wl.build("split_across_ctas", wl.BF16, 4, 1, 128, 16, prior, np.ones(101, np.int64),
                 seed=101, partition_size=65536, with_sinks=True, pool_slack=1.2)
    first = _run(w)
    second = _run(w)
    torch.cuda.synchronize()
    assert pa.pa_device_error() == 0
    assert torch.equal(dev_bits_t(first.out), dev_bits_t(second.out))


def test_non_causal_rows():
    w = wl.random_small(78, dtype=wl.F32, num_seqs=4, head_dim=64, max_prior=100, max_q=9,
                        causal=False)
    check_step(w)


def test_tiny_decode_workload_matches_oracle():
    check_step(wl.workload(0))


def test_tiny_decode_workload_matches_stored_golden():
    import json
    import os
    g = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "tiny_decode_f32.json")))
    dw = DeviceWorkload(wl.workload(0))
    dw.step()
    out = from_dev(dw.out).ravel()
    assert np.max(np.abs(out - np.array(g["out"]))) <= 1e-5


# ---------------------------------------------------------------- invariances
def _run(w, **kw):
    dw = DeviceWorkload(w)
    dw.step(**kw)
    torch.cuda.synchronize()
    return dw


def test_split_equals_no_split_fp32():
    w = wl.random_small(79, dtype=wl.F32, num_seqs=5, head_dim=128, num_q_heads=8,
                        num_kv_heads=2, max_prior=1500, max_q=1, with_sinks=True)
    ref = from_dev(_run(w, partition_size=-1).out)
    for P in (256, 512):
        got = from_dev(_run(w, partition_size=P).out)
        assert np.max(np.abs(got - ref)) <= 1e-6


def test_poisoned_slots_never_reach_output():
    wp = wl.random_small(80, dtype=wl.BF16, num_seqs=5, max_prior=200, max_q=5)
    wz = wl.random_small(80, dtype=wl.BF16, num_seqs=5, max_prior=200, max_q=5, poison=False)
    a = _run(wp).out
    b = _run(wz).out
    assert torch.isfinite(a.float()).all()
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))


def test_page_permutation_is_invisible():
    w = wl.random_small(81, dtype=wl.BF16, num_seqs=4, max_prior=400, max_q=3)
    base = _run(w).out.clone()
    perm = np.random.default_rng(5).permutation(w.num_blocks)
    w2 = wl.random_small(81, dtype=wl.BF16, num_seqs=4, max_prior=400, max_q=3)
    kc2 = np.empty_like(w2.key_cache); vc2 = np.empty_like(w2.value_cache)
    kc2[perm] = w2.key_cache; vc2[perm] = w2.value_cache
    w2.key_cache, w2.value_cache = kc2, vc2
    w2.block_tables = np.where(w2.block_tables >= 0, perm[np.maximum(w2.block_tables, 0)],
                               -1).astype(np.int32)
    bs = w2.block_size
    w2.slot_mapping = (perm[w2.slot_mapping // bs] * bs + w2.slot_mapping % bs).astype(np.int64)
    got = _run(w2).out
    assert torch.equal(base.view(torch.int16), got.view(torch.int16))


def test_block_size_translation_is_invisible():
    """A 32-token-page pool viewed as 16-token pages by a reshape only."""
    w = wl.random_small(82, dtype=wl.BF16, num_seqs=4, block_size=32, max_prior=500, max_q=4)
    dw = _run(w)
    base = dw.out.clone()
    kc16 = dw.key_cache.view(w.num_blocks * 2, 16, w.num_kv_heads, w.head_dim)
    vc16 = dw.value_cache.view(w.num_blocks * 2, 16, w.num_kv_heads, w.head_dim)
    bt = torch.from_numpy(w.block_tables).cuda()
    bt16 = torch.stack([bt * 2, bt * 2 + 1], dim=2).reshape(bt.shape[0], -1)
    bt16 = torch.where(bt16 >= 0, bt16, torch.full_like(bt16, -1)).to(torch.int32).contiguous()
    out = torch.empty_like(base)
    pa.pa_varlen_attention(out, dw.q, kc16, vc16, dw.cu_seqlens_q, dw.seq_lens_k, bt16,
                           max_seqlen_q=w.max_seqlen_q, max_seqlen_k=w.max_seqlen_k,
                           scale=w.scale, causal=True)
    torch.cuda.synchronize()
    assert torch.equal(base.view(torch.int16), out.view(torch.int16))


def test_block_size_144_as_nine_16_token_pages():
    """A 144-token-page pool (the page size of hybrid models) attended directly and
    viewed as nine 16-token pages by a reshape and a block-table expansion
    (pptc.cn, block-size translation): parity with the oracle, identical bits."""
    w = wl.random_small(83, dtype=wl.BF16, num_seqs=4, block_size=144, max_prior=700, max_q=4)
    check_step(w)
    dw = _run(w)
    base = dw.out.clone()
    kc16 = dw.key_cache.view(w.num_blocks * 9, 16, w.num_kv_heads, w.head_dim)
    vc16 = dw.value_cache.view(w.num_blocks * 9, 16, w.num_kv_heads, w.head_dim)
    bt = torch.from_numpy(w.block_tables).cuda()
    bt16 = torch.stack([bt * 9 + k for k in range(9)], dim=2).reshape(bt.shape[0], -1)
    bt16 = torch.where(bt16 >= 0, bt16, torch.full_like(bt16, -1)).to(torch.int32).contiguous()
    out = torch.empty_like(base)
    pa.pa_varlen_attention(out, dw.q, kc16, vc16, dw.cu_seqlens_q, dw.seq_lens_k, bt16,
                           max_seqlen_q=w.max_seqlen_q, max_seqlen_k=w.max_seqlen_k,
                           scale=w.scale, causal=True)
    torch.cuda.synchronize()
    assert torch.equal(base.view(torch.int16), out.view(torch.int16))


FUSED = [
    # (name, workload factory): decode-only and mixed steps; with bf16 at D = 128 /
    # 256 the decode kernel is launched while the scatter runs (only its K/V
    # loads wait for it), fp32 and D = 64 run the kernels one after the other
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
    # 600 short decode requests: CTAs whose work spans several 224-request
    # chunks of the decode kernel's plan scan
    ("decode-600-short", lambda: wl.random_small(96, dtype=wl.BF16, num_seqs=600, head_dim=128,
                                                  num_q_heads=4, num_kv_heads=1, max_prior=200,
                                                  max_q=1)),
]


@pytest.mark.parametrize("P", [0, -1, 32])
@pytest.mark.parametrize("name,make", FUSED, ids=[f[0] for f in FUSED])
def test_scatter_and_attend_equals_two_calls(name, make, P):
    """pa_scatter_and_attend == pa_reshape_and_cache then pa_varlen_attention:
    bit-identical caches and outputs (kwkr.cn kernel table: scatter, then attend;
    the overlapped decode launch must not read a K/V row before it is written)."""
    w = make()
    two = _run(w, partition_size=P)
    one = DeviceWorkload(w)
    one.fused_step(partition_size=P)
    torch.cuda.synchronize()
    assert pa.pa_device_error() == 0
    assert torch.equal(dev_bits_t(two.key_cache), dev_bits_t(one.key_cache))
    assert torch.equal(dev_bits_t(two.value_cache), dev_bits_t(one.value_cache))
    assert torch.equal(dev_bits_t(two.out), dev_bits_t(one.out))


@pytest.mark.parametrize("widx", [1, 3, 4])
def test_scatter_and_attend_full_size(widx):
    """The fused call on the full-size decode, mixed and long-decode workloads:
    bit-identical to the two calls."""
    w = wl.workload(widx)
    two = _run(w)
    one = DeviceWorkload(w)
    one.fused_step()
    torch.cuda.synchronize()
    assert pa.pa_device_error() == 0
    assert torch.equal(dev_bits_t(two.key_cache), dev_bits_t(one.key_cache))
    assert torch.equal(dev_bits_t(two.value_cache), dev_bits_t(one.value_cache))
    assert torch.equal(dev_bits_t(two.out), dev_bits_t(one.out))


def dev_bits_t(t):
    return t.view(torch.int16) if t.dtype == torch.bfloat16 else t.view(torch.int32)


def test_packing_independence():
    w = wl.random_small(83, dtype=wl.F32, num_seqs=4, max_prior=300, max_q=6)
    packed = from_dev(_run(w).out)
    for r in range(w.num_seqs):
        sub = wl.build("alone", wl.F32, w.num_q_heads, w.num_kv_heads, w.head_dim, w.block_size,
                       w.prior_lens[r:r + 1], w.q_lens[r:r + 1], seed=0)
        c0, c1 = int(w.cu_seqlens_q[r]), int(w.cu_seqlens_q[r + 1])
        # same data: reuse the packed workload's pool, block table row and queries
        sub.key_cache, sub.value_cache = w.key_cache, w.value_cache
        sub.block_tables = w.block_tables[r:r + 1]
        sub.q = w.q[c0:c1]
        sub.new_k, sub.new_v = w.new_k[c0:c1], w.new_v[c0:c1]
        sub.slot_mapping = w.slot_mapping[c0:c1]
        alone = from_dev(_run(sub).out)
        assert np.max(np.abs(alone - packed[c0:c1])) <= 1e-6


# ---------------------------------------------------------------- degenerate
def test_zero_length_context_rows_are_zero():
    w = wl.random_small(84, dtype=wl.F32, num_seqs=3, max_prior=40, max_q=1, with_sinks=True)
    dw = DeviceWorkload(w)
    dw.scatter()
    dw.seq_lens_k[1] = 0
    dw.attention(partition_size=32)
    torch.cuda.synchronize()
    row = int(w.cu_seqlens_q[1])
    assert torch.count_nonzero(dw.out[row]) == 0
    w.seq_lens_k = w.seq_lens_k.copy(); w.seq_lens_k[1] = 0
    kc, vc = w.pool_with_new_tokens()
    ref = attention_of(w, key_cache=kc, value_cache=vc)
    assert_close(from_dev(dw.out), ref, w.dtype)


def test_empty_batch_is_a_noop():
    q = torch.empty(0, 4, 64, device="cuda")
    out = torch.empty_like(q)
    kc = torch.zeros(4, 16, 2, 64, device="cuda")
    cu = torch.zeros(1, dtype=torch.int32, device="cuda")
    sl = torch.zeros(0, dtype=torch.int32, device="cuda")
    bt = torch.zeros(0, 1, dtype=torch.int32, device="cuda")
    pa.pa_varlen_attention(out, q, kc, kc, cu, sl, bt, max_seqlen_q=0, max_seqlen_k=0,
                           scale=0.1)


def test_workspace_too_small_is_rejected():
    w = wl.random_small(85, dtype=wl.BF16, max_prior=900, max_q=1)
    dw = DeviceWorkload(w)
    ws = torch.empty(16, dtype=torch.uint8, device="cuda")
    with pytest.raises(pa.PAError, match="WORKSPACE"):
        dw.attention(partition_size=256, workspace=ws)


def test_unsupported_head_dim_is_rejected():
    q = torch.zeros(1, 2, 96, device="cuda")
    kc = torch.zeros(2, 16, 1, 96, device="cuda")
    cu = torch.tensor([0, 1], dtype=torch.int32, device="cuda")
    sl = torch.tensor([5], dtype=torch.int32, device="cuda")
    bt = torch.zeros(1, 1, dtype=torch.int32, device="cuda")
    with pytest.raises(pa.PAError, match="UNSUPPORTED"):
        pa.pa_varlen_attention(torch.empty_like(q), q, kc, kc, cu, sl, bt, max_seqlen_q=1,
                               max_seqlen_k=5, scale=0.1)


# ---------------------------------------------------------------- split reduce
def test_split_kv_reduce_matches_oracle_combine():
    from oracle import oracle as orc
    rng = np.random.default_rng(9)
    S, Hq, D, P = 5, 6, 128, 256
    lens = np.array([0, 1, 300, 2048, 1000], np.int32)
    max_parts = int(math.ceil(lens.max() / P))
    po = rng.standard_normal((S, max_parts, Hq, D)).astype(np.float32)
    pm = (rng.standard_normal((S, max_parts, Hq)) * 4).astype(np.float32)
    pl = rng.uniform(1.0, 300.0, (S, max_parts, Hq)).astype(np.float32)
    cu = np.arange(S + 1, dtype=np.int32)
    sinks = rng.standard_normal(Hq).astype(np.float32)
    ref = orc.split_combine(po, pm, pl, cu, lens, partition_size=P, sinks=sinks)
    for dt, tdt in ((wl.F32, torch.float32), (wl.BF16, torch.bfloat16)):
        out = torch.zeros(S, Hq, D, dtype=tdt, device="cuda")
        pa.pa_split_kv_reduce(out, torch.from_numpy(po).cuda(), torch.from_numpy(pm).cuda(),
                              torch.from_numpy(pl).cuda(), torch.from_numpy(cu).cuda(),
                              torch.from_numpy(lens).cuda(), partition_size=P,
                              sinks=torch.from_numpy(sinks).cuda())
        torch.cuda.synchronize()
        assert_close(from_dev(out), ref, dt, f"reduce {dt}")


# ---------------------------------------------------------------- full-size workloads
def test_workload_gqa_decode_full_size():
    """32 decode rows, contexts U[512, 8192], (32, 8, 128), 40k-page pool, P = 512."""
    check_step(wl.workload(1))


def test_workload_varlen_prefill_full_size():
    """8 requests (3000 + 7 x ~430 tokens), causal prefill, (16, 2, 256): sampled rows."""
    w = wl.workload(2)
    rng = np.random.default_rng(0)
    cu = w.cu_seqlens_q
    rows = set(rng.choice(w.total_q, 40, replace=False).tolist())
    for r in range(w.num_seqs):                      # first, last and tile-edge rows
        rows.update({int(cu[r]), int(cu[r + 1]) - 1, min(int(cu[r]) + 127, int(cu[r + 1]) - 1)})
    check_step(w, rows=sorted(rows))


def test_workload_mixed_step_full_size():
    """64 requests: 40 decode, 16 verify (q = 1 + k), 8 prefill chunks (q = 512)."""
    w = wl.workload(3)
    rng = np.random.default_rng(1)
    rows = []
    for r in range(w.num_seqs):
        c0, c1 = int(w.cu_seqlens_q[r]), int(w.cu_seqlens_q[r + 1])
        if c1 - c0 <= 5:
            rows.extend(range(c0, c1))               # every decode / verify row
        else:
            rows.extend([c0, c1 - 1] + rng.integers(c0, c1, 2).tolist())
    check_step(w, rows=sorted(set(rows)))


@pytest.mark.parametrize("P", [256, 512, -1])
def test_workload_long_decode_sinks_full_size(P):
    """4 x 65536 + 12 x ~4600 contexts, (24, 4, 256), bs 32, sinks; P in {256, 512, none}."""
    check_step(wl.workload(4, partition_size=P))


@pytest.mark.parametrize("scale", [0.0, -0.07])
@pytest.mark.parametrize("dtype", [wl.F32, wl.BF16])
def test_zero_and_negative_scale(scale, dtype):
    """scale 0 gives plain prefix means; a negative scale flips the ordering of
    the scores.  Both must hold on the decode and the multi-query kernels."""
    w = wl.random_small(86, dtype=dtype, num_seqs=5, head_dim=128, num_q_heads=8,
                        num_kv_heads=2, max_prior=400, max_q=6, with_sinks=True)
    w.scale = scale
    check_step(w)


def test_step_staging_one_copy_matches_separate_inputs():
    """StepStaging: the step's inputs packed in one pinned buffer and uploaded in
    one copy give the same caches and output as separately copied inputs."""
    from paged_kv_varlen_gb300.staging import StepStaging
    w = wl.random_small(99, dtype=wl.BF16, num_seqs=9, num_q_heads=8, num_kv_heads=2,
                        head_dim=128, max_prior=900, max_q=4, with_sinks=True)
    ref = DeviceWorkload(w)
    ref.fused_step(partition_size=256)
    got = DeviceWorkload(w)
    names = {"q": got.q, "new_k": got.new_k, "new_v": got.new_v,
             "slot_mapping": got.slot_mapping, "cu_seqlens_q": got.cu_seqlens_q,
             "seq_lens_k": got.seq_lens_k, "block_tables": got.block_tables}
    stage = StepStaging(names, got.q.device)
    for n, t in names.items():
        stage.host[n].copy_(t.cpu())
    stage.upload()
    torch.cuda.synchronize()
    for n, t in names.items():
        assert stage.dev[n].data_ptr() % 256 == 0
        assert torch.equal(stage.dev[n].view(torch.uint8) if t.dtype == torch.bfloat16
                           else stage.dev[n], t.view(torch.uint8) if t.dtype == torch.bfloat16
                           else t)
    d = stage.dev
    out = torch.empty_like(got.q)
    pa.pa_scatter_and_attend(
        d["new_k"], d["new_v"], d["slot_mapping"], out, d["q"], got.key_cache, got.value_cache,
        d["cu_seqlens_q"], d["seq_lens_k"], d["block_tables"], max_seqlen_q=w.max_seqlen_q,
        max_seqlen_k=w.max_seqlen_k, scale=w.scale, sinks=got.sinks, causal=w.causal,
        partition_size=256, workspace=got.poisoned_workspace(256))
    torch.cuda.synchronize()
    assert pa.pa_device_error() == 0
    assert torch.equal(dev_bits_t(ref.key_cache), dev_bits_t(got.key_cache))
    assert torch.equal(dev_bits_t(ref.out), dev_bits_t(out))
