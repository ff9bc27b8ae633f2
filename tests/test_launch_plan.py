"""The launch plan of an attention call (pa_describe_plan / pa_last_plan, the
counterpart of the kwkr.cn hands-on section's dispatch diagnostics), on the
CPU: which kernel serves the single-query rows and the multi-query rows, with
which grid, split-KV partition, reduce and workspace.  The plan is host
arithmetic on the call's sizes alone; the GPU test in test_gpu_edges.py checks
that a real call records the same plan."""
import pytest

from paged_kv_varlen_gb300 import binding as pa

SMS = 152


def plan(*args, **kw):
    return pa.pa_describe_plan(*args, **kw)


def test_gqa_decode_batch_plan():
    p = plan(32, 32, 1, 8192, 32, 8, 128, 512, "bf16", SMS)
    assert p["decode_kernel"] == "paged_decode_tc" and p["decode_grid"] == f"{SMS}x1x1"
    assert p["partition"] == "512" and p["max_parts"] == "16"
    assert p["reduce"] == "split_reduce" and p["reduce_grid"] == "32x32"
    assert p["mq_kernel"] == "none" and p["cache"] == "plain" and p["group"] == "4"
    assert int(p["workspace"]) == pa.pa_varlen_attention_workspace_size(32, 8192, 32, 128, 512)


def test_small_batch_gets_fewer_ctas_than_sms():
    # 2 requests x 1 KV head x 1 partition: two items, two CTAs
    p = plan(2, 2, 1, 300, 4, 1, 128, -1, "bf16", SMS)
    assert p["decode_grid"] == "2x1x1" and p["partition"] == "0" and p["reduce"] == "none"
    assert p["workspace"] == "0"


def test_partition_choice_follows_the_work_budget():
    for (S, Hkv, N), want in (((4, 4, 32768), "512"), ((2, 2, 4096), "256"),
                              ((32, 8, 8192), "1024"), ((512, 8, 2000), "0"), ((8, 8, 400), "0")):
        p = plan(S, S, 1, N, 4 * Hkv, Hkv, 128, 0, "bf16", SMS)
        assert p["partition"] == want == str(pa.pa_choose_partition_size(S, Hkv, N, 0, SMS))


def test_prefill_batch_plan():
    # 8 requests, 6000 packed rows, head_dim 256, G = 8: the persistent
    # multi-query kernel with at most one CTA per SM
    p = plan(8, 6000, 3000, 3000, 16, 2, 256, -1, "bf16", SMS)
    assert p["mq_kernel"] == "paged_prefill_tc" and p["mq_grid"] == f"{SMS}x1x1"
    # the unit plan lives in the workspace even without split-KV
    assert int(p["workspace"]) == pa.pa_varlen_attention_workspace_size(8, 3000, 16, 256, -1) > 0
    # few units: fewer CTAs than SMs (2 requests x 1 KV head, 16 rows each: 2 + 2 units)
    p = plan(2, 32, 16, 100, 8, 1, 128, -1, "bf16", SMS)
    assert p["mq_grid"] == "4x1x1"


def test_float32_plan_uses_the_cuda_core_kernels():
    p = plan(4, 40, 12, 900, 8, 2, 64, 256, "f32", SMS)
    assert p["decode_kernel"] == "paged_decode" and p["decode_grid"] == "4x2x4"   # parts, Hkv, S
    assert p["mq_kernel"] == "paged_decode_rows" and p["mq_grid"] == "40x2x1"     # rows, Hkv
    # bf16 at head_dim 64 decodes on the CUDA cores too
    assert plan(4, 4, 1, 900, 8, 2, 64, 256, "bf16", SMS)["decode_kernel"] == "paged_decode"


def test_quantised_cache_plan():
    p = plan(32, 32, 1, 8192, 32, 8, 128, 512, "bf16", SMS, quantised=True)
    assert p["cache"] == "e4m3" and p["decode_kernel"] == "paged_decode_tc_fp8"
    p = plan(4, 40, 12, 900, 8, 2, 128, 256, "bf16", SMS, quantised=True)
    assert p["mq_kernel"] == "paged_decode_rows"   # multi-query rows: CUDA cores
    with pytest.raises(pa.PAError):
        plan(4, 4, 1, 900, 8, 2, 128, 256, "f32", SMS, quantised=True)


@pytest.mark.parametrize("bad", [dict(num_seqs=0), dict(total_q=0), dict(num_q_heads=6),
                                 dict(partition_size=-2)])
def test_invalid_sizes_are_refused(bad):
    args = dict(num_seqs=4, total_q=4, max_seqlen_q=1, max_seqlen_k=100, num_q_heads=8,
                num_kv_heads=4, head_dim=128, partition_size=0, dtype="bf16", sm_count=SMS)
    args.update(bad)
    with pytest.raises(pa.PAError):
        pa.pa_describe_plan(**args)


def test_no_call_no_last_plan():
    # nothing has launched on this thread (the CPU suite launches no kernel)
    import threading
    seen = []
    t = threading.Thread(target=lambda: seen.append(pa.pa_last_plan()))
    t.start()
    t.join()
    assert seen == [{}]


def test_workspace_query_covers_every_plan():
    """pa_varlen_attention_workspace_size (which has no SM count) is enough for
    the plan of any GPU size: random batch shapes, partition sizes -1 / 0 /
    forced, SM counts from 1 to 256, plain and quantised caches."""
    import random
    rnd = random.Random(5)
    for _ in range(3000):
        S = rnd.randint(1, 300)
        Hkv = rnd.choice([1, 2, 4, 8])
        Hq = Hkv * rnd.randint(1, 8)
        D = rnd.choice([64, 128, 256])
        max_k = rnd.choice([0, 1, 100, 600, 4096, 70000])
        max_q = rnd.choice([1, 1, 5, 300])
        P = rnd.choice([-1, 0, 0, 32, 256, 512, 1024])
        dtype = rnd.choice(["bf16", "f32"])
        quant = dtype == "bf16" and D != 64 and rnd.random() < 0.3
        sms = rnd.randint(1, 256)
        total_q = S * max_q
        p = plan(S, total_q, max_q, max_k, Hq, Hkv, D, P, dtype, sms, quantised=quant)
        need = int(p["workspace"])
        have = pa.pa_varlen_attention_workspace_size(S, max_k, Hq, D, P)
        assert need <= have, (S, Hkv, Hq, D, max_k, max_q, P, dtype, sms, need, have)
        assert int(p["max_parts"]) >= 1
        if p["partition"] != "0":
            assert p["reduce"] == "split_reduce"
            assert int(p["max_parts"]) == -(-max(max_k, 1) // int(p["partition"])) or max_k == 0
