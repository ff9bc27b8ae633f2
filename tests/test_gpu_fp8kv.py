"""GPU parity of the quantised KV cache (E4M3 codes with a float32 scale per
(token, KV head) row -- this library's reading of the TurboQuant helpers the
layered-architecture page names, lqnn.cn section 5).

* pa_reshape_and_cache_fp8 against the oracle's quantisation: codes and scales
  bit for bit over the whole pool (padding tokens and slots past the pool
  skipped, unwritten slots untouched);
* pa_varlen_attention_fp8kv against the oracle's fp64 attention over the
  dequantised rows, at the bf16 tolerances (max abs 2e-2, mean abs 2e-3):
  decode rows (split or not), verify windows and prefill chunks, sinks,
  head_dim 128 and 256, groups 1 to 8, block sizes 16 and 32.
"""
import numpy as np
import pytest
import torch

from harness import assert_close, from_dev, to_dev
from oracle import oracle as orc
from paged_kv_varlen_gb300 import binding as pa
from paged_kv_varlen_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

POISON_CODE = 0x7F          # an E4M3 NaN: a slot the attention must never read
POISON_SCALE = float("nan")


class QuantPools:
    """Quantised pools on the GPU and their oracle twins, filled with every
    context token of a workload (prior context and this step's rows)."""

    def __init__(self, w, slots_override=None, in_dtype=None):
        self.w = w
        k, v, slots = w.all_tokens()
        if slots_override is not None:
            slots = slots_override
        self.in_dtype = in_dtype or w.dtype
        if self.in_dtype == wl.F32 and w.dtype == wl.BF16:   # the same values as float32
            k = (k.astype(np.uint32) << 16).view(np.float32)
            v = (v.astype(np.uint32) << 16).view(np.float32)
        nb, bs, Hkv, D = w.num_blocks, w.block_size, w.num_kv_heads, w.head_dim
        codes0 = np.full((nb, bs, Hkv, D), POISON_CODE, np.uint8)
        scales0 = np.full((nb, bs, Hkv), POISON_SCALE, np.float32)
        # the library skips slots past the pool as padding (reading R5); the
        # oracle refuses them, so it is given them as padding
        oracle_slots = np.where(np.asarray(slots) >= nb * bs, -1, slots)
        self.ref = orc.quantize_kv_fp8(k, v, codes0, codes0, scales0, scales0, oracle_slots, bs,
                                       self.in_dtype)
        self.kc = torch.from_numpy(codes0).cuda()
        self.vc = torch.from_numpy(codes0).cuda()
        self.ks = torch.from_numpy(scales0).cuda()
        self.vs = torch.from_numpy(scales0).cuda()
        kd, vd = to_dev(k, self.in_dtype), to_dev(v, self.in_dtype)
        pa.pa_reshape_and_cache_fp8(kd, vd, self.kc, self.vc, self.ks, self.vs,
                                    torch.from_numpy(np.asarray(slots, np.int64)).cuda())
        torch.cuda.synchronize()

    def check_bits(self):
        kc, vc, ks, vs = self.ref
        assert np.array_equal(self.kc.cpu().numpy(), kc)
        assert np.array_equal(self.vc.cpu().numpy(), vc)
        # scales bit for bit (NaN poison in untouched slots included)
        assert np.array_equal(self.ks.cpu().numpy().view(np.uint32), ks.view(np.uint32))
        assert np.array_equal(self.vs.cpu().numpy().view(np.uint32), vs.view(np.uint32))

    def attention(self, partition_size=0, rows=None):
        w = self.w
        q = to_dev(w.q, w.dtype)
        out = torch.full_like(q, float("nan"))
        sk = torch.from_numpy(w.sinks.astype(np.float32)).cuda() if w.sinks is not None else None
        pa.pa_varlen_attention_fp8kv(out, q, self.kc, self.vc, self.ks, self.vs,
                                     torch.from_numpy(w.cu_seqlens_q).cuda(),
                                     torch.from_numpy(w.seq_lens_k).cuda(),
                                     torch.from_numpy(w.block_tables).cuda(),
                                     max_seqlen_q=w.max_seqlen_q, max_seqlen_k=w.max_seqlen_k,
                                     scale=w.scale, sinks=sk, causal=w.causal,
                                     partition_size=partition_size)
        torch.cuda.synchronize()
        assert pa.pa_device_error() == 0
        kc, vc, ks, vs = self.ref
        sel = np.arange(w.total_q) if rows is None else np.asarray(rows, np.int64)
        ref = orc.paged_attention_kv(w.q, orc.dequantize_kv_fp8(kc, ks),
                                     orc.dequantize_kv_fp8(vc, vs), w.cu_seqlens_q,
                                     w.seq_lens_k, w.block_tables, q_dtype=w.dtype,
                                     num_q_heads=w.num_q_heads, num_kv_heads=w.num_kv_heads,
                                     head_dim=w.head_dim, block_size=w.block_size,
                                     scale=w.scale, causal=w.causal, sinks=w.sinks, rows=sel)
        return assert_close(from_dev(out)[sel], ref, wl.BF16, f"fp8 kv {w.name}")


@pytest.mark.parametrize("in_dtype", [wl.BF16, wl.F32])
@pytest.mark.parametrize("D", [128, 256])
def test_quantising_scatter_is_bit_exact(D, in_dtype):
    w = wl.random_small(300 + D, dtype=wl.BF16, num_seqs=6, num_q_heads=8, num_kv_heads=2,
                        head_dim=D, max_prior=200, max_q=9)
    k, v, slots = w.all_tokens()
    slots = slots.copy()
    nslots = w.num_blocks * w.block_size
    slots[0] = -1                        # padding token
    slots[len(slots) // 2] = nslots + 3  # past the pool: skipped
    pools = QuantPools(w, slots_override=slots, in_dtype=in_dtype)
    pools.check_bits()
    assert pa.pa_device_error() == 0


def test_quantising_scatter_zero_rows():
    w = wl.random_small(333, dtype=wl.BF16, num_seqs=2, num_q_heads=4, num_kv_heads=2,
                        head_dim=128, max_prior=20, max_q=2)
    w.key_cache[:] = 0
    w.value_cache[:] = 0
    w.new_k[:] = 0
    w.new_v[:] = 0
    pools = QuantPools(w)
    pools.check_bits()
    _, _, slots = w.all_tokens()
    bs = w.block_size
    assert (pools.ks.cpu().numpy()[slots // bs, slots % bs] == 0).all()


CASES = [(D, Hq, Hkv, bs) for D in (128, 256)
         for (Hq, Hkv, bs) in ((8, 2, 16), (8, 1, 32), (6, 6, 16), (14, 2, 16))]


@pytest.mark.parametrize("P", [0, -1, 256])
@pytest.mark.parametrize("D,Hq,Hkv,bs", CASES, ids=[f"D{a}-{b}x{c}-bs{d}" for a, b, c, d in CASES])
def test_fp8kv_attention_matches_oracle(D, Hq, Hkv, bs, P):
    w = wl.random_small(310 + D + Hq + bs, dtype=wl.BF16, num_seqs=7, num_q_heads=Hq,
                        num_kv_heads=Hkv, head_dim=D, block_size=bs, max_prior=900, max_q=20,
                        with_sinks=(Hkv == 2))
    pools = QuantPools(w)
    pools.check_bits()
    pools.attention(partition_size=P)


@pytest.mark.parametrize("causal", [True, False])
def test_fp8kv_decode_and_non_causal_rows(causal):
    w = wl.random_small(377, dtype=wl.BF16, num_seqs=9, num_q_heads=16, num_kv_heads=4,
                        head_dim=128, max_prior=2500, max_q=1 if causal else 12, causal=causal,
                        with_sinks=True)
    pools = QuantPools(w)
    pools.attention(partition_size=512)


def test_fp8kv_full_size_decode_batch():
    """The GQA decode batch (32 requests, contexts up to 8192) with its KV
    cache quantised; every row against the oracle."""
    w = wl.workload(1)
    pools = QuantPools(w)
    pools.check_bits()
    pools.attention(partition_size=w.partition_size)


@pytest.mark.parametrize("max_q", [1, 6])
def test_fp8kv_subnormal_codes(max_q):
    """Rows whose codes are E4M3 subnormals (+-m * 2^-9, m = 0..7) except one
    code of 448 in dim 0, with scale 16: the subnormal dims hold values of
    +-1/32 .. 7/32.  K and V share the codes and the softmax scale is 1, so
    the queries (zero in dim 0) score the keys by their subnormal dims alone
    and the output's dims 1.. are a query-weighted mean of them: about 0.045
    on average, against an error of the same size if either K or V lost its
    subnormals (flushed to zero by the decoder or the tensor cores).  Dim 0
    of the output (7168) is compared relative to its size."""
    w = wl.random_small(391 + max_q, dtype=wl.BF16, num_seqs=6, num_q_heads=8, num_kv_heads=2,
                        head_dim=128, max_prior=700, max_q=max_q)
    nb, bs, Hkv, D = w.num_blocks, w.block_size, w.num_kv_heads, w.head_dim
    rng = np.random.default_rng(7)
    sub = rng.integers(0, 8, size=(1, nb, bs, Hkv, D)).astype(np.uint8)     # 0 .. 7 x 2^-9
    sub |= (rng.integers(0, 2, size=sub.shape) << 7).astype(np.uint8)      # random sign
    sub[..., 0] = 0x7E                                                      # 448
    kc = vc = sub[0]
    scales = np.full((nb, bs, Hkv), 16.0, np.float32)
    qf = rng.normal(0, 2, size=(w.total_q, w.num_q_heads, D)).astype(np.float32)
    qf[..., 0] = 0
    q_bits = (qf.view(np.uint32) >> 16).astype(np.uint16)                  # exact in bf16 by truncation
    q = to_dev(q_bits, wl.BF16)
    out = torch.full_like(q, float("nan"))
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()       # noqa: E731
    pa.pa_varlen_attention_fp8kv(out, q, dev(kc), dev(vc), dev(scales), dev(scales),
                                 dev(w.cu_seqlens_q), dev(w.seq_lens_k), dev(w.block_tables),
                                 max_seqlen_q=w.max_seqlen_q, max_seqlen_k=w.max_seqlen_k,
                                 scale=1.0, causal=w.causal, partition_size=-1)
    torch.cuda.synchronize()
    assert pa.pa_device_error() == 0
    ref = orc.paged_attention_kv(q_bits, orc.dequantize_kv_fp8(kc, scales),
                                 orc.dequantize_kv_fp8(vc, scales), w.cu_seqlens_q,
                                 w.seq_lens_k, w.block_tables, q_dtype=wl.BF16,
                                 num_q_heads=w.num_q_heads, num_kv_heads=Hkv, head_dim=D,
                                 block_size=bs, scale=1.0, causal=w.causal)
    got = from_dev(out)
    # the subnormal dims carry the test: their outputs are far from zero
    assert np.abs(ref[..., 1:]).mean() > 0.02
    assert_close(got[..., 1:], ref[..., 1:], wl.BF16, f"fp8 subnormal codes q<={max_q}")
    rel = np.abs(got[..., 0] - ref[..., 0]) / np.maximum(np.abs(ref[..., 0]), 1.0)
    assert rel.max() <= 1e-2
