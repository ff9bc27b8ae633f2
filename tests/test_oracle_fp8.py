"""Pins of the oracle's quantised KV cache (CPU).

The pages name TurboQuant helpers for the KV cache (lqnn.cn, section 5) but
give no format; the reading taken: each (token, KV head) row is stored as E4M3
8-bit floats with one float32 scale, code = E4M3(x * 448 / amax), scale =
amax / 448.  Pinned here against things other than the oracle itself:

* the E4M3 format: every code's value and the rounding of float32 values to
  codes, against PyTorch's independent float8_e4m3fn type;
* the rounding error bound of the format (a code is the nearest one);
* the quantisation's own properties (the row maximum maps to +-448, a zero row
  to zeros, padding tokens and untouched slots);
* attention over the quantised cache equals dense brute force over the
  dequantised rows, and equals the plain attention when every row is exactly
  representable.
"""
import numpy as np
import pytest
import torch

from oracle import oracle as orc
from paged_kv_varlen_gb300 import workloads as wl


def _torch_codes(v):
    return torch.from_numpy(np.asarray(v, np.float32)).to(torch.float8_e4m3fn).view(
        torch.uint8).numpy()


def test_e4m3_values_match_torch():
    table = orc.e4m3_values()
    ref = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    assert np.array_equal(np.isnan(table), np.isnan(ref))
    ok = ~np.isnan(ref)
    assert np.array_equal(table[ok], ref[ok])
    assert table[0x7E] == 448.0 and table[0x01] == 2.0 ** -9 and np.isnan(table[0x7F])


def test_e4m3_rounding_matches_torch_including_ties():
    rng = np.random.default_rng(11)
    finite = orc.e4m3_values()[:0x7F]
    mids = (finite[:-1] + finite[1:]) / 2           # exact ties between neighbours
    v = np.concatenate([rng.uniform(-448, 448, 4000), rng.uniform(-0.03, 0.03, 4000),
                        rng.normal(0, 4, 4000), mids, -mids, [0.0, -0.0, 448.0, -448.0]])
    v = v.astype(np.float32)
    v = v[np.abs(v.astype(np.float64)) < 448.0 + 1e-9]
    assert np.array_equal(orc.e4m3_encode(v), _torch_codes(v))


def test_e4m3_saturates_and_is_the_nearest_code():
    assert orc.e4m3_encode([500.0, -1e6, 448.3])[0] == 0x7E
    assert orc.e4m3_encode([-500.0])[0] == 0xFE
    table = orc.e4m3_values()
    rng = np.random.default_rng(5)
    v = rng.uniform(-448, 448, 3000).astype(np.float32)
    codes = orc.e4m3_encode(v)
    finite = np.abs(table[:0x7F])
    for x, c in zip(v.astype(np.float64), codes):
        err = abs(table[c] - x)
        assert err <= np.min(np.abs(finite - abs(x))) + 0.0   # no code is nearer


def _quantize(w):
    k, v, slots = w.all_tokens()
    nb, bs = w.num_blocks, w.block_size
    kc = np.full((nb, bs, w.num_kv_heads, w.head_dim), 0x5A, np.uint8)
    vc = kc.copy()
    ks = np.full((nb, bs, w.num_kv_heads), -7.0, np.float32)
    vs = ks.copy()
    return orc.quantize_kv_fp8(k, v, kc, vc, ks, vs, slots, bs, w.dtype), (k, v, slots)


@pytest.mark.parametrize("dtype", [wl.BF16, wl.F32])
def test_quantised_rows_max_zero_padding_and_bound(dtype):
    w = wl.random_small(61, dtype=dtype, num_seqs=4, num_q_heads=8, num_kv_heads=2,
                        head_dim=128, max_prior=40, max_q=3)
    k, v, slots = w.all_tokens()
    k = k.copy()
    k[3] = 0                                   # a zero row (both heads)
    slots = slots.copy()
    slots[5] = -1                              # a padding token
    nb, bs, Hkv, D = w.num_blocks, w.block_size, w.num_kv_heads, w.head_dim
    kc0 = np.full((nb, bs, Hkv, D), 0x5A, np.uint8)
    ks0 = np.full((nb, bs, Hkv), -7.0, np.float32)
    kc, vc, ks, vs = orc.quantize_kv_fp8(k, v, kc0, kc0, ks0, ks0, slots, bs, dtype)
    table = orc.e4m3_values()
    kf = k.view(np.float32) if dtype == wl.F32 else \
        (k.astype(np.uint32) << 16).view(np.float32)
    written = np.zeros((nb, bs), bool)
    for t, s in enumerate(slots):
        if s < 0:
            continue
        written[s // bs, s % bs] = True
        for h in range(Hkv):
            codes, scale, x = kc[s // bs, s % bs, h], ks[s // bs, s % bs, h], kf[t, h]
            if t == 3:
                assert scale == 0.0 and not codes.any()
                continue
            amax = np.abs(x).max()
            assert scale == np.float32(amax / np.float32(448.0))
            assert np.abs(table[codes]).max() == 448.0                  # the row's max
            y = x.astype(np.float64) * np.float64(np.float32(448.0) / amax)
            # E4M3 spacing at |y|: 2^(e - 3) for normal values, 2^-9 below 2^-6
            e = np.floor(np.log2(np.maximum(np.abs(y), 2.0 ** -6)))
            assert (np.abs(table[codes] - y) <= 2.0 ** (e - 3) / 2 * (1 + 1e-6) + 1e-12).all()
    # padding token and untouched slots keep their bytes
    assert (kc[~written] == 0x5A).all() and (ks[~written] == -7.0).all()
    # a slot outside the pool is refused
    bad = slots.copy()
    bad[0] = nb * bs
    with pytest.raises(ValueError):
        orc.quantize_kv_fp8(k, v, kc0, kc0, ks0, ks0, bad, bs, dtype)


def _dense(w, kd, vd, slots):
    """Brute force over the dequantised rows, unpaged: request r's keys are the
    rows of its tokens in position order."""
    out = np.zeros((w.total_q, w.num_q_heads, w.head_dim))
    qf = (w.q.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    G = w.num_q_heads // w.num_kv_heads
    t0 = 0
    for r in range(w.num_seqs):
        N, n, c0 = int(w.seq_lens[r]), int(w.q_lens[r]), int(w.cu_seqlens_q[r])
        K, V = kd[t0:t0 + N], vd[t0:t0 + N]
        t0 += N
        for i in range(n):
            nvis = min(N, N - n + i + 1) if w.causal else N
            if nvis <= 0:
                continue
            for h in range(w.num_q_heads):
                s = w.scale * (K[:nvis, h // G] @ qf[c0 + i, h])
                m = s.max()
                if w.sinks is not None:
                    m = max(m, w.sinks[h])
                p = np.exp(s - m)
                den = p.sum() + (np.exp(w.sinks[h] - m) if w.sinks is not None else 0.0)
                out[c0 + i, h] = p @ V[:nvis, h // G] / den
    return out


@pytest.mark.parametrize("D,sinks", [(128, False), (256, True)])
def test_attention_over_quantised_cache_equals_dense_bruteforce(D, sinks):
    w = wl.random_small(71 + D, dtype=wl.BF16, num_seqs=4, num_q_heads=4, num_kv_heads=2,
                        head_dim=D, max_prior=45, max_q=6, with_sinks=sinks)
    (kc, vc, ks, vs), (_, _, slots) = _quantize(w)
    kd, vd = orc.dequantize_kv_fp8(kc, ks), orc.dequantize_kv_fp8(vc, vs)
    got = orc.paged_attention_kv(w.q, kd, vd, w.cu_seqlens_q, w.seq_lens_k, w.block_tables,
                                 q_dtype=w.dtype, num_q_heads=w.num_q_heads,
                                 num_kv_heads=w.num_kv_heads, head_dim=D,
                                 block_size=w.block_size, scale=w.scale, causal=w.causal,
                                 sinks=w.sinks)
    bs = w.block_size
    ref = _dense(w, kd[slots // bs, slots % bs], vd[slots // bs, slots % bs], slots)
    assert np.abs(got - ref).max() < 1e-12


def test_exactly_representable_rows_give_the_plain_attention():
    """Rows whose values are E4M3 values with a maximum of 448 quantise with
    scale 1 and codes equal to the values: attention over the quantised cache
    is then the plain attention over the bf16 cache."""
    w = wl.random_small(83, dtype=wl.BF16, num_seqs=3, num_q_heads=4, num_kv_heads=2,
                        head_dim=128, max_prior=30, max_q=3)
    table = orc.e4m3_values()
    rng = np.random.default_rng(3)
    finite = table[np.isfinite(table)]
    k, v, slots = w.all_tokens()
    vals = rng.choice(finite, size=k.shape).astype(np.float32)
    vals[..., 0] = 448.0
    bits = (vals.view(np.uint32) >> 16).astype(np.uint16)   # exact in bf16 (<= 4 bits)
    assert np.array_equal((bits.astype(np.uint32) << 16).view(np.float32), vals)
    nb, bs = w.num_blocks, w.block_size
    kc0 = np.zeros((nb, bs, w.num_kv_heads, w.head_dim), np.uint8)
    ks0 = np.zeros((nb, bs, w.num_kv_heads), np.float32)
    kc, vc, ks, vs = orc.quantize_kv_fp8(bits, bits, kc0, kc0, ks0, ks0, slots, bs, wl.BF16)
    assert (ks[slots // bs, slots % bs] == 1.0).all()
    kd = orc.dequantize_kv_fp8(kc, ks)
    plain_k = np.zeros((nb, bs, w.num_kv_heads, w.head_dim), np.uint16)
    plain_k[slots // bs, slots % bs] = bits
    got = orc.paged_attention_kv(w.q, kd, kd, w.cu_seqlens_q, w.seq_lens_k, w.block_tables,
                                 q_dtype=w.dtype, num_q_heads=w.num_q_heads,
                                 num_kv_heads=w.num_kv_heads, head_dim=w.head_dim,
                                 block_size=bs, scale=w.scale, causal=w.causal)
    ref = orc.paged_attention(w.q, plain_k, plain_k, w.cu_seqlens_q, w.seq_lens_k,
                              w.block_tables, dtype=w.dtype, num_q_heads=w.num_q_heads,
                              num_kv_heads=w.num_kv_heads, head_dim=w.head_dim, block_size=bs,
                              scale=w.scale, causal=w.causal)
    assert np.abs(got - ref).max() < 1e-12
