"""Pins of the fp64 oracle to things other than itself (CPU only).

Each pin targets a plausible mistake in the oracle:
  * dense brute force on the *unpaged* K/V (contiguous per request, numpy):
    block-table gather, slot arithmetic, GQA head mapping, causal alignment;
  * torch's scaled_dot_product_attention in float64: the softmax formula and
    the scale (a library routine with its own implementation);
  * closed forms: equal keys -> mean of visible V, scale 0 -> prefix mean, a
    single visible key -> that V row, a two-key logistic case, a sink acting as
    one extra key with a zero value vector;
  * invariances the pages fix: permuting physical pages with matching block
    tables, reshape-only block-size translation (32 -> 16, 144 -> 9 x 16),
    poisoned unwritten slots, split-KV (256/512/other) equal to no split,
    packing independence, decode row == last prefill row;
  * the scatter: byte-exact against direct indexing; untouched slots kept.
"""
import math

import numpy as np
import pytest

import oracle
from oracle.oracle import attention_of
from paged_kv_varlen_gb300 import workloads as wl


def dense_bruteforce(w):
    """Contiguous per-request attention from the unpaged K/V arrays."""
    q = wl.to_f64(w.q, w.dtype)
    k_all = wl.to_f64(w.k_ctx, w.dtype)
    v_all = wl.to_f64(w.v_ctx, w.dtype)
    G = w.group
    out = np.zeros((w.total_q, w.num_q_heads, w.head_dim))
    for r in range(w.num_seqs):
        n = int(w.q_lens[r]); N = int(w.seq_lens[r])
        if n == 0:
            continue
        c0 = int(w.cu_seqlens_q[r])
        K = k_all[w.ctx_offsets[r]:w.ctx_offsets[r] + N]
        V = v_all[w.ctx_offsets[r]:w.ctx_offsets[r] + N]
        i = np.arange(n)[:, None]
        j = np.arange(N)[None, :]
        mask = (j <= N - n + i) if w.causal else np.ones((n, N), bool)
        for h in range(w.num_q_heads):
            S = w.scale * q[c0:c0 + n, h] @ K[:, h // G].T
            S = np.where(mask, S, -np.inf)
            m = S.max(axis=1, initial=-np.inf)
            if w.sinks is not None:
                m = np.maximum(m, float(w.sinks[h]))
            m = np.where(np.isfinite(m), m, 0.0)
            P = np.where(mask, np.exp(S - m[:, None]), 0.0)
            den = P.sum(axis=1)
            if w.sinks is not None:
                den = den + np.exp(float(w.sinks[h]) - m)
            O = P @ V[:, h // G]
            has = mask.any(axis=1)
            out[c0:c0 + n, h] = np.where(has[:, None], O / np.where(has, den, 1.0)[:, None], 0.0)
    return out


SMALL_CASES = [
    dict(seed=1, dtype=wl.F32, head_dim=64, num_q_heads=4, num_kv_heads=2, block_size=16),
    dict(seed=2, dtype=wl.BF16, head_dim=128, num_q_heads=8, num_kv_heads=2, block_size=8),
    dict(seed=3, dtype=wl.BF16, head_dim=32, num_q_heads=6, num_kv_heads=1, block_size=32,
         with_sinks=True),
    dict(seed=4, dtype=wl.F32, head_dim=16, num_q_heads=3, num_kv_heads=3, block_size=16,
         causal=False, max_q=9),
    dict(seed=5, dtype=wl.F32, head_dim=64, num_q_heads=8, num_kv_heads=1, block_size=16,
         num_seqs=4, with_sinks=True, max_q=12),
]


@pytest.mark.parametrize("case", SMALL_CASES, ids=lambda c: f"seed{c['seed']}")
def test_oracle_matches_dense_bruteforce(case):
    w = wl.random_small(**case)
    got = attention_of(w)
    ref = dense_bruteforce(w)
    assert np.max(np.abs(got - ref)) < 1e-12


def test_oracle_matches_bruteforce_tiny_decode_workload():
    w = wl.workload(0)
    assert np.max(np.abs(attention_of(w) - dense_bruteforce(w))) < 1e-12


def _sdpa_reference(w, extra_zero_key_logits=None):
    torch = pytest.importorskip("torch")
    import torch.nn.functional as F
    q = torch.from_numpy(wl.to_f64(w.q, w.dtype))
    k_all = torch.from_numpy(wl.to_f64(w.k_ctx, w.dtype))
    v_all = torch.from_numpy(wl.to_f64(w.v_ctx, w.dtype))
    G = w.group
    out = torch.zeros(w.total_q, w.num_q_heads, w.head_dim, dtype=torch.float64)
    for r in range(w.num_seqs):
        n = int(w.q_lens[r]); N = int(w.seq_lens[r]); c0 = int(w.cu_seqlens_q[r])
        K = k_all[w.ctx_offsets[r]:w.ctx_offsets[r] + N].repeat_interleave(G, dim=1)
        V = v_all[w.ctx_offsets[r]:w.ctx_offsets[r] + N].repeat_interleave(G, dim=1)
        Q = q[c0:c0 + n]
        i = torch.arange(n)[:, None]
        j = torch.arange(N)[None, :]
        mask = (j <= N - n + i) if w.causal else torch.ones(n, N, dtype=torch.bool)
        o = F.scaled_dot_product_attention(Q.transpose(0, 1), K.transpose(0, 1),
                                           V.transpose(0, 1), attn_mask=mask, scale=w.scale)
        out[c0:c0 + n] = o.transpose(0, 1)
    return out.numpy()


@pytest.mark.parametrize("case", [c for c in SMALL_CASES if not c.get("with_sinks")],
                         ids=lambda c: f"seed{c['seed']}")
def test_oracle_matches_torch_sdpa_fp64(case):
    w = wl.random_small(**case)
    assert np.max(np.abs(attention_of(w) - _sdpa_reference(w))) < 1e-12


def test_sink_equals_extra_key_with_zero_value():
    """A sink logit behaves as one more key whose score is the sink and whose
    value vector is zero.  MHA (each q head owns its kv head) lets us build, per
    head, a key k = q * sink / (scale * |q|^2) that reproduces the logit."""
    rng = np.random.default_rng(7)
    H, D, N, bs = 3, 16, 21, 8
    q = rng.standard_normal((1, H, D))
    k = rng.standard_normal((N, H, D))
    v = rng.standard_normal((N, H, D))
    sinks = rng.standard_normal(H) * 2
    scale = 0.3
    base = wl.build("sink", wl.F32, H, H, D, bs, [N - 1], [1], seed=0, poison=False)
    base.q = q.astype(np.float32)
    kx = np.concatenate([k, np.zeros((1, H, D))])
    vx = np.concatenate([v, np.zeros((1, H, D))])
    for h in range(H):
        qh = base.q[0, h].astype(np.float64)
        kx[N, h] = qh * sinks[h] / (scale * qh @ qh)
    kx = kx.astype(np.float32); vx = vx.astype(np.float32)

    def pools(kk, vv, n_keys):
        pages = (n_keys + bs - 1) // bs
        kc = np.zeros((pages, bs, H, D), np.float32); vc = np.zeros_like(kc)
        pos = np.arange(n_keys)
        kc[pos // bs, pos % bs] = kk[:n_keys]; vc[pos // bs, pos % bs] = vv[:n_keys]
        return kc, vc, np.arange(pages, dtype=np.int32)[None, :]

    common = dict(dtype=wl.F32, num_q_heads=H, num_kv_heads=H, head_dim=D, block_size=bs,
                  scale=scale, causal=True)
    kc, vc, bt = pools(kx, vx, N)
    with_sink = oracle.paged_attention(base.q, kc, vc, [0, 1], [N], bt, sinks=sinks, **common)
    kc, vc, bt = pools(kx, vx, N + 1)
    extra_key = oracle.paged_attention(base.q, kc, vc, [0, 1], [N + 1], bt, **common)
    assert np.max(np.abs(with_sink - extra_key)) < 1e-6   # k rounded to float32


def test_sink_to_minus_infinity_is_no_sink():
    w = wl.random_small(11, dtype=wl.F32, with_sinks=True)
    a = attention_of(w, sinks=np.full(w.num_q_heads, -1e30))
    b = attention_of(w, sinks=None)
    assert np.max(np.abs(a - b)) < 1e-15


def test_sink_scales_output_by_key_mass():
    """With a sink, out = out_nosink * Z / (Z + e^sink) where Z is the key mass.
    With all scores zero (scale 0), Z = number of visible keys."""
    w = wl.random_small(12, dtype=wl.F32, num_seqs=2, max_q=1, with_sinks=True)
    a = attention_of(w, scale=0.0)
    b = attention_of(w, scale=0.0, sinks=None)
    for r in range(w.num_seqs):
        row = int(w.cu_seqlens_q[r]); N = int(w.seq_lens[r])
        for h in range(w.num_q_heads):
            f = N / (N + math.exp(float(w.sinks[h])))
            assert np.max(np.abs(a[row, h] - f * b[row, h])) < 1e-13


def test_all_keys_equal_gives_mean_of_visible_values():
    w = wl.random_small(13, dtype=wl.F32, max_q=6, poison=False)
    w.k_ctx[:] = w.k_ctx[0]  # every key identical
    kc, vc = w.pool_with_new_tokens()
    # rebuild pool keys from the (now identical) contiguous keys
    bs = w.block_size
    for r in range(w.num_seqs):
        for p in range(int(w.seq_lens[r])):
            kc[w.block_tables[r, p // bs], p % bs] = w.k_ctx[0]
    got = attention_of(w, key_cache=kc, value_cache=vc)
    v = w.v_ctx.astype(np.float64)
    for r in range(w.num_seqs):
        n = int(w.q_lens[r]); N = int(w.seq_lens[r]); c0 = int(w.cu_seqlens_q[r])
        for i in range(n):
            vis = N - n + i + 1
            mean = v[w.ctx_offsets[r]:w.ctx_offsets[r] + vis].mean(axis=0)  # [Hkv, D]
            for h in range(w.num_q_heads):
                assert np.max(np.abs(got[c0 + i, h] - mean[h // w.group])) < 1e-12


def test_scale_zero_gives_causal_prefix_mean():
    w = wl.random_small(14, dtype=wl.BF16, max_q=8)
    got = attention_of(w, scale=0.0)
    v = wl.to_f64(w.v_ctx, w.dtype)
    for r in range(w.num_seqs):
        n = int(w.q_lens[r]); N = int(w.seq_lens[r]); c0 = int(w.cu_seqlens_q[r])
        for i in range(n):
            mean = v[w.ctx_offsets[r]:w.ctx_offsets[r] + N - n + i + 1].mean(axis=0)
            for h in range(w.num_q_heads):
                assert np.max(np.abs(got[c0 + i, h] - mean[h // w.group])) < 1e-12


def test_single_visible_key_returns_its_value():
    """Prefill without prior context: the first row sees only key 0."""
    w = wl.build("one", wl.BF16, 4, 2, 32, 16, [0, 0], [5, 3], seed=15)
    got = attention_of(w)
    v = wl.to_f64(w.v_ctx, w.dtype)
    for r in range(2):
        c0 = int(w.cu_seqlens_q[r])
        for h in range(4):
            assert np.array_equal(got[c0, h], v[w.ctx_offsets[r], h // 2])


def test_two_key_logistic_case():
    """q = e_0, k_0 = a e_0, k_1 = 0: weights are sigma(scale*a) and 1 - sigma."""
    D, a, scale = 4, float(np.float32(1.7)), 0.9   # a as the float32 key stores it
    q = np.zeros((1, 1, D), np.float32); q[0, 0, 0] = 1.0
    kc = np.zeros((1, 2, 1, D), np.float32); kc[0, 0, 0, 0] = a
    vc = np.zeros((1, 2, 1, D), np.float32)
    vc[0, 0, 0] = [1, 2, 3, 4]; vc[0, 1, 0] = [-1, 0, 5, 0.5]
    got = oracle.paged_attention(q, kc, vc, [0, 1], [2], np.array([[0]], np.int32),
                                 dtype=wl.F32, num_q_heads=1, num_kv_heads=1, head_dim=D,
                                 block_size=2, scale=scale, causal=True)
    s = 1.0 / (1.0 + math.exp(-scale * a))
    want = s * vc[0, 0, 0].astype(np.float64) + (1 - s) * vc[0, 1, 0].astype(np.float64)
    assert np.max(np.abs(got[0, 0] - want)) < 1e-15


def test_mha_with_duplicated_kv_heads_equals_gqa():
    w = wl.random_small(16, dtype=wl.BF16, num_q_heads=6, num_kv_heads=2, head_dim=32)
    gqa = attention_of(w)
    kc, vc = w.pool_with_new_tokens()
    kc6 = np.repeat(kc, 3, axis=2); vc6 = np.repeat(vc, 3, axis=2)
    mha = attention_of(w, key_cache=kc6, value_cache=vc6, num_kv_heads=6)
    assert np.array_equal(gqa, mha)


def test_page_permutation_is_invisible():
    w = wl.random_small(17, dtype=wl.BF16, num_seqs=4)
    base = attention_of(w)
    kc, vc = w.pool_with_new_tokens()
    perm = np.random.default_rng(3).permutation(w.num_blocks)  # new page of old page p
    kc2 = np.empty_like(kc); vc2 = np.empty_like(vc)
    kc2[perm] = kc; vc2[perm] = vc
    bt2 = np.where(w.block_tables >= 0, perm[np.maximum(w.block_tables, 0)], -1).astype(np.int32)
    got = oracle.paged_attention(w.q, kc2, vc2, w.cu_seqlens_q, w.seq_lens_k, bt2,
                                 dtype=w.dtype, num_q_heads=w.num_q_heads,
                                 num_kv_heads=w.num_kv_heads, head_dim=w.head_dim,
                                 block_size=w.block_size, scale=w.scale, causal=w.causal)
    assert np.array_equal(base, got)


@pytest.mark.parametrize("big,small", [(32, 16), (144, 16), (16, 8)])
def test_block_size_translation_is_invisible(big, small):
    """A pool of big-token pages viewed as (big/small)x more small pages by a
    reshape only, with block b mapped to small blocks b*f .. b*f+f-1."""
    w = wl.random_small(18, dtype=wl.F32, block_size=big, max_prior=400, max_q=4)
    base = attention_of(w)
    kc, vc = w.pool_with_new_tokens()
    f = big // small
    kcs = kc.reshape(w.num_blocks * f, small, w.num_kv_heads, w.head_dim)
    vcs = vc.reshape(w.num_blocks * f, small, w.num_kv_heads, w.head_dim)
    bt = w.block_tables
    bts = np.full((bt.shape[0], bt.shape[1] * f), -1, np.int32)
    for r in range(bt.shape[0]):
        for b in range(bt.shape[1]):
            if bt[r, b] >= 0:
                bts[r, b * f:(b + 1) * f] = bt[r, b] * f + np.arange(f)
    got = oracle.paged_attention(w.q, kcs, vcs, w.cu_seqlens_q, w.seq_lens_k, bts,
                                 dtype=w.dtype, num_q_heads=w.num_q_heads,
                                 num_kv_heads=w.num_kv_heads, head_dim=w.head_dim,
                                 block_size=small, scale=w.scale, causal=w.causal)
    assert np.array_equal(base, got)


def test_poisoned_unwritten_slots_never_reach_output():
    wp = wl.random_small(19, dtype=wl.BF16, poison=True)
    wz = wl.random_small(19, dtype=wl.BF16, poison=False)
    a = attention_of(wp); b = attention_of(wz)
    assert np.isfinite(a).all()
    assert np.array_equal(a, b)


def test_packing_independence_and_decode_equals_last_prefill_row():
    w = wl.random_small(20, dtype=wl.F32, num_seqs=4, max_q=6)
    packed = attention_of(w)
    kc, vc = w.pool_with_new_tokens()
    for r in range(w.num_seqs):
        c0, c1 = int(w.cu_seqlens_q[r]), int(w.cu_seqlens_q[r + 1])
        alone = oracle.paged_attention(w.q[c0:c1], kc, vc, [0, c1 - c0], w.seq_lens_k[r:r + 1],
                                       w.block_tables[r:r + 1], dtype=w.dtype,
                                       num_q_heads=w.num_q_heads, num_kv_heads=w.num_kv_heads,
                                       head_dim=w.head_dim, block_size=w.block_size,
                                       scale=w.scale, causal=True)
        assert np.array_equal(alone, packed[c0:c1])
        # the last row alone as a decode row (q = 1 over the same N keys)
        dec = oracle.paged_attention(w.q[c1 - 1:c1], kc, vc, [0, 1], w.seq_lens_k[r:r + 1],
                                     w.block_tables[r:r + 1], dtype=w.dtype,
                                     num_q_heads=w.num_q_heads, num_kv_heads=w.num_kv_heads,
                                     head_dim=w.head_dim, block_size=w.block_size,
                                     scale=w.scale, causal=True)
        assert np.array_equal(dec[0], packed[c1 - 1])


def test_no_visible_key_gives_zeros():
    # more query rows than keys under bottom-right alignment: the first rows see nothing
    w = wl.build("empty", wl.F32, 2, 1, 8, 8, [0], [3], seed=21, with_sinks=True)
    w.seq_lens_k = np.array([1], np.int32)
    got = attention_of(w)
    assert np.array_equal(got[:2], np.zeros_like(got[:2]))
    assert np.isfinite(got).all()


@pytest.mark.parametrize("P", [16, 256, 512, 48])
def test_split_kv_equals_no_split(P):
    w = wl.random_small(22, dtype=wl.BF16, num_seqs=5, max_prior=1300, max_q=1,
                        with_sinks=True, head_dim=32)
    kc, vc = w.pool_with_new_tokens()
    max_parts = int(math.ceil(w.max_seqlen_k / P))
    po, pm, pl = oracle.split_partials(w.q, kc, vc, w.cu_seqlens_q, w.seq_lens_k, w.block_tables,
                                       dtype=w.dtype, num_q_heads=w.num_q_heads,
                                       num_kv_heads=w.num_kv_heads, head_dim=w.head_dim,
                                       block_size=w.block_size, scale=w.scale,
                                       partition_size=P, max_parts=max_parts)
    out = oracle.split_combine(po, pm, pl, w.cu_seqlens_q, w.seq_lens_k, partition_size=P,
                               sinks=w.sinks)
    ref = attention_of(w)
    assert np.max(np.abs(out - ref)) < 1e-12


def test_split_partials_single_key_closed_form_and_bounds():
    """Trick 4's partials by their definition: m_p is the partition's log2-domain
    max, so the largest term is 2^0 = 1 and 1 <= l_p <= (keys in the partition);
    a partition holding one key has l_p = 1 exactly and o_p = that key's value row.
    (The combined output alone cannot pin the units of m_p: any reference max
    with its matching exp-sum combines to the same result.)"""
    P = 64
    prior = np.array([2 * P, P, 3 * P - 1, 0], dtype=np.int64)   # N = 2P+1, P+1, 3P, 1
    w = wl.build("partials", wl.F32, 4, 2, 32, 16, prior, np.ones(4, np.int64), seed=31,
                 partition_size=P)
    kc, vc = w.pool_with_new_tokens()
    max_parts = int(math.ceil(w.max_seqlen_k / P))
    po, pm, pl = oracle.split_partials(w.q, kc, vc, w.cu_seqlens_q, w.seq_lens_k, w.block_tables,
                                       dtype=w.dtype, num_q_heads=w.num_q_heads,
                                       num_kv_heads=w.num_kv_heads, head_dim=w.head_dim,
                                       block_size=w.block_size, scale=w.scale,
                                       partition_size=P, max_parts=max_parts)
    v_all = wl.to_f64(w.v_ctx, w.dtype)
    single = 0
    for r in range(w.num_seqs):
        N = int(w.seq_lens[r])
        for p in range((N + P - 1) // P):
            n_p = min(N, (p + 1) * P) - p * P
            for h in range(w.num_q_heads):
                assert 1.0 - 1e-12 <= pl[r, p, h] <= n_p + 1e-12
                if n_p == 1:
                    assert pl[r, p, h] == 1.0
                    v = v_all[w.ctx_offsets[r] + p * P, h // w.group]
                    assert np.max(np.abs(po[r, p, h] - v)) < 1e-12
                    single += 1
    assert single == 3 * w.num_q_heads


def test_scatter_is_byte_exact_and_keeps_untouched_slots():
    w = wl.random_small(23, dtype=wl.BF16, num_seqs=4, max_q=7)
    sm = w.slot_mapping.copy()
    sm[1] = -1  # a padding token
    kc, vc = oracle.reshape_and_cache(w.new_k, w.new_v, w.key_cache, w.value_cache, sm,
                                      w.block_size)
    ek = w.key_cache.copy(); ev = w.value_cache.copy()
    bs = w.block_size
    for t, s in enumerate(sm):
        if s >= 0:
            ek[s // bs, s % bs] = w.new_k[t]; ev[s // bs, s % bs] = w.new_v[t]
    assert np.array_equal(kc.view(np.uint16), ek.view(np.uint16))
    assert np.array_equal(vc.view(np.uint16), ev.view(np.uint16))
    # the padding token's slot still holds its old (poison) bits
    s1 = w.slot_mapping[1]
    assert np.array_equal(kc[s1 // bs, s1 % bs].view(np.uint16),
                          w.key_cache[s1 // bs, s1 % bs].view(np.uint16))


SCATTER_PIN_CASES = [
    # prompt-only: every key of every request reaches the pool through the scatter
    dict(seed=41, dtype=wl.BF16, head_dim=64, num_q_heads=4, num_kv_heads=2, block_size=16,
         num_seqs=4, prior=0, max_q=40),
    dict(seed=42, dtype=wl.F32, head_dim=32, num_q_heads=6, num_kv_heads=3, block_size=8,
         num_seqs=3, prior=0, max_q=30),
    # prior context already in the pool, this step's tokens through the scatter
    dict(seed=43, dtype=wl.BF16, head_dim=64, num_q_heads=8, num_kv_heads=1, block_size=32,
         num_seqs=5, prior=90, max_q=12),
]


@pytest.mark.parametrize("case", SCATTER_PIN_CASES, ids=lambda c: f"seed{c['seed']}")
def test_scatter_then_attention_equals_dense_bruteforce(case):
    """The oracle's scatter pinned by what attention reads back: a poisoned pool
    (every slot NaN) receives this step's K/V rows only through
    oracle.reshape_and_cache; oracle attention over it must equal dense
    attention on the unpaged per-request K/V.  A row scattered to the wrong page
    or slot, or a token dropped, leaves a NaN or a wrong key where attention
    reads, so the pin fails (kwkr.cn kernel table: reshape_and_cache writes the
    rows attention then gathers through the block table)."""
    c = dict(case)
    prior_max, max_q = c.pop("prior"), c.pop("max_q")
    rng = np.random.default_rng(c["seed"])
    S = c.pop("num_seqs")
    prior = rng.integers(0, prior_max, size=S, endpoint=True) if prior_max else np.zeros(S, int)
    q = rng.integers(1, max_q, size=S, endpoint=True)
    seed = c.pop("seed")
    w = wl.build(f"scatter_pin_{seed}", c.pop("dtype"), c.pop("num_q_heads"),
                 c.pop("num_kv_heads"), c.pop("head_dim"), c.pop("block_size"), prior, q,
                 seed=seed, pool_slack=1.5, poison=True)
    assert not c
    kc, vc = oracle.reshape_and_cache(w.new_k, w.new_v, w.key_cache, w.value_cache,
                                      w.slot_mapping, w.block_size)
    got = attention_of(w, key_cache=kc, value_cache=vc)
    assert np.isfinite(got).all()
    assert np.max(np.abs(got - dense_bruteforce(w))) < 1e-12
    # without the scatter the poisoned slots reach attention: the pin can fail
    bad = attention_of(w, key_cache=w.key_cache, value_cache=w.value_cache)
    assert not np.isfinite(bad).all()


def test_scatter_rejects_slot_outside_pool():
    w = wl.random_small(24, dtype=wl.F32)
    sm = w.slot_mapping.copy(); sm[0] = w.num_blocks * w.block_size
    with pytest.raises(ValueError):
        oracle.reshape_and_cache(w.new_k, w.new_v, w.key_cache, w.value_cache, sm, w.block_size)


def test_bf16_rounding_of_inputs_is_nearest_even():
    x = np.array([1.0, 1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, -2.5, 3.0e38], np.float32)
    b = wl.f32_to_bf16_bits(x)
    back = wl.bf16_bits_to_f32(b)
    assert back[0] == 1.0
    assert back[1] == 1.0                  # tie -> even (down)
    assert back[2] == 1.0 + 2 ** -6        # tie -> even (up)
    assert back[3] == -2.5
    assert np.isfinite(back[4])


def test_oracle_reproduces_stored_tiny_decode_golden():
    """Regression pin: the stored values were written by tests/golden/make_golden.py
    (oracle only).  Any later change to the oracle's arithmetic shows up here."""
    import json
    import os
    path = os.path.join(os.path.dirname(__file__), "golden", "tiny_decode_f32.json")
    g = json.load(open(path))
    w = wl.workload(0)
    assert w.block_tables.tolist() == g["block_tables"]
    assert abs(float(np.asarray(w.q, np.float64).sum()) - g["q_checksum"]) < 1e-9
    out = attention_of(w)
    assert np.max(np.abs(out.ravel() - np.array(g["out"]))) < 1e-13
