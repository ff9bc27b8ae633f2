"""Seeded synthetic inputs for paged varlen attention.

This module only *builds inputs*: request lengths, a shuffled page pool with
per-request block tables, packed queries, K/V rows and sink logits.  It holds
none of the attention arithmetic, so both the CUDA path and the CPU oracle can
consume what it produces without sharing any of the method's code.

Input recipe (one ``numpy.random.Generator(PCG64(seed))`` per workload, drawn in
this fixed order): request lengths -> page permutation -> Q -> K -> V -> sinks.
Values are N(0, 1) float32; for bf16 workloads they are rounded to bf16 on the
host (round to nearest, ties to even), so every consumer sees identical bits.

Layouts (matching the library's C ABI):
  q            [total_q, H_q, D]                 packed query rows
  key_cache    [num_blocks, block_size, H_kv, D] page pool (K); value_cache alike
  new_k/new_v  [total_q, H_kv, D]                this step's K/V rows, scattered
                                                 into the pool via slot_mapping
  cu_seqlens_q [num_seqs + 1] int32, seq_lens_k [num_seqs] int32 (includes this
  step's tokens), block_tables [num_seqs, max_blocks_per_seq] int32 (-1 padded),
  slot_mapping [total_q] int64 = page * block_size + offset.

Pool slots that no request owns, and the slots that this step's scatter has not
yet written, hold NaN bit patterns ("poison") unless ``poison=False``.

The five named workloads follow the shapes of the pages' workloads (a decode
batch, a GQA decode batch, a varlen prefill with one long prompt, a mixed packed
step with decode / speculative-verify / chunked-prefill rows, and long-context
decode with attention sinks); the seed of workload ``c`` is ``1000 + c``.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional

import numpy as np

F32 = "f32"
BF16 = "bf16"

# Bit patterns used to poison pool slots that must never reach an output.
_POISON_F32 = np.uint32(0x7FC00000)
_POISON_BF16 = np.uint16(0x7FC0)


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bf16 (nearest, ties to even); return uint16 bits."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    nan = (u & 0x7FFFFFFF) > 0x7F800000
    lsb = (u >> 16) & 1
    r = ((u.astype(np.uint64) + 0x7FFF + lsb) >> 16).astype(np.uint16)
    r[nan] = _POISON_BF16
    return r


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns to float32."""
    return (np.ascontiguousarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def to_f64(arr: np.ndarray, dtype: str) -> np.ndarray:
    """Values of a stored array (float32, or bf16 bits as uint16) as float64."""
    if dtype == BF16:
        return bf16_bits_to_f32(arr).astype(np.float64)
    return np.asarray(arr, dtype=np.float32).astype(np.float64)


def elem_bytes(dtype: str) -> int:
    return 2 if dtype == BF16 else 4


@dataclasses.dataclass
class Workload:
    name: str
    dtype: str
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    block_size: int
    num_blocks: int
    prior_lens: np.ndarray          # [S] int64: context already in the pool
    q_lens: np.ndarray              # [S] int64: this step's query tokens
    scale: float
    causal: bool
    partition_size: int             # 0 auto, -1 no split, 256/512 forced
    # arrays (filled by build)
    q: np.ndarray = None
    key_cache: np.ndarray = None
    value_cache: np.ndarray = None
    new_k: np.ndarray = None
    new_v: np.ndarray = None
    slot_mapping: np.ndarray = None
    cu_seqlens_q: np.ndarray = None
    seq_lens_k: np.ndarray = None
    block_tables: np.ndarray = None
    sinks: Optional[np.ndarray] = None
    # unpaged copies: per-request contiguous K/V over all N positions
    k_ctx: np.ndarray = None        # [sum N, H_kv, D] stored dtype
    v_ctx: np.ndarray = None
    ctx_offsets: np.ndarray = None  # [S + 1] int64 offsets into k_ctx/v_ctx

    @property
    def num_seqs(self) -> int:
        return int(len(self.q_lens))

    @property
    def total_q(self) -> int:
        return int(self.q_lens.sum())

    @property
    def seq_lens(self) -> np.ndarray:
        return self.prior_lens + self.q_lens

    @property
    def max_seqlen_q(self) -> int:
        return int(self.q_lens.max()) if self.num_seqs else 0

    @property
    def max_seqlen_k(self) -> int:
        return int(self.seq_lens.max()) if self.num_seqs else 0

    @property
    def max_blocks_per_seq(self) -> int:
        return int(self.block_tables.shape[1])

    @property
    def group(self) -> int:
        return self.num_q_heads // self.num_kv_heads

    def kv_bytes_read(self) -> int:
        """K and V bytes one attention call must read: every context token once
        per kv head (for the decode rows, the whole context)."""
        e = elem_bytes(self.dtype)
        return int(self.seq_lens.sum()) * self.num_kv_heads * self.head_dim * e * 2

    def pool_with_new_tokens(self):
        """Pool arrays with this step's K/V placed at their slots: the state the
        cache is in after the scatter.  Used to give a kernel-only test an
        already-populated cache."""
        kc = self.key_cache.copy()
        vc = self.value_cache.copy()
        bs = self.block_size
        for t, slot in enumerate(self.slot_mapping):
            if slot < 0:
                continue
            kc[slot // bs, slot % bs] = self.new_k[t]
            vc[slot // bs, slot % bs] = self.new_v[t]
        return kc, vc

    def all_tokens(self):
        """Every context token of the batch as one step's input: K and V rows
        [T, H_kv, D] in request and position order (the prior context read back
        out of the pool, then this step's new rows) with their slots [T].  A
        cache in another format (the quantised one) is filled from these, so
        that it holds the same context as ``key_cache`` after this step."""
        kc, vc = self.pool_with_new_tokens()
        bs = self.block_size
        slots = []
        for r in range(self.num_seqs):
            pages = self.block_tables[r]
            for pos in range(int(self.seq_lens[r])):
                slots.append(int(pages[pos // bs]) * bs + pos % bs)
        slots = np.asarray(slots, dtype=np.int64)
        return kc[slots // bs, slots % bs], vc[slots // bs, slots % bs], slots


def _normal(rng: np.random.Generator, shape, dtype: str) -> np.ndarray:
    x = rng.standard_normal(size=shape, dtype=np.float32)
    return f32_to_bf16_bits(x) if dtype == BF16 else x


def build(name: str, dtype: str, num_q_heads: int, num_kv_heads: int, head_dim: int,
          block_size: int, prior_lens, q_lens, *, seed: int, num_blocks: Optional[int] = None,
          pool_slack: float = 1.0, scale: Optional[float] = None, causal: bool = True,
          with_sinks: bool = False, partition_size: int = 0, poison: bool = True,
          rng: Optional[np.random.Generator] = None) -> Workload:
    """Build one workload.  ``rng`` (if given) has already drawn the lengths;
    otherwise a fresh PCG64(seed) is used and the lengths are taken as given."""
    if rng is None:
        rng = np.random.Generator(np.random.PCG64(seed))
    prior_lens = np.asarray(prior_lens, dtype=np.int64)
    q_lens = np.asarray(q_lens, dtype=np.int64)
    S = len(q_lens)
    N = prior_lens + q_lens
    bs = block_size
    pages_per_seq = (N + bs - 1) // bs
    need = int(pages_per_seq.sum())
    if num_blocks is None:
        num_blocks = max(1, int(math.ceil(need * pool_slack)))
    if need > num_blocks:
        raise ValueError(f"pool of {num_blocks} pages cannot hold {need} pages")
    mbps = max(1, int(pages_per_seq.max()) if S else 1)

    # page permutation -> block tables (each request owns distinct random pages)
    perm = rng.permutation(num_blocks).astype(np.int32)
    block_tables = np.full((S, mbps), -1, dtype=np.int32)
    off = 0
    for r in range(S):
        n_p = int(pages_per_seq[r])
        block_tables[r, :n_p] = perm[off:off + n_p]
        off += n_p

    Hq, Hkv, D = num_q_heads, num_kv_heads, head_dim
    total_q = int(q_lens.sum())
    q = _normal(rng, (total_q, Hq, D), dtype)
    ctx_offsets = np.zeros(S + 1, dtype=np.int64)
    ctx_offsets[1:] = np.cumsum(N)
    k_ctx = _normal(rng, (int(N.sum()), Hkv, D), dtype)
    v_ctx = _normal(rng, (int(N.sum()), Hkv, D), dtype)
    sinks = rng.standard_normal(size=Hq, dtype=np.float32) if with_sinks else None

    store = np.uint16 if dtype == BF16 else np.float32
    poison_bits = _POISON_BF16 if dtype == BF16 else _POISON_F32
    shape = (num_blocks, bs, Hkv, D)
    if poison:
        if dtype == BF16:
            key_cache = np.full(shape, poison_bits, dtype=np.uint16)
        else:
            key_cache = np.full(shape, poison_bits, dtype=np.uint32).view(np.float32)
    else:
        key_cache = np.zeros(shape, dtype=store)
    value_cache = key_cache.copy()

    new_k = np.empty((total_q, Hkv, D), dtype=store)
    new_v = np.empty((total_q, Hkv, D), dtype=store)
    slot_mapping = np.empty(total_q, dtype=np.int64)
    cu = np.zeros(S + 1, dtype=np.int32)
    cu[1:] = np.cumsum(q_lens)
    t = 0
    for r in range(S):
        base = int(ctx_offsets[r])
        n_prior = int(prior_lens[r])
        if n_prior:
            pos = np.arange(n_prior)
            pages = block_tables[r, pos // bs]
            key_cache[pages, pos % bs] = k_ctx[base:base + n_prior]
            value_cache[pages, pos % bs] = v_ctx[base:base + n_prior]
        for j in range(int(q_lens[r])):
            p = n_prior + j
            slot_mapping[t] = int(block_tables[r, p // bs]) * bs + p % bs
            new_k[t] = k_ctx[base + p]
            new_v[t] = v_ctx[base + p]
            t += 1

    return Workload(
        name=name, dtype=dtype, num_q_heads=Hq, num_kv_heads=Hkv, head_dim=D,
        block_size=bs, num_blocks=num_blocks, prior_lens=prior_lens, q_lens=q_lens,
        scale=float(scale if scale is not None else 1.0 / math.sqrt(D)), causal=causal,
        partition_size=partition_size, q=q, key_cache=key_cache, value_cache=value_cache,
        new_k=new_k, new_v=new_v, slot_mapping=slot_mapping, cu_seqlens_q=cu,
        seq_lens_k=N.astype(np.int32), block_tables=block_tables, sinks=sinks,
        k_ctx=k_ctx, v_ctx=v_ctx, ctx_offsets=ctx_offsets)


# ---------------------------------------------------------------------------
# The five named workloads.
# ---------------------------------------------------------------------------

WORKLOAD_NAMES = {
    0: "tiny decode fp32 (S=2, N=17/40, Hq=4 Hkv=2 D=64, bs=16, 16-page pool)",
    1: "GQA decode bf16 (S=32, N~U[512,8192], Hq=32 Hkv=8 D=128, bs=16, 40k-page pool, P=512)",
    2: "varlen causal prefill bf16 (S=8: 1x3000 + 7x~430, Hq=16 Hkv=2 D=256, bs=16)",
    3: "mixed packed step bf16 (S=64: 40 decode, 16 verify q=1+k, 8 prefill-chunk q=512; "
       "prior~U[1024,16384], Hq=32 Hkv=8 D=128, bs=16)",
    4: "long-context decode with sinks bf16 (S=16: 4x65536 + 12x~4600, Hq=24 Hkv=4 D=256, bs=32)",
}


def workload(index: int, *, partition_size: Optional[int] = None, poison: bool = True) -> Workload:
    """The named workload ``index`` (0..4) at full size."""
    seed = 1000 + index
    rng = np.random.Generator(np.random.PCG64(seed))
    if index == 0:
        w = build("tiny_decode_f32", F32, 4, 2, 64, 16, [16, 39], [1, 1], seed=seed,
                  num_blocks=16, partition_size=0, poison=poison, rng=rng)
    elif index == 1:
        n = rng.integers(512, 8192, size=32, endpoint=True)
        w = build("gqa_decode_bf16", BF16, 32, 8, 128, 16, n - 1, np.ones(32, np.int64),
                  seed=seed, num_blocks=40000, partition_size=512, poison=poison, rng=rng)
    elif index == 2:
        n = np.concatenate([[3000], rng.integers(410, 450, size=7, endpoint=True)])
        pages = int(((n + 15) // 16).sum())
        pool = max(512, int(2 ** math.ceil(math.log2(pages))))
        w = build("varlen_prefill_bf16", BF16, 16, 2, 256, 16, np.zeros(8, np.int64), n,
                  seed=seed, num_blocks=pool, partition_size=0, poison=poison, rng=rng)
    elif index == 3:
        prior = rng.integers(1024, 16384, size=64, endpoint=True)
        kinds = np.array([0] * 40 + [1] * 16 + [2] * 8)
        kinds = kinds[rng.permutation(64)]
        k_draft = rng.integers(1, 4, size=64, endpoint=True)
        q = np.where(kinds == 0, 1, np.where(kinds == 1, 1 + k_draft, 512))
        n_total = prior + q
        pages = int(((n_total + 15) // 16).sum())
        w = build("mixed_step_bf16", BF16, 32, 8, 128, 16, prior, q, seed=seed,
                  num_blocks=int(pages * 1.1) + 1, partition_size=0, poison=poison, rng=rng)
    elif index == 4:
        n = np.concatenate([np.full(4, 65536), rng.integers(4400, 4800, size=12, endpoint=True)])
        pages = int(((n + 31) // 32).sum())
        w = build("long_decode_sinks_bf16", BF16, 24, 4, 256, 32, n - 1, np.ones(16, np.int64),
                  seed=seed, num_blocks=int(math.ceil(pages * 1.25)), with_sinks=True,
                  partition_size=0, poison=poison, rng=rng)
    else:
        raise ValueError(f"no workload {index}")
    if partition_size is not None:
        w.partition_size = partition_size
    return w


def padded(w: Workload, *, seed: int = 7) -> Workload:
    """The same batch laid out padded instead of packed: every request gets
    max(q) query rows and max(N) keys (prior = max(N) - max(q)), the shape a
    padded [B, H, T_max, D] attention computes on.  The rows and keys past a
    request's own lengths are padding: the work they cost is the price of not
    packing (aisignalhub.me, "packed queries and paged KV": batch A vs B)."""
    S = w.num_seqs
    qmax = int(w.q_lens.max())
    nmax = int(w.seq_lens.max())
    pages = S * ((nmax + w.block_size - 1) // w.block_size)
    return build(w.name + "_padded", w.dtype, w.num_q_heads, w.num_kv_heads, w.head_dim,
                 w.block_size, np.full(S, nmax - qmax, np.int64), np.full(S, qmax, np.int64),
                 seed=seed, num_blocks=int(math.ceil(pages * 1.1)) + 1, causal=w.causal,
                 with_sinks=w.sinks is not None, partition_size=w.partition_size)


def random_small(seed: int, *, dtype: str = BF16, num_seqs: int = 3, num_q_heads: int = 4,
                 num_kv_heads: int = 2, head_dim: int = 64, block_size: int = 16,
                 max_prior: int = 70, max_q: int = 5, causal: bool = True,
                 with_sinks: bool = False, partition_size: int = 0, pool_slack: float = 1.5,
                 poison: bool = True) -> Workload:
    """A small random ragged workload (lengths drawn from PCG64(seed))."""
    rng = np.random.Generator(np.random.PCG64(seed))
    prior = rng.integers(0, max_prior, size=num_seqs, endpoint=True)
    q = rng.integers(1, max_q, size=num_seqs, endpoint=True)
    pages = int(((prior + q + block_size - 1) // block_size).sum())
    return build(f"random_small_{seed}", dtype, num_q_heads, num_kv_heads, head_dim, block_size,
                 prior, q, seed=seed, num_blocks=max(1, int(math.ceil(pages * pool_slack))),
                 causal=causal, with_sinks=with_sinks, partition_size=partition_size,
                 poison=poison, rng=rng)
