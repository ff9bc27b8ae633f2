// decode_tc.cuh -- single-query (decode) requests on the 5th-generation
// tensor cores, bf16.
//
// What it computes (kwkr.cn, "What is Paged Attention": the GQA decode section
// and trick 4; aisignalhub.me, "packed queries and paged KV"): for every
// decode request r and query head, softmax(scale * q K^T) V over the request's
// paged keys -- or, with the keys cut into partitions of P, one partial per
// partition (log2-domain reference max, exp-sum, normalised output) for the
// shared split-KV reduce.
//
// GB300 design (persistent: one CTA per SM, 224 threads)
//  * A work item is (request, KV head, partition).  Every CTA scans the batch
//    once, weighs each item by five per key tile plus three (item_cost; an item's fixed
//    cost -- Q load, pipeline turn, epilogue -- measured at about 0.6 tile), and
//    takes, in order, the items whose cumulative work starts inside its
//    1/gridDim share.
//  * Keys are the MMA rows: S^T[128 keys x 16] = K_tile . Q^T with the G query
//    heads of the KV head padded to N = 16, so one M = 128 MMA per 16-dim step
//    serves the whole GQA group however small G is; O^T[d x 16] += V^T . P^T
//    reads the V tile in place as an MN-major A operand.  The CUDA cores only
//    see G scores per key instead of G * D multiply-adds.
//  * Warps 4 and 7 stream the K tiles (warp 4 also Q^T once per item), warps
//    5 and 8 the V tiles, into two rings of 32 KB stages (128 keys x 128
//    dims, the tensor cores' 128-byte-swizzled layout) by TMA, one box per
//    run of box_rows keys of a page and 64-dim half; the two warps of a ring
//    each load half of every stage's page runs, one box per lane.  A 16-token
//    page holds only 2 KB of one head's K, and issuing a TMA box holds its
//    warp for ~120 ns: measured on GB300, boxes this small reach ~15 GB/s per
//    SM from one lane of one warp, ~26 from eight lanes, ~52 from two warps of
//    eight lanes.  The page ids of each tile reach shared memory by 4-byte
//    cp.async three tiles ahead and the next request's lengths are loaded a
//    request ahead, so the producers never wait on a load.
//  * Warp 6 (MMA) allocates TMEM, issues S^T into one of two TMEM buffers and
//    O^T into the accumulator of the item's parity; commits release stages.
//  * Warps 0-3 (one thread per key = TMEM lane): scale S^T into the log2
//    domain, take each head's tile max across the four warps, keep a
//    reference max that moves only when the max grows by more than 2^8
//    (then O^T and the running sums are rescaled), write P^T as bf16, and at
//    the end of an item sum the exp-sums and write the output or the partial.
//    Value rows past the last key of a partial tile are zeroed before the PV
//    MMA reads them (a zero weight times a NaN pool slot would still be NaN).
//  * Programmatic dependent launch: the kernel may start while the previous
//    kernel of the stream runs.  It waits for that kernel before its first
//    global read -- or, after this step's scatter (which writes only the new
//    K/V rows), only before the K/V loads, so its setup, work plan and first
//    page ids overlap the scatter -- and lets the next kernel (the reduce)
//    be scheduled from its start.
//  * Every barrier wait is bounded (pa::mbar_wait_ool); nothing spins forever.
//    The waits' retry loop is out of line, one copy for all wait sites: the
//    smaller code (114 -> 105 KB) measured 107.4 -> 104.0 us on the GQA decode
//    batch.  (Taking the item iterator or the item store out of line as well
//    was slower: their structures then live on the stack.)
#pragma once

#include <climits>

#include "pa_common.cuh"
#include "pa_internal.h"
#include "tc_common.cuh"

namespace pa {

template <int D>
struct DtcCfg {
    static constexpr int KS = D / 128;             // 128-dim chunks of a K (or V) row
    static constexpr int KCH = D / 64;             // 64-dim (128-byte) sub-chunks
    static constexpr int BN = 128;                 // keys per tile = MMA M
    static constexpr int NP = 16;                  // MMA N: query heads padded to 16
    static constexpr int SLOT = BN * 256;          // ring stage: 128 keys x 128 dims bf16
    static constexpr int SUB = BN * 128;           // one 64-dim sub-chunk of a stage
    static constexpr int NR = 3;                   // stages of the K ring and of the V ring
    static constexpr int Q_BUF = KCH * NP * 128;   // [KCH][16 rows][128 B]
    static constexpr int P_BUF = 2 * NP * 128;     // [2 key halves][16 rows][128 B]
    static constexpr int OFF_K = 0;
    static constexpr int OFF_V = NR * SLOT;
    static constexpr int OFF_Q = 2 * NR * SLOT;    // two Q^T buffers
    static constexpr int OFF_P = OFF_Q + 2 * Q_BUF;   // two P^T buffers
    static constexpr int OFF_BAR = OFF_P + 2 * P_BUF;
    static constexpr int NBAR = 4 * NR + 7 * 2;
    static constexpr int OFF_RED = OFF_BAR + NBAR * 8;   // float [2][4][8] max, [2][4][8] sum
    static constexpr int PGR = 4;                  // page-id ring of each producer (tiles)
    static constexpr int OFF_PG = OFF_RED + 2 * 2 * 4 * 8 * 4;   // int [4 producers][PGR][16]
    static constexpr int OFF_MISC = OFF_PG + 4 * PGR * 16 * 4;
    // 4 softmax warps, 2 K and 2 V producer warps, the MMA warp
    static constexpr int THREADS = 288;
    // batches of at most THREADS requests: their cu_seqlens_q and seq_lens_k,
    // read once by the work-plan scan
    static constexpr int OFF_LENS = OFF_MISC + 192;   // int [THREADS + 1] cu, int [THREADS] sl
    static constexpr int SMEM_BYTES = OFF_LENS + (2 * THREADS + 4) * 4 + 1024;   // + alignment slack
    static constexpr int S_COL = 0;                // two S^T buffers of NP columns
    static constexpr int O_COL = 2 * NP;           // two O^T accumulators of KS * NP columns
    static constexpr int TMEM_COLS = 128;
    static_assert(O_COL + 2 * KS * NP <= TMEM_COLS, "TMEM columns");
    static_assert(SMEM_BYTES <= 227 * 1024, "shared memory");
    static_assert(OFF_Q % 1024 == 0 && OFF_P % 1024 == 0 && Q_BUF % 1024 == 0, "swizzle atoms");
};

// Work of one decode request: its (partition, KV head) items, ordered
// partition-major, each weighed by five per key tile plus a.item_cost.
struct DtcReq {
    int items;   // 0 when the request has no decode work here
    int np;      // partitions
    int N;       // keys
    int wfull;   // work of an item of a full partition
    int wlast;   // work of an item of the last partition
};

// c0, c1 = cu_seqlens_q[r], cu_seqlens_q[r + 1]; sl = seq_lens_k[r]
__device__ __forceinline__ DtcReq dtc_request_from(const DecodeTcArgs &a, int c0, int c1, int sl) {
    DtcReq q = {0, 0, 0, 0, 0};
    if (c1 - c0 != 1) return q;                       // multi-query request: other kernel
    int N = max(0, min(sl, a.max_blocks_per_seq * a.block_size));
    q.N = N;
    const int P = a.partition_size;
    if (P > 0) {
        // partials exist for max_parts partitions only (the reduce reads no more)
        N = min(N, a.max_parts * P);
        q.N = N;
        q.np = (N + P - 1) / P;
        if (q.np == 0) return q;                      // no keys: the reduce writes zeros
        q.wfull = 5 * ((P + 127) / 128) + a.item_cost;
        q.wlast = 5 * ((N - (q.np - 1) * P + 127) / 128) + a.item_cost;
    } else {
        q.np = 1;                                     // one item, even with no keys
        q.wfull = q.wlast = 5 * ((N + 127) / 128) + a.item_cost;
    }
    q.items = q.np * a.num_kv_heads;
    return q;
}

__device__ __forceinline__ DtcReq dtc_request(const DecodeTcArgs &a, int r) {
    return dtc_request_from(a, a.cu_seqlens_q[r], a.cu_seqlens_q[r + 1], a.seq_lens_k[r]);
}

__device__ __forceinline__ int64_t dtc_work(const DtcReq &q, int hkv) {
    return q.items == 0 ? 0 : ((int64_t)(q.np - 1) * q.wfull + q.wlast) * hkv;
}

// A position in the CTA's sequence of items.  The next request's lengths are
// loaded when a request is entered, so moving on never waits for memory.
struct DtcIter {
    int r, k;          // request, item index inside the request
    int64_t s;         // cumulative work before the item
    DtcReq q;
    int h, p, k0, k1, ntiles;
    int64_t row;       // the request's packed query row (cu_seqlens_q[r])
    int cu1;           // cu_seqlens_q[r + 1]
    int pf_cu, pf_sl;  // cu_seqlens_q[r + 2], seq_lens_k[r + 1] (in flight)
};

__device__ __forceinline__ void dtc_enter(const DecodeTcArgs &a, DtcIter &it, int r, int c0,
                                          int c1, int sl) {
    it.r = r;
    it.row = c0;
    it.cu1 = c1;
    it.q = dtc_request_from(a, c0, c1, sl);
    if (r + 1 < a.num_seqs) {
        it.pf_cu = __ldg(a.cu_seqlens_q + r + 2);
        it.pf_sl = __ldg(a.seq_lens_k + r + 1);
    }
}

// dtc_enter with the next request's lengths already known.
__device__ __forceinline__ void dtc_enter_from(const DecodeTcArgs &a, DtcIter &it, int r, int c0,
                                               int c1, int sl, int pf_cu, int pf_sl) {
    it.r = r;
    it.row = c0;
    it.cu1 = c1;
    it.q = dtc_request_from(a, c0, c1, sl);
    it.pf_cu = pf_cu;
    it.pf_sl = pf_sl;
}

// The CTA's share of the items cut at tile boundaries: its first item (start
// s_lo) begins at tile j_lo, and the item starting at s_hi is run up to tile
// j_hi (exclusive) when j_hi > 0 -- the next CTA runs the rest of it.
struct DtcCut {
    int64_t s_lo, s_hi;
    int j_lo, j_hi;
};

__device__ __forceinline__ void dtc_fill(const DecodeTcArgs &a, DtcIter &it, const DtcCut &cut) {
    it.p = it.k / a.num_kv_heads;
    it.h = it.k - it.p * a.num_kv_heads;
    if (a.partition_size > 0) {
        it.k0 = it.p * a.partition_size;
        it.k1 = min(it.q.N, it.k0 + a.partition_size);
    } else {
        it.k0 = 0;
        it.k1 = it.q.N;
    }
    it.ntiles = (it.k1 - it.k0 + 127) / 128;
    const int j1 = it.s == cut.s_hi ? min(it.ntiles, cut.j_hi) : it.ntiles;
    const int j0 = it.s == cut.s_lo ? cut.j_lo : 0;
    if (j0 > 0 || j1 < it.ntiles) {
        it.k1 = min(it.k1, it.k0 + j1 * 128);
        it.k0 += j0 * 128;
        it.ntiles = max(0, j1 - j0);
    }
}

__device__ __forceinline__ void dtc_next(const DecodeTcArgs &a, DtcIter &it, const DtcCut &cut) {
    it.s += (it.k < (it.q.np - 1) * a.num_kv_heads) ? it.q.wfull : it.q.wlast;
    if (++it.k >= it.q.items) {
        it.k = 0;
        do {
            const int r = it.r + 1;
            if (r >= a.num_seqs) {
                it.r = r;
                return;
            }
            dtc_enter(a, it, r, it.cu1, it.pf_cu, it.pf_sl);
        } while (it.q.items == 0);
    }
    dtc_fill(a, it, cut);
}

// Where the share boundary at offset `off` (0 <= off < the request's work)
// cuts request q's items: the upper side starts at item k (returned), tile
// *j (in [0, tiles of k)), *start being item k's start; k == q.items when the
// boundary falls at the request's end.  With split partials an item of two or
// more tiles is cut at the tile boundary nearest to `off` (items weigh five
// per tile plus item_cost); otherwise an item goes whole to the side its start
// lies on.
__device__ __forceinline__ int dtc_cut(const DtcReq &q, int hkv, int item_cost, bool split,
                                       int64_t off, int *j, int64_t *start) {
    const int64_t nf = (int64_t)(q.np - 1) * hkv;   // items of full partitions
    const int64_t wf = nf * q.wfull;
    int64_t k, st;
    int w;
    if (off < wf) {
        k = off / q.wfull;
        st = k * q.wfull;
        w = q.wfull;
    } else {
        k = nf + (off - wf) / q.wlast;
        st = wf + (k - nf) * q.wlast;
        w = q.wlast;
    }
    const int n = (w - item_cost) / 5;   // the item's tiles
    int jj;
    if (split && n >= 2) jj = (int)(((off - st) * 2 * n + w) / (2 * w));   // nearest boundary
    else jj = off == st ? 0 : n;
    if (jj >= n && off != st) {   // the whole item stays below the boundary
        st += w;
        ++k;
        jj = 0;
    }
    *j = jj;
    *start = st;
    return (int)k;
}

// Inclusive scan over the block's threads; *total = the block's sum.
template <int NT>
__device__ __forceinline__ int64_t dtc_block_scan(int64_t v, long long *scratch, int64_t *total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    long long x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const long long y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) scratch[warp] = x;
    __syncthreads();
    long long before = 0, tot = 0;
#pragma unroll
    for (int w = 0; w < NT / 32; ++w) {
        const long long t = scratch[w];
        if (w < warp) before += t;
        tot += t;
    }
    __syncthreads();   // scratch is reused by the next scan
    *total = tot;
    return x + before;
}

// Shared-memory records of a CTA's share of the batch: written by
// dtc_plan_share, read by dtc_first_item.
struct DtcPlanSmem {
    int *lens_cu;         // [NT + 1] cu_seqlens_q when num_seqs <= NT
    int *lens_sl;         // [NT] seq_lens_k when num_seqs <= NT
    int *plan_rk;         // [4] first item (request, index); cut item (request, index)
    long long *plan_s;    // [2] s_lo, s_hi
    int *plan_j;          // [2] j_lo, j_hi
    long long *scratch;   // [NT / 32] block-scan scratch
};

// Every thread of the CTA (NT threads) calls it; the records in `ps` are
// complete after the CTA's next __syncthreads.  Expects ps.plan_rk[0] = S,
// plan_rk[1] = 0, plan_rk[2] = -1, plan_rk[3] = 0, plan_s = {0, INT64_MAX},
// plan_j = {0, 0} set before the call.
template <int NT>
__device__ __forceinline__ void dtc_plan_share(const DecodeTcArgs &a, const DtcPlanSmem &ps) {
    const int tid = threadIdx.x;
    const int S = a.num_seqs;
    const int hkv = a.num_kv_heads;
    int *lens_cu = ps.lens_cu;
    int *lens_sl = ps.lens_sl;
    int *plan_rk = ps.plan_rk;
    long long *plan_s = ps.plan_s;
    int *plan_j = ps.plan_j;
    long long *scratch = ps.scratch;
    // ---- this CTA's share [lo, hi) of the batch's cumulative work, cut at
    // tile boundaries (see dtc_cut): the request containing lo (resp. hi)
    // records where the share starts (ends).  With at most THREADS requests
    // one pass suffices: thread r reads request r's lengths once (kept in
    // shared memory for the iterators), one block scan gives every request's
    // cumulative work and the total.
    const bool one_pass = S <= NT;
    const bool split = a.partition_size > 0;
    {
        int64_t acc = 0;
        DtcReq q1 = {0, 0, 0, 0, 0};
        if (one_pass) {
            if (tid < S) {
                const int c0 = a.cu_seqlens_q[tid], c1 = a.cu_seqlens_q[tid + 1];
                const int sl = a.seq_lens_k[tid];
                lens_cu[tid] = c0;
                lens_sl[tid] = sl;
                if (tid == S - 1) lens_cu[S] = c1;
                q1 = dtc_request_from(a, c0, c1, sl);
                acc = dtc_work(q1, hkv);
            }
        } else {
            for (int r = tid; r < S; r += NT) acc += dtc_work(dtc_request(a, r), hkv);
        }
        int64_t W;
        const int64_t incl = dtc_block_scan<NT>(acc, scratch, &W);   // (orders setup writes)
        const int64_t nb = gridDim.x, b = blockIdx.x;
        const int64_t lo = (W / nb) * b + (W % nb) * b / nb;
        const int64_t hi = (W / nb) * (b + 1) + (W % nb) * (b + 1) / nb;
        // Items are cut between CTAs only when a share holds fewer than ten
        // full-partition items: whole items then leave the shares up to ~5 %
        // apart, while a cut starts the next CTA mid-item, out of step with
        // the others' item boundaries -- measured on GB300 to cost ~8 % of a
        // GQA decode batch of 4-tile items, and to gain ~3.5 % on a batch of
        // 8-tile items at 8 items per CTA.
        const bool cut_items =
            split && W / nb < 10 * (5 * (int64_t)((a.partition_size + 127) / 128) + a.item_cost);
        // request r (cumulative work E, total w) containing lo or hi; the one
        // containing lo also warms L2 with the block-table entries of the first
        // tiles (the producers fetch them next)
        auto boundaries = [&](int r, const DtcReq &q, int64_t E, int64_t w) {
            if (q.items == 0 || lo >= hi) return;
            if (E <= lo && lo < E + w) {
                int j;
                int64_t st;
                const int k = dtc_cut(q, hkv, a.item_cost, cut_items, lo - E, &j, &st);
                plan_rk[0] = r;
                plan_rk[1] = k;
                plan_s[0] = E + st;
                plan_j[0] = j;
                if (k < q.items) {
                    const int kt0 = (split ? (k / hkv) * a.partition_size : 0) + j * 128;
                    const int b0 = kt0 / a.block_size;   // < max_blocks_per_seq: keys there
                    const int32_t *bt = a.block_tables + (int64_t)r * a.max_blocks_per_seq + b0;
                    prefetch_l2(bt);
                    if (b0 + 32 < a.max_blocks_per_seq) prefetch_l2(bt + 32);
                }
            }
            if (E <= hi && hi < E + w) {
                int j;
                int64_t st;
                const int k = dtc_cut(q, hkv, a.item_cost, cut_items, hi - E, &j, &st);
                plan_s[1] = E + st;
                plan_j[1] = j;
                if (j > 0) {
                    plan_rk[2] = r;
                    plan_rk[3] = k;
                }
            }
        };
        if (one_pass) {
            if (tid < S) boundaries(tid, q1, incl - acc, acc);
        } else {
            int64_t carry = 0;
            for (int base = 0; base < S && lo < hi && carry <= hi; base += NT) {
                const int r = base + tid;
                const DtcReq q = r < S ? dtc_request(a, r) : DtcReq{0, 0, 0, 0, 0};
                const int64_t w = dtc_work(q, hkv);
                int64_t tot;
                const int64_t E = carry + dtc_block_scan<NT>(w, scratch, &tot) - w;
                if (r < S) boundaries(r, q, E, w);
                carry += tot;
            }
        }
    }
}

// The CTA's first item and the bounds of its share (after dtc_plan_share and a
// __syncthreads); thread 0 records the item cut at the share's end in the cut
// table.  Returns an iterator with r == num_seqs when the share holds no tile.
template <int NT>
__device__ __forceinline__ DtcIter dtc_first_item(const DecodeTcArgs &a, const DtcPlanSmem &ps,
                                                  DtcCut *cut_out, int64_t *range_end) {
    const int tid = threadIdx.x;
    const int S = a.num_seqs;
    const int hkv = a.num_kv_heads;
    const bool one_pass = S <= NT;
    const bool split = a.partition_size > 0;
    const int *lens_cu = ps.lens_cu;
    const int *lens_sl = ps.lens_sl;
    const int *plan_rk = ps.plan_rk;
    const long long *plan_s = ps.plan_s;
    const int *plan_j = ps.plan_j;
    DtcCut &cut = *cut_out;
    cut.s_lo = plan_s[0];
    cut.s_hi = plan_s[1];
    cut.j_lo = plan_j[0];
    cut.j_hi = plan_j[1];
    // items: from (s_lo, tile j_lo) up to (s_hi, tile j_hi)
    *range_end = cut.s_hi + (cut.j_hi > 0 ? 1 : 0);
    DtcIter it0;
    it0.r = plan_rk[0];
    it0.k = plan_rk[1];
    it0.s = cut.s_lo;
    const bool has_work =
        it0.r < S && (cut.s_lo < cut.s_hi || (cut.s_lo == cut.s_hi && cut.j_lo < cut.j_hi));
    if (!has_work) it0.r = S;
    if (it0.r < S) {
        const int r = it0.r;
        if (one_pass) {   // the lengths of this request and the next one from shared memory
            dtc_enter_from(a, it0, r, lens_cu[r], lens_cu[r + 1], lens_sl[r],
                           r + 1 < S ? lens_cu[r + 2] : 0, r + 1 < S ? lens_sl[r + 1] : 0);
        } else {
            dtc_enter(a, it0, r, a.cu_seqlens_q[r], a.cu_seqlens_q[r + 1], a.seq_lens_k[r]);
        }
        if (it0.k >= it0.q.items) {   // the share starts with the next request
            it0.k = it0.q.items - 1;
            it0.s -= it0.q.wlast;   // (dtc_next adds the last item's weight back)
            dtc_next(a, it0, cut);
        } else {
            dtc_fill(a, it0, cut);
        }
    }
    // the table of items cut at a share's end (their first part's partial is
    // in the CTA's extra slot; the reduce merges it).  A CTA whose share holds
    // no tile writes no partial and records none.
    if (split && a.cut_tab != nullptr && tid == 0) {
        const int cr = plan_rk[2], ck = plan_rk[3];
        a.cut_tab[blockIdx.x] = has_work && cr >= 0 ? make_int4(cr, ck % hkv, ck / hkv, 0)
                                                    : make_int4(-1, 0, 0, 0);
    }
    return it0;
}

// Writes an item's result for query heads h * G .. h * G + G - 1 from the
// thread of TMEM lane t (dims t, t + 128, ...): with split partials, the
// normalised partial, exp-sum and reference max (the first part of an item cut
// at the share's end into the CTA's extra slot); otherwise the output rows,
// with the sink in the denominator.
template <int D, int G>
__device__ __forceinline__ void dtc_store_item(const DecodeTcArgs &a, const DtcIter &cur,
                                               const DtcCut &cut, int t,
                                               const float (&o)[D / 128][8], const float (&L)[G],
                                               const float (&m_ref)[G]) {
    using C = DtcCfg<D>;
    const bool split = a.partition_size > 0;
    const int Hq = a.num_q_heads;
    const int hq0 = cur.h * G;
    if (split) {
        // the first part of an item cut at the share's end goes to the
        // CTA's extra slot, every other partial to its partition's slot
        const bool tail = cur.s == cut.s_hi && cut.j_hi > 0;
        const int64_t slot0 =
            tail ? (int64_t)blockIdx.x * G
                 : ((int64_t)cur.r * a.max_parts + cur.p) * Hq + hq0;
        float *po = tail ? a.xpart_o : a.part_o;
        float *pm = tail ? a.xpart_m : a.part_m;
        float *pl = tail ? a.xpart_l : a.part_l;
#pragma unroll
        for (int g = 0; g < G; ++g) {
            const float inv = L[g] > 0.f ? 1.f / L[g] : 0.f;
#pragma unroll
            for (int c = 0; c < C::KS; ++c)
                po[(slot0 + g) * D + c * 128 + t] = o[c][g] * inv;
            if (t == g) {
                pm[slot0 + g] = m_ref[g];
                pl[slot0 + g] = L[g];
            }
        }
    } else {
        __nv_bfloat16 *orow =
            reinterpret_cast<__nv_bfloat16 *>(a.out) + (cur.row * Hq + hq0) * D;
#pragma unroll
        for (int g = 0; g < G; ++g) {
            float sc = 0.f;
            if (L[g] > 0.f) {
                if (a.sinks) {
                    const float sk2 = a.sinks[hq0 + g] * kLog2e;
                    const float M2 = fmaxf(m_ref[g], sk2);
                    const float f = exp2f(m_ref[g] - M2);
                    sc = f / (L[g] * f + exp2f(sk2 - M2));
                } else {
                    sc = 1.f / L[g];
                }
            }
#pragma unroll
            for (int c = 0; c < C::KS; ++c)
                orow[g * D + c * 128 + t] = __float2bfloat16_rn(o[c][g] * sc);
        }
    }
}

template <int D, int G>
__global__ void __launch_bounds__(288, 1)
    paged_decode_tc_kernel(const __grid_constant__ CUtensorMap qmap,
                           const __grid_constant__ CUtensorMap kmap,
                           const __grid_constant__ CUtensorMap vmap, const DecodeTcArgs a) {
    using C = DtcCfg<D>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = smem_u32(smem);
    const uint32_t kring = sbase + C::OFF_K;
    const uint32_t vring = sbase + C::OFF_V;
    const uint32_t q_smem = sbase + C::OFF_Q;
    const uint32_t p_smem = sbase + C::OFF_P;
    // barriers (each waited by its parties in order, never two phases behind)
    const uint32_t bar_k_full = sbase + C::OFF_BAR;            // [NR] K stage loaded
    const uint32_t bar_k_empty = bar_k_full + 8 * C::NR;       // [NR] K stage read
    const uint32_t bar_v_full = bar_k_empty + 8 * C::NR;       // [NR] V stage loaded
    const uint32_t bar_v_empty = bar_v_full + 8 * C::NR;       // [NR] V stage read
    const uint32_t bar_q_full = bar_v_empty + 8 * C::NR;       // [2] Q^T loaded
    const uint32_t bar_q_empty = bar_q_full + 16;              // [2] last S^T of the item done
    const uint32_t bar_s_full = bar_q_empty + 16;              // [2] S^T in TMEM
    const uint32_t bar_s_free = bar_s_full + 16;               // [2] S^T read
    const uint32_t bar_p_full = bar_s_free + 16;               // [2] P^T written
    const uint32_t bar_o_done = bar_p_full + 16;               // [2] PV that read P buffer b done
    const uint32_t bar_o_full = bar_o_done + 16;               // [2] item's last PV done
    float *red_max = reinterpret_cast<float *>(smem + C::OFF_RED);   // [2][4 warps][8]
    float *red_sum = red_max + 64;                                   // [2][4 warps][8]
    int *pgring = reinterpret_cast<int *>(smem + C::OFF_PG);         // [4][PGR][16] page ids
    uint8_t *misc = smem + C::OFF_MISC;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(misc);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(misc + 8);
    int *plan_rk = reinterpret_cast<int *>(misc + 16);               // [4] first item r, k; cut item r, k
    long long *plan_s = reinterpret_cast<long long *>(misc + 32);    // [2] s_lo, s_hi
    int *plan_j = reinterpret_cast<int *>(misc + 48);                // [2] j_lo, j_hi
    long long *scratch = reinterpret_cast<long long *>(misc + 64);   // [THREADS / 32]
    int *lens_cu = reinterpret_cast<int *>(smem + C::OFF_LENS);      // [S + 1] when S <= THREADS
    int *lens_sl = lens_cu + C::THREADS + 1;                          // [S]

    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;
    const int S = a.num_seqs;
    const int hkv = a.num_kv_heads;

    // ---------------------------------------------------------------- setup
    pdl_trigger();   // the reduce (or the next kernel) may be scheduled meanwhile
    if (tid == 0) {
        for (int s = 0; s < C::NR; ++s) {
            mbar_init(bar_k_full + 8 * s, 2);   // an expect-tx arrival per producer warp
            mbar_init(bar_k_empty + 8 * s, 1);
            mbar_init(bar_v_full + 8 * s, 2);
            mbar_init(bar_v_empty + 8 * s, 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(bar_q_full + 8 * b, 1);
            mbar_init(bar_q_empty + 8 * b, 1);
            mbar_init(bar_s_full + 8 * b, 1);
            mbar_init(bar_s_free + 8 * b, 4);
            mbar_init(bar_p_full + 8 * b, 4);
            mbar_init(bar_o_done + 8 * b, 1);
            mbar_init(bar_o_full + 8 * b, 1);
        }
        fence_barrier_init();
        *abort_flag = 0;
        plan_rk[0] = S;   // no item unless the share starts inside a request
        plan_rk[1] = 0;
        plan_rk[2] = -1;   // the item cut at the share's end
        plan_rk[3] = 0;
        plan_s[0] = 0;
        plan_s[1] = INT64_MAX;   // (the share reaches the batch's end)
        plan_j[0] = 0;
        plan_j[1] = 0;
    }
    if (warp == 6) {
        tmem_alloc(smem_u32(tmem_slot), C::TMEM_COLS);
        tmem_relinquish();
    }
    // Q^T and P^T rows past the G heads are never written: make them zero once
    // so the padded MMA columns stay finite.
    for (int i = tid; i < (2 * C::Q_BUF + 2 * C::P_BUF) / 16; i += C::THREADS)
        *reinterpret_cast<uint4 *>(smem + C::OFF_Q + 16 * i) = make_uint4(0, 0, 0, 0);
    fence_proxy_async_smem();

    // the launch may overlap the previous kernel of the stream: wait for it
    // before reading global memory (only before the K/V loads when that
    // kernel is this step's scatter)
    if (!a.after_scatter) pdl_wait();

    const DtcPlanSmem ps = {lens_cu, lens_sl, plan_rk, plan_s, plan_j, scratch};
    dtc_plan_share<C::THREADS>(a, ps);
    const bool split = a.partition_size > 0;
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    DtcCut cut;
    int64_t range_end;
    const DtcIter it0 = dtc_first_item<C::THREADS>(a, ps, &cut, &range_end);
    auto valid = [&](const DtcIter &x) { return x.r < S && x.s < range_end; };

    // one tile forward along the sequence; itx counts the non-empty items left
    auto adv = [&](DtcIter &x, int &jj, int &itx) {
        if (++jj >= x.ntiles) {
            jj = 0;
            ++itx;
            do dtc_next(a, x, cut);
            while (valid(x) && x.ntiles == 0);
        }
    };
    if (warp == 4 || warp == 5 || warp == 7 || warp == 8) {
        // ============================================================ producers
        // Warps 4 and 7 stream K (warp 4 also Q^T once per item), warps 5 and 8
        // stream V, into their ring by TMA: one box per (run of box_rows keys in
        // a page, 64-dim half); warp ph of a ring takes page runs [0, h0) (ph 0)
        // or [h0, nbox) (ph 1) of every stage.  Lanes fetch the page ids of each
        // tile into a shared ring by 4-byte cp.async three tiles ahead, so no
        // load is waited on.
        const bool is_k = warp == 4 || warp == 7;
        const int ph = warp >= 7 ? 1 : 0;
        const CUtensorMap *map = is_k ? &kmap : &vmap;
        const uint32_t ring0 = is_k ? kring : vring;
        const uint32_t bfull = is_k ? bar_k_full : bar_v_full;
        const uint32_t bempty = is_k ? bar_k_empty : bar_v_empty;
        int *pgr = pgring + ((is_k ? 0 : 2) + ph) * C::PGR * 16;
        const int bs = a.block_size;
        const int BR = a.box_rows;
        const uint64_t pol = policy_evict_first();   // every K/V byte is read once
        if (lane == 0) {
            prefetch_tensormap(map);
            if (is_k) prefetch_tensormap(&qmap);
        }
        auto fetch_pages = [&](const DtcIter &x, int jj, int t) {
            if (valid(x)) {
                const int kt = x.k0 + jj * C::BN;
                const int nbox = (min(C::BN, x.k1 - kt) + BR - 1) / BR;
                if (lane < nbox)
                    cp_async4(smem_u32(pgr + (t % C::PGR) * 16 + lane),
                              a.block_tables + (int64_t)x.r * a.max_blocks_per_seq +
                                  (kt + lane * BR) / bs);
            }
            cp_async_commit();   // one group per tile, empty or not
        };
        DtcIter cur = it0, la = it0;
        int j = 0, itn = 0, jl = 0, itl = 0;
        while (valid(cur) && cur.ntiles == 0) dtc_next(a, cur, cut);
        while (valid(la) && la.ntiles == 0) dtc_next(a, la, cut);
        for (int t = 0; t < C::PGR - 1; ++t) {
            fetch_pages(la, jl, t);
            if (valid(la)) adv(la, jl, itl);
        }
        if (a.after_scatter) pdl_wait();   // this step's K/V rows are in the caches
        int t = 0, issued = 0;
        int q_last[2] = {-1, -1};
        while (valid(cur)) {
            fetch_pages(la, jl, t + C::PGR - 1);
            if (valid(la)) adv(la, jl, itl);
            cp_async_wait<C::PGR - 1>();   // tile t's page ids have landed
            __syncwarp();
            int bad = 0;
            if (lane == 0 && is_k && ph == 0 && j == 0) {   // Q^T of the item: its G heads
                const int qb = itn & 1;
                if (itn >= 2)
                    bad = !mbar_wait_ool(bar_q_empty + 8 * qb, ((itn >> 1) - 1) & 1, a.err,
                                     abort_flag);
                if (!bad) {
                    mbar_arrive_expect_tx(bar_q_full + 8 * qb, C::KCH * G * 128);
#pragma unroll
                    for (int c = 0; c < C::KCH; ++c)
                        tma_load_3d(q_smem + qb * C::Q_BUF + c * C::NP * 128, &qmap, c * 64,
                                    cur.h * G, (int)cur.row, bar_q_full + 8 * qb, pol);
                    q_last[0] = q_last[1];
                    q_last[1] = itn;
                }
            }
            const int kt = cur.k0 + j * C::BN;
            const int nbox = (min(C::BN, cur.k1 - kt) + BR - 1) / BR;
            const int *pgt = pgr + (t % C::PGR) * 16;
            // lane 2i + hf issues the box of page run u = u0 + i, 64-dim half hf
            const int h0 = (nbox + 1) >> 1;
            const int u0 = ph ? h0 : 0, u1 = ph ? nbox : h0;
            const int u = u0 + (lane >> 1), hf = lane & 1;
            const int row0 = u < u1 ? pgt[u] * bs + (kt + u * BR) % bs : 0;
            for (int c = 0; c < C::KS; ++c) {   // the tile's 128-dim chunks
                const int idx = t * C::KS + c;
                const int slot = idx % C::NR;
                if (lane == 0 && !bad) {
                    if (idx >= C::NR)
                        bad = !mbar_wait_ool(bempty + 8 * slot, ((idx / C::NR) - 1) & 1, a.err,
                                         abort_flag);
                    if (!bad) mbar_arrive_expect_tx(bfull + 8 * slot, (u1 - u0) * BR * 256);
                }
                if (__shfl_sync(0xffffffffu, bad, 0)) break;
                if (u < u1)
                    tma_load_3d(ring0 + slot * C::SLOT + hf * C::SUB + u * BR * 128, map,
                                c * 128 + hf * 64, cur.h, row0, bfull + 8 * slot, pol);
                issued = idx + 1;
            }
            if (__shfl_sync(0xffffffffu, bad, 0)) break;
            ++t;
            adv(cur, j, itn);
        }
        cp_async_wait<0>();
        // copies in flight land before the CTA can exit (bounded)
        if (lane == 0) {
            for (int i = max(0, issued - C::NR); i < issued; ++i)
                mbar_drain(bfull + 8 * (i % C::NR), (i / C::NR) & 1, kWaitLimitCycles / 8);
            for (int i = 0; i < 2; ++i)
                if (q_last[i] >= 0 && q_last[i] >= itn - 2)
                    mbar_drain(bar_q_full + 8 * (q_last[i] & 1), (q_last[i] >> 1) & 1,
                               kWaitLimitCycles / 8);
        }
    } else if (warp == 6) {
        // ============================================================ MMA issuer
        if (lane == 0) {
            constexpr uint32_t IDESC_S = idesc_bf16_f32(128, C::NP, 0, 0);
            constexpr uint32_t IDESC_O = idesc_bf16_f32(128, C::NP, 1, 0);
            // O^T[ob] (+)= V^T . P^T for global tile g_t
            auto issue_pv = [&](int g_t, int ob, bool first, bool last) {
                const int pb = g_t & 1;
                mbar_wait_ool(bar_p_full + 8 * pb, (g_t >> 1) & 1, a.err, abort_flag);
#pragma unroll
                for (int c = 0; c < C::KS; ++c) {
                    const int idx = g_t * C::KS + c;
                    mbar_wait_ool(bar_v_full + 8 * (idx % C::NR), (idx / C::NR) & 1, a.err,
                              abort_flag);
                }
                tc_fence_after();
                const uint32_t ps = p_smem + pb * C::P_BUF;
#pragma unroll
                for (int c = 0; c < C::KS; ++c) {
                    const int idx = g_t * C::KS + c;
                    const uint32_t vs = vring + (idx % C::NR) * C::SLOT;
                    const uint32_t od = tmem + C::O_COL + (ob * C::KS + c) * C::NP;
#pragma unroll
                    for (int kk = 0; kk < C::BN / 16; ++kk) {
                        // V^T as MN-major A: atoms of 64 dims x 8 keys; LBO steps the
                        // 64-dim sub-chunks, SBO the 8-key groups; 16 keys per step
                        const uint64_t ad = smem_desc_sw128(vs + kk * 16 * 128, C::SUB, 1024);
                        const uint64_t bd =
                            smem_desc_sw128(ps + (kk >> 2) * C::NP * 128 + (kk & 3) * 32, 16, 1024);
                        tc_mma_bf16(od, ad, bd, IDESC_O, (!first || kk > 0) ? 1u : 0u);
                    }
                }
                tc_commit(bar_o_done + 8 * pb);
#pragma unroll
                for (int c = 0; c < C::KS; ++c)
                    tc_commit(bar_v_empty + 8 * ((g_t * C::KS + c) % C::NR));
                if (last) tc_commit(bar_o_full + 8 * ob);
            };
            DtcIter cur = it0;
            int gt = 0, itn = 0;
            bool pv_pending = false, pv_first = false, pv_last = false;
            int pv_ob = 0;
            while (valid(cur)) {
                if (cur.ntiles == 0) {
                    dtc_next(a, cur, cut);
                    continue;
                }
                const int qb = itn & 1;
                const int ob = itn & 1;
                mbar_wait_ool(bar_q_full + 8 * qb, (itn >> 1) & 1, a.err, abort_flag);
                const uint32_t qs = q_smem + qb * C::Q_BUF;
                for (int j = 0; j < cur.ntiles; ++j) {
                    const int sb = gt & 1;
                    if (gt >= 2)
                        mbar_wait_ool(bar_s_free + 8 * sb, ((gt >> 1) - 1) & 1, a.err, abort_flag);
#pragma unroll
                    for (int c = 0; c < C::KS; ++c) {
                        const int idx = gt * C::KS + c;
                        mbar_wait_ool(bar_k_full + 8 * (idx % C::NR), (idx / C::NR) & 1, a.err,
                                  abort_flag);
                    }
                    tc_fence_after();
#pragma unroll
                    for (int c = 0; c < C::KS; ++c) {
                        const uint32_t ks = kring + ((gt * C::KS + c) % C::NR) * C::SLOT;
#pragma unroll
                        for (int kk = 0; kk < 8; ++kk) {
                            const int kg = c * 8 + kk;   // 16-dim step over the head row
                            const uint64_t ad =
                                smem_desc_sw128(ks + (kk >> 2) * C::SUB + (kk & 3) * 32, 16, 1024);
                            const uint64_t bd = smem_desc_sw128(
                                qs + (kg >> 2) * C::NP * 128 + (kg & 3) * 32, 16, 1024);
                            tc_mma_bf16(tmem + C::S_COL + sb * C::NP, ad, bd, IDESC_S,
                                        kg > 0 ? 1u : 0u);
                        }
                    }
                    tc_commit(bar_s_full + 8 * sb);
#pragma unroll
                    for (int c = 0; c < C::KS; ++c)
                        tc_commit(bar_k_empty + 8 * ((gt * C::KS + c) % C::NR));
                    if (j == cur.ntiles - 1) tc_commit(bar_q_empty + 8 * qb);
                    // the PV of the previous tile, which may close the previous item:
                    // S of an item's first tile never waits for the last PV before it
                    if (pv_pending) issue_pv(gt - 1, pv_ob, pv_first, pv_last);
                    pv_pending = true;
                    pv_ob = ob;
                    pv_first = j == 0;
                    pv_last = j == cur.ntiles - 1;
                    ++gt;
                }
                ++itn;
                dtc_next(a, cur, cut);
            }
            if (pv_pending) issue_pv(gt - 1, pv_ob, pv_first, pv_last);
            // every MMA is finished before TMEM is freed (bounded)
            if (gt > 0)
                mbar_drain(bar_o_done + 8 * ((gt - 1) & 1), ((gt - 1) >> 1) & 1,
                           kWaitLimitCycles / 8);
        }
    } else {
        // ============================================================ softmax
        const int t = tid;   // key of the tile = TMEM lane
        const uint32_t t_lane = tmem + ((uint32_t)(warp * 32) << 16);
        const float qsc = a.qscale;
        const int Hq = a.num_q_heads;
        DtcIter cur = it0;
        int gt = 0, itn = 0, ie = 0;
        while (valid(cur)) {
            const int ob = itn & 1;
            float m_run[G], m_ref[G], l[G];
#pragma unroll
            for (int g = 0; g < G; ++g) {
                m_run[g] = -INFINITY;
                m_ref[g] = -INFINITY;
                l[g] = 0.f;
            }
            for (int j = 0; j < cur.ntiles; ++j) {
                const int sb = gt & 1;
                mbar_wait_ool(bar_s_full + 8 * sb, (gt >> 1) & 1, a.err, abort_flag);
                tc_fence_after();
                float sv[8];
                tmem_ld8(t_lane + C::S_COL + sb * C::NP, sv);
                tmem_wait_ld();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar_s_free + 8 * sb);

                const int kt = cur.k0 + j * C::BN;
                const int cnt = min(C::BN, cur.k1 - kt);
                const bool kv = t < cnt;
                float x[G];
#pragma unroll
                for (int g = 0; g < G; ++g) x[g] = kv ? sv[g] * qsc : -INFINITY;
                // tile max of each head across the four warps
                float *rm = red_max + (gt & 1) * 32;
#pragma unroll
                for (int g = 0; g < G; ++g) {
                    const float mx = warp_max(x[g]);
                    if (lane == 0) rm[warp * 8 + g] = mx;
                }
                named_barrier_sync(1, 128);
                float mnew[G];
                bool need[G];
                bool any = false;
#pragma unroll
                for (int g = 0; g < G; ++g) {
                    const float M = fmaxf(fmaxf(rm[g], rm[8 + g]), fmaxf(rm[16 + g], rm[24 + g]));
                    mnew[g] = fmaxf(m_run[g], M);
                    need[g] = (mnew[g] != -INFINITY) &&
                              (m_ref[g] == -INFINITY || mnew[g] > m_ref[g] + 8.f);
                    any = any || need[g];
                }
                if (any) {   // uniform: every thread sees the same maxima
                    float f[8];
#pragma unroll
                    for (int g = 0; g < 8; ++g) f[g] = 1.f;
#pragma unroll
                    for (int g = 0; g < G; ++g)
                        if (need[g]) f[g] = m_ref[g] == -INFINITY ? 0.f : exp2f(m_ref[g] - mnew[g]);
                    if (j >= 1) {   // O^T holds PVs of this item: rescale after the last one
                        mbar_wait_ool(bar_o_done + 8 * ((gt - 1) & 1), ((gt - 1) >> 1) & 1, a.err,
                                  abort_flag);
                        tc_fence_after();
#pragma unroll
                        for (int c = 0; c < C::KS; ++c) {
                            const uint32_t oa = t_lane + C::O_COL + (ob * C::KS + c) * C::NP;
                            float o[8];
                            tmem_ld8(oa, o);
                            tmem_wait_ld();
#pragma unroll
                            for (int e = 0; e < 8; ++e) o[e] *= f[e];
                            tmem_st8(oa, o);
                        }
                        tmem_wait_st();
                    }
#pragma unroll
                    for (int g = 0; g < G; ++g)
                        if (need[g]) {
                            l[g] *= f[g];
                            m_ref[g] = mnew[g];
                        }
                }
#pragma unroll
                for (int g = 0; g < G; ++g) m_run[g] = mnew[g];

                // value rows past the tile's last key may hold anything (pool slots
                // past the sequence, older stages): zero them once they have landed
                if (cnt < C::BN) {
#pragma unroll
                    for (int c = 0; c < C::KS; ++c) {
                        const int idx = gt * C::KS + c;
                        mbar_wait_ool(bar_v_full + 8 * (idx % C::NR), (idx / C::NR) & 1, a.err,
                                  abort_flag);
                        if (!kv) {
                            uint4 *r0 = reinterpret_cast<uint4 *>(
                                smem + C::OFF_V + (idx % C::NR) * C::SLOT + t * 128);
                            uint4 *r1 = reinterpret_cast<uint4 *>(
                                smem + C::OFF_V + (idx % C::NR) * C::SLOT + C::SUB + t * 128);
#pragma unroll
                            for (int e = 0; e < 8; ++e) {
                                r0[e] = make_uint4(0, 0, 0, 0);
                                r1[e] = make_uint4(0, 0, 0, 0);
                            }
                        }
                    }
                }
                // P^T buffer pb was last read by PV(gt - 2)
                const int pb = gt & 1;
                if (gt >= 2)
                    mbar_wait_ool(bar_o_done + 8 * pb, ((gt >> 1) - 1) & 1, a.err, abort_flag);
                uint8_t *prow = smem + C::OFF_P + pb * C::P_BUF + (t >> 6) * (C::NP * 128);
                const int kc = t & 63;
#pragma unroll
                for (int g = 0; g < G; ++g) {
                    const float pg =
                        (kv && m_ref[g] != -INFINITY) ? ex2_approx(x[g] - m_ref[g]) : 0.f;
                    l[g] += pg;
                    *reinterpret_cast<__nv_bfloat16 *>(
                        prow + g * 128 + ((((kc >> 3) ^ g) & 7) << 4) + (kc & 7) * 2) =
                        __float2bfloat16_rn(pg);
                }
                fence_proxy_async_smem();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar_p_full + 8 * pb);
                ++gt;
            }

            // ---- epilogue: exp-sums over the 128 keys, then O^T from TMEM
            float L[G];
            {
                float *rs = red_sum + (ie & 1) * 32;
#pragma unroll
                for (int g = 0; g < G; ++g) {
                    const float sl = warp_sum(l[g]);
                    if (lane == 0) rs[warp * 8 + g] = sl;
                }
                named_barrier_sync(1, 128);
#pragma unroll
                for (int g = 0; g < G; ++g) L[g] = (rs[g] + rs[8 + g]) + (rs[16 + g] + rs[24 + g]);
            }
            float o[C::KS][8];
            if (cur.ntiles > 0) {
                mbar_wait_ool(bar_o_full + 8 * ob, (itn >> 1) & 1, a.err, abort_flag);
                tc_fence_after();
#pragma unroll
                for (int c = 0; c < C::KS; ++c)
                    tmem_ld8(t_lane + C::O_COL + (ob * C::KS + c) * C::NP, o[c]);
                tmem_wait_ld();
                tc_fence_before();
            } else {
#pragma unroll
                for (int c = 0; c < C::KS; ++c)
#pragma unroll
                    for (int e = 0; e < 8; ++e) o[c][e] = 0.f;
            }
            dtc_store_item<D, G>(a, cur, cut, t, o, L, m_ref);
            if (cur.ntiles > 0) ++itn;
            ++ie;
            dtc_next(a, cur, cut);
        }
    }

    // ---------------------------------------------------------------- teardown
    tc_fence_before();
    __syncthreads();
    if (warp == 6) {
        tc_fence_after();
        tmem_dealloc(tmem, C::TMEM_COLS);
    }
}

template <int D, int G>
cudaError_t launch_decode_tc_t(const CUtensorMap &qmap, const CUtensorMap &kmap,
                               const CUtensorMap &vmap, const DecodeTcArgs &a, int grid,
                               cudaStream_t stream) {
    using C = DtcCfg<D>;
    auto kern = paged_decode_tc_kernel<D, G>;
    static bool configured = false;   // benign race: idempotent attribute set
    if (!configured) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             C::SMEM_BYTES);
        if (e != cudaSuccess) return e;
        configured = true;
    }
    return launch_pdl(kern, dim3(grid), dim3(C::THREADS), C::SMEM_BYTES, stream, qmap, kmap, vmap,
                      a);
}

template <int D>
cudaError_t launch_decode_tc_group(int group, const CUtensorMap &qmap, const CUtensorMap &kmap,
                                   const CUtensorMap &vmap, const DecodeTcArgs &a, int grid,
                                   cudaStream_t stream) {
    switch (group) {
        case 1: return launch_decode_tc_t<D, 1>(qmap, kmap, vmap, a, grid, stream);
        case 2: return launch_decode_tc_t<D, 2>(qmap, kmap, vmap, a, grid, stream);
        case 3: return launch_decode_tc_t<D, 3>(qmap, kmap, vmap, a, grid, stream);
        case 4: return launch_decode_tc_t<D, 4>(qmap, kmap, vmap, a, grid, stream);
        case 5: return launch_decode_tc_t<D, 5>(qmap, kmap, vmap, a, grid, stream);
        case 6: return launch_decode_tc_t<D, 6>(qmap, kmap, vmap, a, grid, stream);
        case 7: return launch_decode_tc_t<D, 7>(qmap, kmap, vmap, a, grid, stream);
        case 8: return launch_decode_tc_t<D, 8>(qmap, kmap, vmap, a, grid, stream);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace pa
