// prefill_tc.cuh -- multi-query rows (speculative-verify windows, prefill
// chunks) on the 5th-generation tensor cores, persistent.
//
// What it computes (aisignalhub.me, "packed queries and paged KV"; kwkr.cn,
// "What is Paged Attention" and the kernel table): for the query rows of a
// request with n > 1 rows, softmax(scale * Q K^T) V over the request's paged
// keys, causal rows bottom-right aligned (row i sees keys j <= N - n + i),
// with the sink logit of each head counted once in the denominator.
//
// GB300 design (one CTA per SM, 480 threads, 15 warps):
//  * A work unit is (request, KV head, query block of BQ = 128 / G rows): its
//    MMA rows are the (query row, head) pairs of the G heads that share the
//    KV head, so every K/V page read serves the whole GQA group.  CTAs claim
//    units from a counter, heaviest request first (order written by
//    mq_plan_kernel), so no SM idles while heavy units wait.
//  * The CTA's units form one stream of 128-key tiles t = 0, 1, ...: the
//    tensor cores compute S(t) = Q K(t)^T into one of two TMEM buffers while
//    the softmax of tile t - 1 runs, and O += P(t-1) V(t-1); loads, MMAs and
//    the softmax run across unit boundaries without draining.
//  * Warp 14 (scheduler) claims units, publishes them in a ring of NU
//    entries, and loads each unit's Q (TMA, 3-D box over [total_q, H_q, D])
//    into one of NQB buffers.
//  * Warps 8-9 fill a ring of NKS 16 KB K sub-tiles (one 64-dim chunk of a
//    tile's 128 keys), warps 10-11 a ring of NVS V sub-tiles (128 / (D / 64)
//    keys of every dimension).  A sub-tile's TMA boxes (a page run of box_rows
//    keys x 64 dims, 128-byte swizzled) are issued by one warp of its ring
//    (round robin), one box per lane.  K/V of a request whose rows fit one
//    unit is read once per head and marked evict-first; longer requests' K/V
//    is re-read by their other units and kept (evict-last).
//  * The tensor cores are fed by two issuing threads: tcgen05.mma issue
//    blocks while the MMA queue is full, so a thread waiting on a barrier
//    leaves the tensor pipe idle.  Warp 12 issues S(t) once K(t) has landed
//    and PV(t - NSB) has read P(t - NSB) out of its TMEM buffer; warp 13 issues
//    PV(t) once the softmax has written P(t) and V(t) has landed.  Each ring
//    is freed by its own issuer in the order it is filled, which is what the
//    parity waits on its barriers rely on.  Warp 12 owns the 512 TMEM columns
//    -- S buffers [0, 256), O accumulators from 256.  P is written by the
//    softmax over its own S columns (bf16, two per column) and read by the PV
//    MMA as its A operand from TMEM.
//  * Warps 0-7 (two softmax warpgroups, one thread per TMEM lane = MMA row;
//    warpgroup w takes keys [64 w, 64 w + 64) of every tile): mask, scale into
//    the log2 domain, exchange row maxima through shared memory, rescale O
//    lazily (only when a row's max grows by more than 2^8), write P, and at
//    the end of a unit normalise O into the output.
//  * V rows past a partial tile's last key may hold anything (pool slots
//    past the sequence): the PV MMAs skip the 16-key steps past it, and the
//    softmax zeroes the rows left in the last step (a zero weight times a NaN
//    would still be NaN).
//  * Every mbarrier wait is bounded; the named barriers of the softmax
//    warpgroups are reached the same number of times by all 256 threads (the
//    stop decision at a unit boundary is a barrier reduction).  The waits'
//    retry loop is out of line (mbar_wait_ool): one copy instead of one per
//    wait site keeps the roles' loops in the instruction cache (measured:
//    77 -> 59 KB of code, 151 -> 142 us on the varlen prefill batch).
#pragma once

#include "pa_common.cuh"
#include "pa_internal.h"
#include "tc_common.cuh"

namespace pa {

// A claimed work unit as the scheduler publishes it (r < 0: no more units).
struct MqUnit {
    int r, h, c0, n;           // request, KV head, first packed row, query rows
    int N, i0, rows, kend;     // keys, first row of the block, its rows, keys it reads
    int ntiles, reuse, pad0, pad1;   // key tiles; reuse: other units read the same K/V
};

template <int D, int G>
struct MqCfg {
    static constexpr int BQ = 128 / G;                  // query rows per unit
    static constexpr int M_USED = BQ * G;               // MMA rows in use (<= 128)
    static constexpr int BN = 128;                      // keys per tile
    static constexpr int KCH = D / 64;                  // 128-byte chunks of a head row
    static constexpr int SUB = KCH;                     // K (and V) sub-tiles per tile
    static constexpr int SLOT = BN * 128;               // bytes of a ring slot (16 KB)
    static constexpr int VKEYS = BN / SUB;              // keys of a V sub-tile
    static constexpr int NQB = D >= 256 ? 1 : 2;        // Q buffers
    static constexpr int NSB = D >= 256 ? 2 : 3;        // S/P buffers in TMEM
    static constexpr int NOB = D <= 64 ? 2 : 1;         // O accumulators
    static constexpr int Q_BYTES = KCH * 128 * 128;     // [KCH][128 rows][128 B]
    static constexpr int NKS = D >= 128 ? 5 : 6;         // K ring slots
    static constexpr int NVS = NKS;                      // V ring slots
    static constexpr int NU = 8;                        // unit ring entries
    static constexpr int OFF_SLOT = NQB * Q_BYTES;
    static constexpr int OFF_VSLOT = OFF_SLOT + NKS * SLOT;
    static constexpr int OFF_BAR = OFF_VSLOT + NVS * SLOT;
    static constexpr int NBAR = 2 * NQB + 2 * NKS + 2 * NVS + 3 * NSB + NOB + 2 * NU;
    static constexpr int OFF_RED = OFF_BAR + ((NBAR * 8 + 15) & ~15);   // float [2][128]
    static constexpr int OFF_UNIT = OFF_RED + 2 * 128 * 4;              // MqUnit [NU]
    static constexpr int OFF_MISC = OFF_UNIT + NU * (int)sizeof(MqUnit);   // TMEM base, abort
    static constexpr int SMEM_BYTES = OFF_MISC + 16 + 1024;             // + alignment slack
    static constexpr int NPK = 2, NPV = 2;               // K and V producer warps
    static constexpr int W_MMA_S = 8 + NPK + NPV;       // S-issuing warp (TMEM owner)
    static constexpr int W_MMA_PV = W_MMA_S + 1;        // PV-issuing warp
    static constexpr int W_SCHED = W_MMA_S + 2;         // scheduler warp
    static constexpr int THREADS = 32 * (W_SCHED + 1);
    static_assert(THREADS == 480, "launch bounds below");
    static constexpr int TMEM_COLS = 512;
    static constexpr int O_COL = NSB * BN;              // after the S buffers
    static_assert(VKEYS * 128 * KCH == SLOT, "a V sub-tile fills a slot");
    static_assert(O_COL + NOB * D <= TMEM_COLS, "TMEM columns");
    static_assert(SMEM_BYTES <= 227 * 1024, "shared memory");
    static_assert(Q_BYTES % 1024 == 0 && SLOT % 1024 == 0, "swizzle atoms");
};

// Or over `nthreads` threads of named barrier `id` (all of them get the result).
__device__ __forceinline__ bool barrier_or(int id, int nthreads, bool v) {
    uint32_t out;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 q, %1, 0;\n\t"
        "bar.red.or.pred p, %2, %3, q;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(out)
        : "r"((uint32_t)v), "r"(id), "r"(nthreads)
        : "memory");
    return out != 0;
}

template <int D, int G>
__global__ void __launch_bounds__(480, 1)
    paged_prefill_tc_kernel(const __grid_constant__ CUtensorMap qmap,
                            const __grid_constant__ CUtensorMap kmap,
                            const __grid_constant__ CUtensorMap vmap, const TcArgs a) {
    using C = MqCfg<D, G>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = smem_u32(smem);
    const uint32_t q_smem = sbase;
    const uint32_t kring0 = sbase + C::OFF_SLOT;                      // K ring [NKS][16 KB]
    const uint32_t vring0 = sbase + C::OFF_VSLOT;                     // V ring [NVS][16 KB]
    // barriers (each waited by its parties in order, never two phases behind)
    const uint32_t bar_q_full = sbase + C::OFF_BAR;                   // [NQB]
    const uint32_t bar_q_empty = bar_q_full + 8 * C::NQB;             // [NQB] last S of the unit done
    const uint32_t bar_kfull = bar_q_empty + 8 * C::NQB;              // [NKS] owner's arrival + bytes
    const uint32_t bar_kempty = bar_kfull + 8 * C::NKS;               // [NKS] its S MMAs done
    const uint32_t bar_vfull = bar_kempty + 8 * C::NKS;               // [NVS] owner's arrival + bytes
    const uint32_t bar_vempty = bar_vfull + 8 * C::NVS;               // [NVS] its PV MMAs done
    const uint32_t bar_s_full = bar_vempty + 8 * C::NVS;              // [NSB] S(t) in TMEM
    const uint32_t bar_p_full = bar_s_full + 8 * C::NSB;              // [NSB] P(t) in TMEM (8 warps)
    const uint32_t bar_o_done = bar_p_full + 8 * C::NSB;              // [NSB] PV(t) done
    const uint32_t bar_o_free = bar_o_done + 8 * C::NSB;              // [NOB] O read out (8 warps)
    const uint32_t bar_u_full = bar_o_free + 8 * C::NOB;              // [NU] unit published
    const uint32_t bar_u_empty = bar_u_full + 8 * C::NU;              // [NU] unit read (13 warps)
    float *xr = reinterpret_cast<float *>(smem + C::OFF_RED);         // [2][128]
    MqUnit *units = reinterpret_cast<MqUnit *>(smem + C::OFF_UNIT);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + C::OFF_MISC);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + C::OFF_MISC + 8);

    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;
    const int bs = a.block_size;

    // ---------------------------------------------------------------- setup
    if (tid == 0) {
        for (int b = 0; b < C::NQB; ++b) {
            mbar_init(bar_q_full + 8 * b, 1);
            mbar_init(bar_q_empty + 8 * b, 1);
        }
        for (int s = 0; s < C::NKS; ++s) {
            mbar_init(bar_kfull + 8 * s, 1);   // the owning producer warp's arrival
            mbar_init(bar_kempty + 8 * s, 1);
        }
        for (int s = 0; s < C::NVS; ++s) {
            mbar_init(bar_vfull + 8 * s, 1);
            mbar_init(bar_vempty + 8 * s, 1);
        }
        for (int b = 0; b < C::NSB; ++b) {
            mbar_init(bar_s_full + 8 * b, 1);
            mbar_init(bar_p_full + 8 * b, 8);
            mbar_init(bar_o_done + 8 * b, 1);
        }
        for (int b = 0; b < C::NOB; ++b) mbar_init(bar_o_free + 8 * b, 8);
        for (int u = 0; u < C::NU; ++u) {
            mbar_init(bar_u_full + 8 * u, 1);
            mbar_init(bar_u_empty + 8 * u, 10 + C::NPK + C::NPV);   // every role but the scheduler
        }
        fence_barrier_init();
        *abort_flag = 0;
    }
    if (warp == C::W_MMA_S) {
        tmem_alloc(smem_u32(tmem_slot), C::TMEM_COLS);
        tmem_relinquish();
    }
    if (C::M_USED < 128) {
        // Q rows past the (query row, head) pairs are never loaded: zero them
        // once so their score rows stay finite
        constexpr int PAD = (128 - C::M_USED) * 8;   // 16-byte pieces per chunk
        for (int b = 0; b < C::NQB; ++b)
            for (int c = 0; c < C::KCH; ++c)
                for (int q = tid; q < PAD; q += C::THREADS)
                    *reinterpret_cast<uint4 *>(smem + b * C::Q_BYTES + c * 128 * 128 +
                                               C::M_USED * 128 + q * 16) = make_uint4(0, 0, 0, 0);
        fence_proxy_async_smem();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    // the unit of sequence number k (waits for it to be published); false
    // when the wait gave up
    auto take_unit = [&](int k, MqUnit &u) -> bool {
        const bool ok = mbar_wait_ool(bar_u_full + 8 * (k % C::NU), (k / C::NU) & 1, a.err, abort_flag);
        if (ok) u = units[k % C::NU];
        return ok;
    };
    auto tile_of = [](const MqUnit &, int j) { return j; };

    if (warp == C::W_SCHED) {
        // ============================================================ scheduler
        if (lane == 0) {
            prefetch_tensormap(&qmap);
            pdl_wait();   // the plan (and this step's inputs) are written
            int *hdr = a.plan;
            const int *order = hdr + kPlanHeader;
            const int *P = order + a.num_seqs;
            const int count = hdr[1];
            const int total = hdr[2];
            const int max_keys = a.max_blocks_per_seq * bs;
            const uint64_t pol_q = policy_evict_first();
            int itn = 0;   // units with tiles so far (Q buffers)
            int q_last[2] = {-1, -1};
            for (int k = 0;; ++k) {
                const int us = k % C::NU;
                if (k >= C::NU &&
                    !mbar_wait_ool(bar_u_empty + 8 * us, ((k / C::NU) - 1) & 1, a.err, abort_flag))
                    break;   // (aborted: publish nothing more; waiters give up too)
                const int c = atomicAdd(hdr, 1);
                MqUnit u;
                u.r = -1;
                if (c < total) {
                    int lo = 0, hi = count - 1;   // last k' with P[k'] <= c
                    while (lo < hi) {
                        const int mid = (lo + hi + 1) >> 1;
                        if (__ldg(P + mid) <= c) lo = mid;
                        else hi = mid - 1;
                    }
                    const int r = __ldg(order + lo);
                    const int local = c - __ldg(P + lo);
                    const int c0 = __ldg(a.cu_seqlens_q + r);
                    const int n = __ldg(a.cu_seqlens_q + r + 1) - c0;
                    const int nblk = (n + C::BQ - 1) / C::BQ;
                    const int lp = local / a.num_kv_heads;
                    u.r = r;
                    u.h = local - lp * a.num_kv_heads;
                    u.c0 = c0;
                    u.n = n;
                    u.N = max(0, min(__ldg(a.seq_lens_k + r), max_keys));
                    u.i0 = (nblk - 1 - lp) * C::BQ;   // heaviest (last) block first
                    u.rows = min(C::BQ, n - u.i0);
                    u.kend = max(0, a.causal ? min(u.N, u.N - n + u.i0 + u.rows) : u.N);
                    u.ntiles = (u.kend + C::BN - 1) / C::BN;
                    u.reuse = nblk > 1;
                    // a unit outside the batch (an inconsistent plan) is never
                    // published: report it and stop claiming
                    if (r < 0 || r >= a.num_seqs || c0 < 0 || n < 2 || c0 + n > a.total_q ||
                        u.i0 < 0 || u.rows < 1) {
                        report_error(a.err, 3);
                        u.r = -1;
                    }
                }
                units[us] = u;
                mbar_arrive(bar_u_full + 8 * us);   // (release: the unit is visible)
                if (u.r < 0) break;
                if (u.ntiles > 0) {
                    const int qb = itn % C::NQB;
                    if (itn >= C::NQB &&
                        !mbar_wait_ool(bar_q_empty + 8 * qb, ((itn / C::NQB) - 1) & 1, a.err,
                                   abort_flag))
                        break;
                    mbar_arrive_expect_tx(bar_q_full + 8 * qb, C::KCH * C::M_USED * 128);
#pragma unroll
                    for (int ch = 0; ch < C::KCH; ++ch)
                        tma_load_3d(q_smem + qb * C::Q_BYTES + ch * 128 * 128, &qmap, ch * 64,
                                    u.h * G, u.c0 + u.i0, bar_q_full + 8 * qb, pol_q);
                    q_last[qb] = itn;
                    ++itn;
                }
            }
            // Q loads in flight land before the CTA can exit (bounded)
            for (int b = 0; b < C::NQB; ++b)
                if (q_last[b] >= 0)
                    mbar_drain(bar_q_full + 8 * b, (q_last[b] / C::NQB) & 1, kWaitLimitCycles / 8);
        }
    } else if (warp >= 8 && warp < 8 + C::NPK + C::NPV) {
        // ============================================================ producers
        // K warps fill the K ring, V warps the V ring.  Sub-tile sequence
        // number seq of a ring belongs to warp seq % (warps of that ring):
        // that warp alone waits for the slot, arms it with the sub-tile's
        // bytes and issues its boxes (at most 16), one per lane.
        const bool is_k = warp < 8 + C::NPK;
        const int pw = is_k ? warp - 8 : warp - 8 - C::NPK;
        const int nw = is_k ? C::NPK : C::NPV;
        const int NS = is_k ? C::NKS : C::NVS;
        const uint32_t full0 = is_k ? bar_kfull : bar_vfull;
        const uint32_t empty0 = is_k ? bar_kempty : bar_vempty;
        const uint32_t ring0 = is_k ? kring0 : vring0;
        const CUtensorMap *map = is_k ? &kmap : &vmap;
        if (lane == 0 && pw == 0) prefetch_tensormap(map);
        pdl_wait();   // block tables and this step's K/V rows are written
        const int BR = a.box_rows;
        const uint64_t pol_keep = policy_evict_last();    // re-read by the request's other units
        const uint64_t pol_once = policy_evict_first();   // read by this unit alone
        uint64_t pol = pol_keep;
        int seq = 0;        // sequence number of the ring's next sub-tile
        bool bad = false;
        // waits for the slot of `seq` to be free and arms it with the sub-tile's
        // bytes (arm = false only in the failure-path test); `bad` when the wait
        // gave up
        auto acquire = [&](int bytes, bool arm) -> uint32_t {
            const int slot = seq % NS;
            if (lane == 0) {
                if (seq >= NS)
                    bad = !mbar_wait_ool(empty0 + 8 * slot, ((seq / NS) - 1) & 1, a.err, abort_flag);
                if (!bad && arm) mbar_arrive_expect_tx(full0 + 8 * slot, bytes);
            }
            bad = __shfl_sync(0xffffffffu, (int)bad, 0);
            return (uint32_t)slot;
        };
        // page id of page run `lane` of tile j of unit u (0 past the tile)
        auto load_pg = [&](const MqUnit &u, int j) -> int {
            const int kt = j * C::BN;
            const int runs = (min(C::BN, u.kend - kt) + BR - 1) / BR;
            return lane < runs ? __ldg(a.block_tables + (int64_t)u.r * a.max_blocks_per_seq +
                                       (kt + lane * BR) / bs)
                               : 0;
        };
        int t = 0;
        for (int k = 0; !bad; ++k) {
            MqUnit u;
            const int ok = __all_sync(0xffffffffu, take_unit(k, u));   // (every lane acquires)
            __syncwarp();
            if (lane == 0) mbar_arrive(bar_u_empty + 8 * (k % C::NU));
            if (!ok || u.r < 0) break;
            if (u.ntiles == 0) continue;
            pol = u.reuse ? pol_keep : pol_once;
            int pg_cur = load_pg(u, 0);
            int pg_nxt = u.ntiles > 1 ? load_pg(u, 1) : 0;
            for (int j = 0; j < u.ntiles && !bad; ++j) {
                const int kt = j * C::BN;
                const int cnt = min(C::BN, u.kend - kt);
                const int runs = (cnt + BR - 1) / BR;   // <= 16 page runs
                // (failure-path test: the CTA's first K tile is neither armed
                // nor loaded, so the S issuer's bounded wait for it runs out)
                const bool skip = is_k && t == 0 && a.test_skip_first_k;
#pragma unroll 1
                for (int s = 0; s < C::SUB && !bad; ++s, ++seq) {
                    if (is_k) {
                        // K sub-tile s: 64-dim chunk s of the tile's keys, one box
                        // per page run, lane u loads run u
                        if (seq % nw == pw) {
                            const uint32_t slot = acquire(runs * BR * 128, !skip);
                            if (!bad && !skip && lane < runs)
                                tma_load_3d(ring0 + slot * C::SLOT + lane * BR * 128, map, s * 64,
                                            u.h, pg_cur * bs + (kt + lane * BR) % bs,
                                            full0 + 8 * slot, pol);
                        }
                    } else {
                        // V sub-tile s: keys [s VKEYS, (s + 1) VKEYS) of every 64-dim
                        // chunk; lane b loads run u_lo + b / KCH, chunk b % KCH
                        const int u_lo = s * (C::VKEYS / BR);
                        const int u_hi = min(runs, (s + 1) * (C::VKEYS / BR));
                        const int nbox = max(0, u_hi - u_lo) * C::KCH;
                        const int ul = lane / C::KCH, ch = lane % C::KCH;
                        const int ru = u_lo + ul;
                        const int pgu = __shfl_sync(0xffffffffu, pg_cur, ru & 31);
                        if (seq % nw == pw) {
                            const uint32_t slot = acquire(nbox * BR * 128, true);
                            if (!bad && lane < nbox)
                                tma_load_3d(ring0 + slot * C::SLOT + ch * (C::VKEYS * 128) +
                                                ul * BR * 128,
                                            map, ch * 64, u.h, pgu * bs + (kt + ru * BR) % bs,
                                            full0 + 8 * slot, pol);
                        }
                    }
                }
                pg_cur = pg_nxt;
                if (j + 2 < u.ntiles) pg_nxt = load_pg(u, j + 2);
                ++t;
            }
        }
        // copies in flight land before the CTA can exit (bounded)
        if (lane == 0)
            for (int i = max(0, seq - NS); i < seq; ++i)
                mbar_drain(full0 + 8 * (i % NS), (i / NS) & 1, kWaitLimitCycles / 8);
    } else if (warp == C::W_MMA_S) {
        // ============================================================ S issuer
        // S(t) = Q K(t)^T into TMEM buffer t % NSB, once PV(t - NSB) has read P(t - NSB)
        // out of it; K sub-tiles are freed in the order they were filled.
        if (lane == 0) {
            constexpr uint32_t IDESC_S = idesc_bf16_f32(128, C::BN, 0, 0);
            int t = 0, itn = 0;
            uint32_t last_commit = 0, last_parity = 0;   // drained before TMEM is freed
            bool any = false;
            for (int k = 0;; ++k) {
                MqUnit u;
                const bool ok = take_unit(k, u);
                mbar_arrive(bar_u_empty + 8 * (k % C::NU));
                if (!ok || u.r < 0 || *abort_flag) break;
                if (u.ntiles == 0) continue;
                const int qb = itn % C::NQB;
                mbar_wait_ool(bar_q_full + 8 * qb, (itn / C::NQB) & 1, a.err, abort_flag);
                const uint32_t qs = q_smem + qb * C::Q_BYTES;
                for (int j = 0; j < u.ntiles; ++j) {
                    const int sb = t % C::NSB;
                    if (t >= C::NSB)   // PV(t - NSB) has read P(t - NSB) out of buffer sb
                        mbar_wait_ool(bar_o_done + 8 * sb, ((t - C::NSB) / C::NSB) & 1, a.err,
                                  abort_flag);
                    const int p0 = t * C::SUB;
#pragma unroll
                    for (int s = 0; s < C::SUB; ++s)
                        mbar_wait_ool(bar_kfull + 8 * ((p0 + s) % C::NKS), ((p0 + s) / C::NKS) & 1,
                                  a.err, abort_flag);
                    tc_fence_after();
#pragma unroll
                    for (int s = 0; s < C::SUB; ++s) {   // 64-dim chunk s of K and Q
                        const uint32_t ks = kring0 + ((p0 + s) % C::NKS) * C::SLOT;
#pragma unroll
                        for (int kl = 0; kl < 4; ++kl) {
                            const uint32_t off = kl * 32;   // 16 bf16 within the 128-B row
                            const uint64_t ad =
                                smem_desc_sw128(qs + s * 128 * 128 + off, 16, 1024);
                            const uint64_t bd = smem_desc_sw128(ks + off, 16, 1024);
                            tc_mma_bf16(tmem + sb * C::BN, ad, bd, IDESC_S,
                                        (s > 0 || kl > 0) ? 1u : 0u);
                        }
                    }
#pragma unroll
                    for (int s = 0; s < C::SUB; ++s)
                        tc_commit(bar_kempty + 8 * ((p0 + s) % C::NKS));
                    tc_commit(bar_s_full + 8 * sb);
                    last_commit = bar_s_full + 8 * sb;
                    last_parity = (t / C::NSB) & 1;
                    any = true;
                    if (j == u.ntiles - 1) tc_commit(bar_q_empty + 8 * qb);
                    ++t;
                }
                ++itn;
            }
            // every MMA is finished before TMEM is freed (bounded, also when
            // the pipeline was aborted)
            if (any) mbar_drain(last_commit, last_parity, kWaitLimitCycles / 8);
        }
    } else if (warp == C::W_MMA_PV) {
        // ============================================================ PV issuer
        // O += P(t) V(t) once the softmax has written P(t); V sub-tiles are
        // freed in the order they were filled.
        if (lane == 0) {
            constexpr uint32_t IDESC_O = idesc_bf16_f32(128, D, 0, 1);
            constexpr int KPS = C::VKEYS / 16;   // 16-key steps per V sub-tile
            int t = 0, itn = 0;
            uint32_t last_commit = 0, last_parity = 0;
            bool any = false;
            for (int k = 0;; ++k) {
                MqUnit u;
                const bool ok = take_unit(k, u);
                mbar_arrive(bar_u_empty + 8 * (k % C::NU));
                if (!ok || u.r < 0 || *abort_flag) break;
                if (u.ntiles == 0) continue;
                const int ob = itn % C::NOB;
                const uint32_t od = tmem + C::O_COL + ob * D;
                for (int j = 0; j < u.ntiles; ++j) {
                    if (j == 0 && itn >= C::NOB)   // the unit NOB back has read its O out
                        mbar_wait_ool(bar_o_free + 8 * ob, ((itn / C::NOB) - 1) & 1, a.err,
                                  abort_flag);
                    mbar_wait_ool(bar_p_full + 8 * (t % C::NSB), (t / C::NSB) & 1, a.err, abort_flag);
                    const int cnt = min(C::BN, u.kend - j * C::BN);
                    const int nk = (cnt + 15) / 16;   // 16-key steps holding keys
                    const int p0 = t * C::SUB;
#pragma unroll
                    for (int s = 0; s < C::SUB; ++s)
                        mbar_wait_ool(bar_vfull + 8 * ((p0 + s) % C::NVS), ((p0 + s) / C::NVS) & 1,
                                  a.err, abort_flag);
                    tc_fence_after();
                    const uint32_t pt = tmem + (t % C::NSB) * C::BN;
#pragma unroll
                    for (int s = 0; s < C::SUB; ++s) {
                        const uint32_t vs = vring0 + ((p0 + s) % C::NVS) * C::SLOT;
#pragma unroll
                        for (int kl = 0; kl < KPS; ++kl) {
                            const int kk = s * KPS + kl;
                            if (kk >= nk) break;
                            // V as MN-major B: atoms of 64 dims x 8 keys; LBO steps
                            // the 64-dim chunks, SBO the 8-key groups
                            const uint64_t bd =
                                smem_desc_sw128(vs + kl * 16 * 128, C::VKEYS * 128, 1024);
                            // P of keys [16 kk, 16 kk + 16): warpgroup kk / 4's columns
                            const uint32_t pa = pt + 64 * (kk >> 2) + (kk & 3) * 8;
                            tc_mma_bf16_ts(od, pa, bd, IDESC_O, (j == 0 && kk == 0) ? 0u : 1u);
                        }
                    }
#pragma unroll
                    for (int s = 0; s < C::SUB; ++s)
                        tc_commit(bar_vempty + 8 * ((p0 + s) % C::NVS));
                    tc_commit(bar_o_done + 8 * (t % C::NSB));
                    last_commit = bar_o_done + 8 * (t % C::NSB);
                    last_parity = (t / C::NSB) & 1;
                    any = true;
                    ++t;
                }
                ++itn;
            }
            if (any) mbar_drain(last_commit, last_parity, kWaitLimitCycles / 8);
        }
    } else {
        // ============================================================ softmax
        // Warpgroup wg takes keys [64 wg, 64 wg + 64) of every tile, and half
        // of O's columns when O is rescaled or written out.  Row maxima and
        // sums of the two halves meet in shared memory.
        constexpr int HB = 64;
        const int wg = warp >> 2;
        const int m = ((warp & 3) << 5) | lane;           // MMA row = TMEM lane
        const int kb = wg * HB;
        const int i = m / G, g = m % G;
        const uint32_t t_lane = tmem + ((uint32_t)((warp & 3) * 32) << 16);
        auto exchange = [&](float v) -> float {
            xr[wg * 128 + m] = v;
            named_barrier_sync(1, 256);
            const float o = xr[(1 - wg) * 128 + m];
            named_barrier_sync(1, 256);
            return o;
        };
        const float qs = a.qscale;
        const int Hq = a.num_q_heads;
        int t = 0, itn = 0;
        for (int k = 0;; ++k) {
            MqUnit u;
            const bool ok = take_unit(k, u);
            __syncwarp();
            if (lane == 0) mbar_arrive(bar_u_empty + 8 * (k % C::NU));
            // one decision for all 256 threads: the named barriers below stay matched
            if (barrier_or(2, 256, !ok || u.r < 0)) break;
            const bool row_ok = (m < C::M_USED) && (i < u.rows) && u.c0 + u.i0 + i < a.total_q;
            const int qi = u.i0 + i;
            const int N = u.N, n = u.n;
            const int lim = min(N - 1, a.causal ? N - n + qi : N - 1);   // last visible key
            const int lim_all = min(N - 1, a.causal ? N - n + u.i0 : N - 1);   // of every row
            const int ob = itn % C::NOB;
            const uint32_t o_lane = t_lane + C::O_COL + ob * D + wg * (D / 2);
            float m_run = -INFINITY, m_ref = -INFINITY, l = 0.f;   // l: this half's sum
            for (int j = 0; j < u.ntiles; ++j) {
                const int sb = t % C::NSB;
                mbar_wait_ool(bar_s_full + 8 * sb, (t / C::NSB) & 1, a.err, abort_flag);
                tc_fence_after();
                float s[HB];
                tmem_ld32(t_lane + sb * C::BN + kb, s);
                tmem_ld32(t_lane + sb * C::BN + kb + 32, s + 32);
                tmem_wait_ld();

                // Tiles that reach past a row's last visible key are masked and
                // scaled here (masked keys become -inf); fully visible tiles keep
                // raw scores and are scaled inside the exponent.
                const int kt0 = tile_of(u, j) * C::BN;
                const bool tmask = kt0 + C::BN - 1 > lim_all;
                if (tmask) {
#pragma unroll
                    for (int c = 0; c < HB; ++c)
                        s[c] = (row_ok && kt0 + kb + c <= lim) ? s[c] * qs : -INFINITY;
                }
                const float sc = tmask ? 1.f : qs;
                // max of sc * s over this half (8 independent chains)
                const bool neg = sc < 0.f;
                float mx[8];
#pragma unroll
                for (int q = 0; q < 8; ++q) mx[q] = neg ? -s[q] : s[q];
#pragma unroll
                for (int c = 8; c < HB; c += 8)
#pragma unroll
                    for (int q = 0; q < 8; ++q) mx[q] = fmaxf(mx[q], neg ? -s[c + q] : s[c + q]);
#pragma unroll
                for (int q = 4; q > 0; q >>= 1)
#pragma unroll
                    for (int e = 0; e < q; ++e) mx[e] = fmaxf(mx[e], mx[e + q]);
                const float hmax = mx[0] == -INFINITY ? -INFINITY : mx[0] * fabsf(sc);
                const float tmax = fmaxf(hmax, exchange(hmax));   // the whole row's tile max
                const float m_new = fmaxf(m_run, tmax);
                m_run = m_new;
                const bool need =
                    (m_new != -INFINITY) && (m_ref == -INFINITY || m_new > m_ref + 8.f);

                // value rows of the last 16-key step past the tile's last key
                // may hold anything: zero them before the PV MMA reads them
                const int cnt = min(C::BN, u.kend - kt0);
                if (cnt & 15) {
                    const int s_v = cnt / C::VKEYS;                  // V sub-tile holding them
                    const int pos = t * C::SUB + s_v;                // its V ring sequence number
                    // A parity wait tells the phase of `pos` from that of pos - NVS
                    // only once the latter has completed.  If pos - NVS belongs to a
                    // tile tp > t - NSB, PV(tp) may not even have started: wait for
                    // it.  Older sub-tiles were read by PV(t - NSB) or earlier, which
                    // finished before S(t) was issued.
                    const int tp = pos >= C::NVS ? (pos - C::NVS) / C::SUB : -1;
                    if (tp >= 0 && tp > t - C::NSB)
                        mbar_wait_ool(bar_o_done + 8 * (tp % C::NSB), (tp / C::NSB) & 1, a.err,
                                  abort_flag);
                    mbar_wait_ool(bar_vfull + 8 * (pos % C::NVS), (pos / C::NVS) & 1, a.err,
                              abort_flag);
                    uint8_t *vsp = smem + C::OFF_VSLOT + (pos % C::NVS) * C::SLOT;
                    const int k0 = cnt - s_v * C::VKEYS;             // first row to clear
                    const int nclr = 16 - (cnt & 15);
                    for (int q = wg * 128 + m; q < nclr * C::KCH * 8; q += 256) {
                        const int row = k0 + q / (C::KCH * 8);
                        const int ch = (q >> 3) % C::KCH;
                        *reinterpret_cast<uint4 *>(vsp + ch * C::VKEYS * 128 + row * 128 +
                                                   (q & 7) * 16) = make_uint4(0, 0, 0, 0);
                    }
                }
                // O changes only when a row's reference max moves: then PV(t - 1)
                // of this unit must be done.  Each warpgroup rescales its half.
                if (j >= 1 && __any_sync(0xffffffffu, need)) {
                    mbar_wait_ool(bar_o_done + 8 * ((t - 1) % C::NSB), ((t - 1) / C::NSB) & 1, a.err,
                              abort_flag);
                    tc_fence_after();
                    const float f = need ? (m_ref == -INFINITY ? 0.f : exp2f(m_ref - m_new)) : 1.f;
#pragma unroll 1
                    for (int c = 0; c < D / 64; ++c) {
                        float o[32];
                        tmem_ld32(o_lane + 32 * c, o);
                        tmem_wait_ld();
#pragma unroll
                        for (int e = 0; e < 32; ++e) o[e] *= f;
                        tmem_st32(o_lane + 32 * c, o);
                    }
                    tmem_wait_st();
                }
                if (need) {
                    l *= (m_ref == -INFINITY) ? 0.f : exp2f(m_ref - m_new);
                    m_ref = m_new;
                }
                // P = 2^(sc * s - m_ref) as bf16 (masked keys: 2^-inf = 0) over this
                // half's own S columns, two keys per 32-bit column
                const float2 qs2 = make_float2(sc, sc);
                const float mu = (m_ref == -INFINITY) ? 0.f : -m_ref;
                const float2 mu2 = make_float2(mu, mu);
                float2 sum2[4];
#pragma unroll
                for (int q = 0; q < 4; ++q) sum2[q] = make_float2(0.f, 0.f);
                const uint32_t pt = t_lane + sb * C::BN + kb;
#pragma unroll
                for (int k16 = 0; k16 < HB / 16; ++k16) {
                    uint32_t w8[8];
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        float2 x = __ffma2_rn(
                            make_float2(s[k16 * 16 + 2 * e], s[k16 * 16 + 2 * e + 1]), qs2, mu2);
                        x.x = ex2_approx(x.x);
                        x.y = ex2_approx(x.y);
                        sum2[e & 3] = __fadd2_rn(sum2[e & 3], x);
                        w8[e] = pack_bf16x2(x.x, x.y);
                    }
                    tmem_st8u(pt + k16 * 8, w8);
                }
                const float2 sa = __fadd2_rn(sum2[0], sum2[1]);
                const float2 sbb = __fadd2_rn(sum2[2], sum2[3]);
                l += (sa.x + sa.y) + (sbb.x + sbb.y);
                tmem_wait_st();
                fence_proxy_async_smem();   // zeroed V rows (generic writes) reach the tensor core
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar_p_full + 8 * sb);
                ++t;
            }
            // ---- epilogue: out = O / (l + sink term); each warpgroup writes half of D
            if (u.ntiles > 0) {
                mbar_wait_ool(bar_o_done + 8 * ((t - 1) % C::NSB), ((t - 1) / C::NSB) & 1, a.err,
                          abort_flag);
                tc_fence_after();
            }
            const float l_row = l + exchange(l);
            float scale_out = 0.f;
            if (l_row > 0.f) {
                if (a.sinks) {
                    const float sk2 = a.sinks[u.h * G + g] * kLog2e;
                    const float M2 = fmaxf(m_ref, sk2);
                    const float f = exp2f(m_ref - M2);
                    scale_out = f / (l_row * f + exp2f(sk2 - M2));
                } else {
                    scale_out = 1.f / l_row;
                }
            }
            __nv_bfloat16 *orow = reinterpret_cast<__nv_bfloat16 *>(a.out) +
                                  (((int64_t)u.c0 + qi) * Hq + (int64_t)u.h * G + g) * D +
                                  wg * (D / 2);
            // O is read out of TMEM into packed bf16 registers first, two 32-column
            // loads in flight, and handed back to the PV issuer before the stores
            uint32_t pk[D / 4];   // this thread's D / 2 outputs, two per register
            if (u.ntiles > 0) {
#pragma unroll
                for (int c = 0; c < D / 64; c += 2) {
                    float o[64];
                    tmem_ld32(o_lane + 32 * c, o);
                    if (c + 1 < D / 64) tmem_ld32(o_lane + 32 * (c + 1), o + 32);
                    tmem_wait_ld();
#pragma unroll
                    for (int e = 0; e < 32 * min(2, D / 64 - c); e += 2)
                        pk[16 * c + e / 2] = pack_bf16x2(o[e] * scale_out, o[e + 1] * scale_out);
                }
                // O may now be overwritten by the unit NOB ahead
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar_o_free + 8 * ob);
                ++itn;
            } else {
#pragma unroll
                for (int e = 0; e < D / 4; ++e) pk[e] = 0u;   // no key visible: zeros
            }
            if (row_ok) {
                uint4 *dst = reinterpret_cast<uint4 *>(orow);
#pragma unroll
                for (int q = 0; q < D / 16; ++q)
                    dst[q] = make_uint4(pk[4 * q], pk[4 * q + 1], pk[4 * q + 2], pk[4 * q + 3]);
            }
        }
    }

    // ---------------------------------------------------------------- teardown
    tc_fence_before();
    __syncthreads();
    if (warp == C::W_MMA_S) {
        tc_fence_after();
        tmem_dealloc(tmem, C::TMEM_COLS);
    }
}

template <int D, int G>
cudaError_t launch_prefill_tc_t(const CUtensorMap &qmap, const CUtensorMap &kmap,
                                const CUtensorMap &vmap, const TcArgs &a, int grid,
                                cudaStream_t stream) {
    using C = MqCfg<D, G>;
    auto kern = paged_prefill_tc_kernel<D, G>;
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
cudaError_t launch_prefill_tc_group(int group, const CUtensorMap &qmap, const CUtensorMap &kmap,
                                    const CUtensorMap &vmap, const TcArgs &a, int grid,
                                    cudaStream_t stream) {
    switch (group) {
        case 1: return launch_prefill_tc_t<D, 1>(qmap, kmap, vmap, a, grid, stream);
        case 2: return launch_prefill_tc_t<D, 2>(qmap, kmap, vmap, a, grid, stream);
        case 3: return launch_prefill_tc_t<D, 3>(qmap, kmap, vmap, a, grid, stream);
        case 4: return launch_prefill_tc_t<D, 4>(qmap, kmap, vmap, a, grid, stream);
        case 5: return launch_prefill_tc_t<D, 5>(qmap, kmap, vmap, a, grid, stream);
        case 6: return launch_prefill_tc_t<D, 6>(qmap, kmap, vmap, a, grid, stream);
        case 7: return launch_prefill_tc_t<D, 7>(qmap, kmap, vmap, a, grid, stream);
        case 8: return launch_prefill_tc_t<D, 8>(qmap, kmap, vmap, a, grid, stream);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace pa
