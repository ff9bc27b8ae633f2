// prefill_tc.cuh -- multi-query rows (speculative-verify windows, prefill
// chunks) on the 5th-generation tensor cores.
//
// What it computes (aisignalhub.me, "packed queries and paged KV"; kwkr.cn,
// "What is Paged Attention" and the kernel table): for the query rows of a
// request with n > 1 rows, softmax(scale * Q K^T) V over the request's paged
// keys, causal rows bottom-right aligned (row i sees keys j <= N - n + i),
// with the sink logit of each head counted once in the denominator.
//
// GB300 design (one CTA per (request, KV head, query block), 352 threads):
//  * An MMA row is a (query row, head) pair: BQ = 128 / G query rows times the
//    G heads of one KV head fill M = 128, so every K/V page read serves the
//    whole GQA group.  The grid walks virtual query blocks: request r owns
//    blocks cu_seqlens_q[r] / BQ + r onward, found by a binary search over
//    cu_seqlens_q; blocks are visited heaviest (last, causally) first.
//  * Warps 4 and 6 (producers): TMA loads Q once (3-D box over [total_q, H_q,
//    D]) and streams the K and the V tiles of BN keys page by page through
//    separate stage rings, 128-byte-swizzled (the tensor cores' canonical
//    layout); a K stage is released as soon as its QK^T is done, so the next
//    K tiles load while the softmax and PV of earlier tiles run.
//  * Warp 5 (MMA): allocates 512 TMEM columns, issues S = Q K^T into one of
//    two TMEM buffers (so QK of tile j+1 overlaps the softmax of tile j) and
//    O += P V with V read MN-major; commits signal mbarriers.
//  * Warps 0-3 and 7-10 (two softmax warpgroups, one thread per TMEM lane = MMA
//    row in each, each taking half of every tile's keys): load S, mask and
//    scale into the log2 domain, keep a running max with lazy rescaling of O
//    (only when the max grows by more than 2^8), write P as bf16 into one of
//    two TMEM buffers (the PV MMA reads its A operand from TMEM, which leaves
//    shared memory for a third K stage), and finally normalise O from TMEM
//    into the output.  The softmax waits for a PV only to reuse its P buffer
//    (two tiles back) or to rescale O, so softmax and MMAs overlap.
//  * V rows past the last key of a partial tile are zeroed before the PV MMA
//    reads them: pool slots past the sequence may hold anything, and a
//    zero-weight NaN would still poison the tensor-core sum.
#pragma once

#include "pa_common.cuh"
#include "pa_internal.h"
#include "tc_common.cuh"

namespace pa {

template <int D, int G>
struct TcCfg {
    static constexpr int BQ = 128 / G;                 // query rows per block
    static constexpr int M_USED = BQ * G;              // MMA rows in use (<= 128)
    static constexpr int BN = tc_tile_keys(D);         // keys per K/V tile
    static constexpr int KCH = D / 64;                 // 128-byte chunks of a head row
    static constexpr int Q_BYTES = KCH * 128 * 128;    // [KCH][128 rows][128 B]
    // K/V tile layout [KCH][BN rows][128 B] (the tensor cores' 128-byte-swizzled
    // canonical layout), one TMA box per (page, 128-byte chunk).
    static constexpr int KV_TILE = KCH * BN * 128;
    // K and V stages.  V is held from its load until the PV that follows the
    // softmax, K only until its S is done, so V gets the deeper ring.
    static constexpr int NK = D >= 256 ? 2 : (D >= 128 ? 3 : 4);
    static constexpr int NV = D >= 128 ? 3 : 4;
    static constexpr int OFF_K = Q_BYTES;
    static constexpr int OFF_V = OFF_K + NK * KV_TILE;
    static constexpr int NBAR = 1 + 2 * NK + 2 * NV + 2 + 2 + 2 + 2;
    static constexpr int OFF_BAR = OFF_V + NV * KV_TILE;
    static constexpr int OFF_RED = OFF_BAR + NBAR * 8;    // float [2 warpgroups][128 rows]
    static constexpr int PGR = 4;                         // page-id ring per producer (tiles)
    static constexpr int OFF_PG = OFF_RED + 2 * 128 * 4;  // int [2 producers][PGR][16]
    static constexpr int OFF_MISC = OFF_PG + 2 * PGR * 16 * 4;   // TMEM base, abort flag
    static constexpr int SMEM_BYTES = OFF_MISC + 16 + 1024;
    static constexpr int TMEM_COLS = 512;
    static constexpr int O_COL = 2 * BN;
    static constexpr int P_COL = 2 * BN + D;           // two P buffers, BN / 2 columns each
    // softmax warpgroup 0 (warps 0-3), K producer, MMA, V producer, softmax warpgroup 1
    static constexpr int THREADS = 352;
    static_assert(P_COL + BN <= TMEM_COLS, "TMEM columns");
    static_assert(SMEM_BYTES <= 227 * 1024, "shared memory");
    static_assert(BN % 64 == 0 && D % 64 == 0, "tile shape");
};

// One CTA per (request, KV head, query block of BQ rows).  Virtual block p
// belongs to the last request r with cu_seqlens_q[r] / BQ + r <= p (a
// request of n rows owns ceil(n / BQ) <= n / BQ + 1 of them); single-row
// requests and the padding of the numbering leave at once.
template <int D, int G>
__global__ void __launch_bounds__(352, 1)
    paged_prefill_tc_kernel(const __grid_constant__ CUtensorMap qmap,
                            const __grid_constant__ CUtensorMap kmap,
                            const __grid_constant__ CUtensorMap vmap, const TcArgs a) {
    using C = TcCfg<D, G>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = smem_u32(smem);
    const uint32_t q_smem = sbase;
    const uint32_t k_smem = sbase + C::OFF_K;
    const uint32_t v_smem = sbase + C::OFF_V;
    // barriers (each waited by one party in order, never two phases behind)
    const uint32_t bar_q = sbase + C::OFF_BAR;
    const uint32_t bar_k_full = bar_q + 8;                          // [NK]
    const uint32_t bar_k_empty = bar_k_full + 8 * C::NK;            // [NK]
    const uint32_t bar_v_full = bar_k_empty + 8 * C::NK;            // [NV]
    const uint32_t bar_v_empty = bar_v_full + 8 * C::NV;            // [NV]
    const uint32_t bar_s_full = bar_v_empty + 8 * C::NV;            // [2] S buffer
    const uint32_t bar_s_free = bar_s_full + 16;                    // [2]
    const uint32_t bar_p_full = bar_s_free + 16;                    // [2] P buffer
    const uint32_t bar_o_done = bar_p_full + 16;                    // [2] PV of P buffer b done
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + C::OFF_MISC);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + C::OFF_MISC + 8);

    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;
    const int h = blockIdx.y;
    const int Hq = a.num_q_heads;
    const int bs = a.block_size;

    // ---------------------------------------------------------------- work item
    const int p = blockIdx.x;
    int r;
    {
        int lo = 0, hi = a.num_seqs - 1;
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (a.cu_seqlens_q[mid] / C::BQ + mid <= p) lo = mid;
            else hi = mid - 1;
        }
        r = lo;
    }
    int i0, rows, kend;
    {
        const int c0r = a.cu_seqlens_q[r];
        const int nr = a.cu_seqlens_q[r + 1] - c0r;
        const int nblk = (nr + C::BQ - 1) / C::BQ;
        const int lp = p - (c0r / C::BQ + r);
        if (nr <= 1 || lp < 0 || lp >= nblk) return;
        const int qb = nblk - 1 - lp;                       // heaviest (last) block first
        i0 = qb * C::BQ;
        rows = min(C::BQ, nr - i0);
        int Nr = a.seq_lens_k[r];
        Nr = max(0, min(Nr, a.max_blocks_per_seq * bs));
        kend = max(0, a.causal ? min(Nr, Nr - nr + i0 + rows) : Nr);
    }
    const int rot_seed = p;
    const int c0 = a.cu_seqlens_q[r];
    const int n = a.cu_seqlens_q[r + 1] - c0;
    int N = a.seq_lens_k[r];
    N = max(0, min(N, a.max_blocks_per_seq * bs));
    const int ntiles = (kend + C::BN - 1) / C::BN;
    const int64_t row_base = (int64_t)c0 + i0;
    // The blocks of one request read the same keys: each starts at its own tile
    // and wraps around, so they do not all hit the same L2 lines at once (the
    // online softmax does not depend on the order of the tiles).
    const int rot = ntiles > 1
        ? (int)(((uint32_t)rot_seed * 2654435761u + (uint32_t)blockIdx.y * 40503u) % ntiles)
        : 0;
    auto tile_of = [&](int j) { const int jt = j + rot; return jt >= ntiles ? jt - ntiles : jt; };

    // ---------------------------------------------------------------- setup
    if (tid == 0) {
        mbar_init(bar_q, 1);
        for (int s = 0; s < C::NK; ++s) {
            mbar_init(bar_k_full + 8 * s, 1);
            mbar_init(bar_k_empty + 8 * s, 1);
        }
        for (int s = 0; s < C::NV; ++s) {
            mbar_init(bar_v_full + 8 * s, 1);
            mbar_init(bar_v_empty + 8 * s, 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(bar_s_full + 8 * b, 1);
            mbar_init(bar_s_free + 8 * b, 8);   // the 8 softmax warps
            mbar_init(bar_p_full + 8 * b, 8);
            mbar_init(bar_o_done + 8 * b, 1);
        }
        fence_barrier_init();
        *abort_flag = 0;
    }
    if (warp == 5) {
        tmem_alloc(smem_u32(tmem_slot), C::TMEM_COLS);
        tmem_relinquish();
    }
    if (C::M_USED < 128) {
        // Q rows past the (query row, head) pairs are never loaded: make them
        // zero so their score rows stay finite
        constexpr int PAD = (128 - C::M_USED) * 8;   // 16-byte chunks per region
        for (int c = 0; c < C::KCH; ++c)
            for (int q = tid; q < PAD; q += C::THREADS)
                *reinterpret_cast<uint4 *>(smem + c * 128 * 128 + C::M_USED * 128 + q * 16) =
                    make_uint4(0, 0, 0, 0);
        fence_proxy_async_smem();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == 4 || warp == 6) {
        // ============================================================ producers
        // warp 4 streams Q and the K tiles, warp 6 the V tiles; K stage j is
        // released as soon as S(j) is done, V stage j after PV(j).
        const bool is_k = (warp == 4);
        const CUtensorMap *map = is_k ? &kmap : &vmap;
        const uint32_t bar_full = is_k ? bar_k_full : bar_v_full;
        const uint32_t bar_empty = is_k ? bar_k_empty : bar_v_empty;
        const uint32_t stage0 = is_k ? k_smem : v_smem;
        const int NS = is_k ? C::NK : C::NV;             // stages of this ring
        const int BR = a.box_rows;
        const uint64_t pol_kv = policy_evict_last();   // re-read by the request's other blocks
        if (lane == 0) {
            prefetch_tensormap(map);
            if (is_k) {
                prefetch_tensormap(&qmap);
                mbar_arrive_expect_tx(bar_q, C::KCH * C::M_USED * 128);
                const uint64_t pol_q = policy_evict_first();
#pragma unroll
                for (int c = 0; c < C::KCH; ++c)
                    tma_load_3d(q_smem + c * 128 * 128, &qmap, c * 64, h * G, (int)row_base,
                                bar_q, pol_q);
            }
        }
        const int32_t *bt = a.block_tables + (int64_t)r * a.max_blocks_per_seq;
        // page ids of tile jj's boxes reach a shared ring slot by 4-byte cp.async
        // PGR - 1 tiles ahead (one commit group per tile), so no load is waited on
        int *pgr = reinterpret_cast<int *>(smem + C::OFF_PG) + (is_k ? 0 : C::PGR * 16);
        auto fetch_pages = [&](int jj) {
            if (jj < ntiles) {
                const int kt = tile_of(jj) * C::BN;
                const int nsub = (min(C::BN, kend - kt) + BR - 1) / BR;
                if (lane < nsub)
                    cp_async4(smem_u32(pgr + (jj % C::PGR) * 16 + lane), bt + (kt + lane * BR) / bs);
            }
            cp_async_commit();
        };
        for (int jj = 0; jj < C::PGR - 1; ++jj) fetch_pages(jj);
        int issued = 0;
        for (int j = 0; j < ntiles; ++j) {
            fetch_pages(j + C::PGR - 1);
            cp_async_wait<C::PGR - 1>();   // tile j's page ids have landed
            __syncwarp();
            const int *pgt = pgr + (j % C::PGR) * 16;
            const int st = j % NS;
            const int use = j / NS;
            int bad = 0;
            if (lane == 0 && use > 0)
                bad = !mbar_wait(bar_empty + 8 * st, (use - 1) & 1, a.err, abort_flag);
            if (__shfl_sync(0xffffffffu, bad, 0)) break;
            const int kt = tile_of(j) * C::BN;
            const int cnt = min(C::BN, kend - kt);
            const int nsub = (cnt + BR - 1) / BR;
            // (failure-path test: the K tile 0 is neither armed nor loaded, so the
            // MMA warp's bounded wait for it runs out)
            const bool skip = is_k && j == 0 && a.test_skip_first_k;
            if (lane == 0 && !skip) mbar_arrive_expect_tx(bar_full + 8 * st, nsub * C::KCH * BR * 128);
            __syncwarp();
            const uint32_t dst = stage0 + st * C::KV_TILE;
            // one box per lane (page run u = lane / KCH, 128-byte chunk lane % KCH):
            // a box issue holds its warp for ~120 ns, so spreading the tile's
            // boxes over the lanes keeps many issues in flight
            {
                const int u = lane / C::KCH, c = lane % C::KCH;
                if (u < nsub && !skip) {
                    const int row0 = pgt[u] * bs + (kt + u * BR) % bs;
                    tma_load_3d(dst + c * C::BN * 128 + u * BR * 128, map, c * 64, h, row0,
                                bar_full + 8 * st, pol_kv);
                }
            }
            __syncwarp();
            issued = j + 1;
        }
        cp_async_wait<0>();   // page-id copies in flight land before the warp leaves
        if (lane == 0) {
            if (is_k) mbar_drain(bar_q, 0, kWaitLimitCycles / 8);
            for (int j = max(0, issued - NS); j < issued; ++j)
                mbar_drain(bar_full + 8 * (j % NS), (j / NS) & 1,
                           kWaitLimitCycles / 8);
        }
    } else if (warp == 5) {
        // ============================================================ MMA issuer
        if (lane == 0 && ntiles > 0) {
            constexpr uint32_t IDESC_S = idesc_bf16_f32(128, C::BN, 0, 0);
            constexpr uint32_t IDESC_O = idesc_bf16_f32(128, D, 0, 1);
            mbar_wait(bar_q, 0, a.err, abort_flag);
            auto issue_pv = [&](int jj) {
                const int pb = jj & 1;
                const int stp = jj % C::NV;
                mbar_wait(bar_p_full + 8 * pb, (jj >> 1) & 1, a.err, abort_flag);
                mbar_wait(bar_v_full + 8 * stp, (jj / C::NV) & 1, a.err, abort_flag);
                tc_fence_after();
                const uint32_t vs = v_smem + stp * C::KV_TILE;
                const uint32_t pt = tmem + C::P_COL + pb * (C::BN / 2);   // P in TMEM
#pragma unroll
                for (int kk = 0; kk < C::BN / 16; ++kk) {
                    // V as MN-major B: atoms of 64 d x 8 keys; LBO steps d-chunks, SBO
                    // steps 8-key groups; one k-step is 16 keys (8 P columns)
                    const uint64_t bd = smem_desc_sw128(vs + kk * 16 * 128, C::BN * 128, 1024);
                    tc_mma_bf16_ts(tmem + C::O_COL, pt + kk * 8, bd, IDESC_O,
                                   (jj > 0 || kk > 0) ? 1u : 0u);
                }
                tc_commit(bar_o_done + 8 * pb);
                tc_commit(bar_v_empty + 8 * stp);
            };
            for (int j = 0; j < ntiles; ++j) {
                const int st = j % C::NK;
                const int sb = j & 1;
                mbar_wait(bar_k_full + 8 * st, (j / C::NK) & 1, a.err, abort_flag);
                if (j >= 2) mbar_wait(bar_s_free + 8 * sb, ((j >> 1) - 1) & 1, a.err, abort_flag);
                tc_fence_after();
                const uint32_t ks = k_smem + st * C::KV_TILE;
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint32_t off = (kk & 3) * 32;   // 16 bf16 within the 128-B row
                    const uint64_t ad =
                        smem_desc_sw128(q_smem + (kk >> 2) * 128 * 128 + off, 16, 1024);
                    const uint64_t bd =
                        smem_desc_sw128(ks + (kk >> 2) * C::BN * 128 + off, 16, 1024);
                    tc_mma_bf16(tmem + sb * C::BN, ad, bd, IDESC_S, kk > 0 ? 1u : 0u);
                }
                tc_commit(bar_s_full + 8 * sb);
                tc_commit(bar_k_empty + 8 * st);
                if (j >= 1) issue_pv(j - 1);
            }
            issue_pv(ntiles - 1);
            // every MMA must be finished before TMEM is freed (bounded wait that
            // also holds on an aborted pipeline)
            mbar_drain(bar_o_done + 8 * ((ntiles - 1) & 1), ((ntiles - 1) >> 1) & 1,
                       kWaitLimitCycles / 8);
        }
    } else {
        // ============================================================ softmax
        // Two warpgroups share every tile: warpgroup wg takes keys
        // [wg * BN / 2, (wg + 1) * BN / 2) of each row (TMEM lane), and half of
        // O's columns when O is rescaled or written out.  Row maxima and sums
        // of the two halves meet in shared memory.
        constexpr int HB = C::BN / 2;                     // keys per warpgroup and tile
        const int wg = warp >= 7 ? 1 : 0;
        const int m = ((warp & 3) << 5) | lane;           // MMA row = TMEM lane
        const int sm_tid = wg * 128 + m;                  // 0..255 over both warpgroups
        const int kb = wg * HB;                           // first key of this half
        const int i = m / G, g = m % G;
        const bool row_ok = (m < C::M_USED) && (i < rows);
        const int qi = i0 + i;
        const int lim = min(N - 1, a.causal ? N - n + qi : N - 1);   // last visible key
        // keys up to lim_all are visible to every row of the block
        const int lim_all = min(N - 1, a.causal ? N - n + i0 : N - 1);
        const uint32_t t_lane = tmem + ((uint32_t)((warp & 3) * 32) << 16);
        float *xr = reinterpret_cast<float *>(smem + C::OFF_RED);   // [2][128]
        // the other half's value of this row (write, meet, read, meet)
        auto exchange = [&](float v) -> float {
            xr[wg * 128 + m] = v;
            named_barrier_sync(1, 256);
            const float o = xr[(1 - wg) * 128 + m];
            named_barrier_sync(1, 256);
            return o;
        };
        const float qs = a.qscale;
        float m_run = -INFINITY, m_ref = -INFINITY, l = 0.f;   // l: this half's sum
        for (int j = 0; j < ntiles; ++j) {
            const int sb = j & 1;
            const int pb = j & 1;
            const int st = j % C::NV;                     // V stage of tile j
            mbar_wait(bar_s_full + 8 * sb, (j >> 1) & 1, a.err, abort_flag);
            tc_fence_after();
            float s[HB];
#pragma unroll
            for (int c = 0; c < HB / 32; ++c)
                tmem_ld32(t_lane + sb * C::BN + kb + 32 * c, s + 32 * c);
            tmem_wait_ld();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar_s_free + 8 * sb);

            // Tiles that reach past a row's last visible key are masked and scaled
            // here (masked keys become -inf); fully visible tiles keep raw scores
            // and are scaled inside the exponent.  sc = scale still to apply.
            const int kt0 = tile_of(j) * C::BN;
            const bool tmask = kt0 + C::BN - 1 > lim_all;
            if (tmask) {
#pragma unroll
                for (int c = 0; c < HB; ++c)
                    s[c] = (row_ok && kt0 + kb + c <= lim) ? s[c] * qs : -INFINITY;
            }
            const float sc = tmask ? 1.f : qs;
            // max of sc * s over this half (8 independent chains), via max(s) or max(-s)
            const bool neg = sc < 0.f;
            float mx[8];
#pragma unroll
            for (int k = 0; k < 8; ++k) mx[k] = neg ? -s[k] : s[k];
#pragma unroll
            for (int c = 8; c < HB; c += 8)
#pragma unroll
                for (int k = 0; k < 8; ++k) mx[k] = fmaxf(mx[k], neg ? -s[c + k] : s[c + k]);
#pragma unroll
            for (int k = 4; k > 0; k >>= 1)
#pragma unroll
                for (int q = 0; q < k; ++q) mx[q] = fmaxf(mx[q], mx[q + k]);
            const float hmax = mx[0] == -INFINITY ? -INFINITY : mx[0] * fabsf(sc);
            const float tmax = fmaxf(hmax, exchange(hmax));   // the whole row's tile max
            const float m_new = fmaxf(m_run, tmax);
            m_run = m_new;
            const bool need = (m_new != -INFINITY) && (m_ref == -INFINITY || m_new > m_ref + 8.f);

            // Value rows past the tile's last key may hold anything: zero them
            // before the PV MMA (a zero weight times NaN is still NaN).
            const int cnt = min(C::BN, kend - kt0);
            if (cnt < C::BN) {
                mbar_wait(bar_v_full + 8 * st, (j / C::NV) & 1, a.err, abort_flag);
                uint8_t *vsp = smem + C::OFF_V + st * C::KV_TILE;
                const int nchunk = (C::BN - cnt) * C::KCH * 8;   // 16-byte pieces to clear
                for (int q = sm_tid; q < nchunk; q += 256) {
                    const int k = cnt + q / (C::KCH * 8);          // key row of the tile
                    const int c = (q >> 3) % C::KCH;               // 128-byte chunk of the row
                    const int off = c * C::BN * 128 + k * 128;
                    *reinterpret_cast<uint4 *>(vsp + off + (q & 7) * 16) = make_uint4(0, 0, 0, 0);
                }
            }
            // O changes only when a row's reference max moves: then PV(j-1) must be
            // done.  Each warpgroup rescales its half of O's columns.
            if (j >= 1 && __any_sync(0xffffffffu, need)) {
                mbar_wait(bar_o_done + 8 * ((j - 1) & 1), ((j - 1) >> 1) & 1, a.err, abort_flag);
                tc_fence_after();
                const float f = need ? (m_ref == -INFINITY ? 0.f : exp2f(m_ref - m_new)) : 1.f;
#pragma unroll 1
                for (int c = 0; c < D / 64; ++c) {
                    float o[32];
                    const uint32_t oa = t_lane + C::O_COL + wg * (D / 2) + 32 * c;
                    tmem_ld32(oa, o);
                    tmem_wait_ld();
#pragma unroll
                    for (int e = 0; e < 32; ++e) o[e] *= f;
                    tmem_st32(oa, o);
                }
                tmem_wait_st();
            }
            if (need) {
                l *= (m_ref == -INFINITY) ? 0.f : exp2f(m_ref - m_new);
                m_ref = m_new;
            }
            // P buffer pb was last read by PV(j-2)
            if (j >= 2) mbar_wait(bar_o_done + 8 * pb, ((j >> 1) - 1) & 1, a.err, abort_flag);
            // P = 2^(sc * s - m_ref) as bf16 (masked keys: 2^-inf = 0) into this
            // row's TMEM lane, two keys per 32-bit column: the A operand of PV
            const float2 qs2 = make_float2(sc, sc);
            const float mu = (m_ref == -INFINITY) ? 0.f : -m_ref;
            const float2 mu2 = make_float2(mu, mu);
            float2 sum2[4];
#pragma unroll
            for (int k = 0; k < 4; ++k) sum2[k] = make_float2(0.f, 0.f);
            const uint32_t pt = t_lane + C::P_COL + pb * (C::BN / 2) + kb / 2;
#pragma unroll
            for (int k16 = 0; k16 < HB / 16; ++k16) {
                uint32_t w8[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    float2 x = __ffma2_rn(make_float2(s[k16 * 16 + 2 * e], s[k16 * 16 + 2 * e + 1]),
                                          qs2, mu2);
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
            if (lane == 0) mbar_arrive(bar_p_full + 8 * pb);
        }
        // ---- epilogue: out = O / (l + sink term); each warpgroup writes half of D
        if (ntiles > 0) {
            mbar_wait(bar_o_done + 8 * ((ntiles - 1) & 1), ((ntiles - 1) >> 1) & 1, a.err,
                      abort_flag);
            tc_fence_after();
        }
        const float l_row = l + exchange(l);
        float scale_out = 0.f;
        if (l_row > 0.f) {
            if (a.sinks) {
                const float sk2 = a.sinks[h * G + g] * kLog2e;
                const float M2 = fmaxf(m_ref, sk2);
                const float f = exp2f(m_ref - M2);
                scale_out = f / (l_row * f + exp2f(sk2 - M2));
            } else {
                scale_out = 1.f / l_row;
            }
        }
        __nv_bfloat16 *orow = reinterpret_cast<__nv_bfloat16 *>(a.out) +
                              ((row_base + i) * Hq + (int64_t)h * G + g) * D + wg * (D / 2);
#pragma unroll 1
        for (int c = 0; c < D / 64; ++c) {
            float o[32];
            if (ntiles > 0) {
                tmem_ld32(t_lane + C::O_COL + wg * (D / 2) + 32 * c, o);
                tmem_wait_ld();
            } else {
#pragma unroll
                for (int e = 0; e < 32; ++e) o[e] = 0.f;
            }
            if (row_ok) {
                uint4 *dst = reinterpret_cast<uint4 *>(orow + 32 * c);
#pragma unroll
                for (int q = 0; q < 4; ++q)
                    dst[q] = make_uint4(pack_bf16x2(o[8 * q + 0] * scale_out, o[8 * q + 1] * scale_out),
                                        pack_bf16x2(o[8 * q + 2] * scale_out, o[8 * q + 3] * scale_out),
                                        pack_bf16x2(o[8 * q + 4] * scale_out, o[8 * q + 5] * scale_out),
                                        pack_bf16x2(o[8 * q + 6] * scale_out, o[8 * q + 7] * scale_out));
            }
        }
    }

    // ---------------------------------------------------------------- teardown
    tc_fence_before();
    __syncthreads();
    if (warp == 5) {
        tc_fence_after();
        tmem_dealloc(tmem, C::TMEM_COLS);
    }
}

template <int D, int G>
cudaError_t launch_prefill_tc_t(const CUtensorMap &qmap, const CUtensorMap &kmap,
                                const CUtensorMap &vmap, const TcArgs &a, dim3 grid,
                                cudaStream_t stream) {
    using C = TcCfg<D, G>;
    auto kern = paged_prefill_tc_kernel<D, G>;
    static bool configured = false;
    if (!configured) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             C::SMEM_BYTES);
        if (e != cudaSuccess) return e;
        configured = true;
    }
    kern<<<grid, C::THREADS, C::SMEM_BYTES, stream>>>(qmap, kmap, vmap, a);
    return cudaGetLastError();
}

template <int D>
cudaError_t launch_prefill_tc_group(int group, const CUtensorMap &qmap, const CUtensorMap &kmap,
                                    const CUtensorMap &vmap, const TcArgs &a, dim3 grid,
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
