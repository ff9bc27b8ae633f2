// prefill_tc.cuh -- multi-query rows (speculative-verify windows, prefill
// chunks) on the 5th-generation tensor cores.
//
// What it computes (aisignalhub.me, "packed queries and paged KV"; kwkr.cn,
// "What is Paged Attention" and the kernel table): for the query rows of a
// request with n > 1 rows, softmax(scale * Q K^T) V over the request's paged
// keys, causal rows bottom-right aligned (row i sees keys j <= N - n + i),
// with the sink logit of each head counted once in the denominator.
//
// GB300 design (one CTA per (request, KV head, query block), 224 threads):
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
//  * Warps 0-3 (softmax, one thread per TMEM lane = MMA row): load S, mask and
//    scale into the log2 domain, keep a running max with lazy rescaling of O
//    (only when the max grows by more than 2^8), write P as bf16 into one of
//    two shared-memory buffers for the PV MMA, and finally normalise O from
//    TMEM into the output.  The softmax waits for a PV only to reuse its P
//    buffer (two tiles back) or to rescale O, so softmax and MMAs overlap.
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
    static constexpr int NSTAGE = D >= 128 ? 2 : 3;    // K stages (and as many V stages)
    static constexpr int P_BYTES = (BN / 64) * 128 * 128;   // [BN/64][128 rows][128 B]
    static constexpr int OFF_K = Q_BYTES;
    static constexpr int OFF_V = OFF_K + NSTAGE * KV_TILE;
    static constexpr int OFF_P = OFF_V + NSTAGE * KV_TILE;  // two P buffers
    static constexpr int NBAR = 1 + 4 * NSTAGE + 2 + 2 + 2 + 2;
    static constexpr int OFF_BAR = OFF_P + 2 * P_BYTES;
    static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;   // TMEM base, abort flag
    static constexpr int SMEM_BYTES = OFF_MISC + 16 + 1024;
    static constexpr int TMEM_COLS = 512;
    static constexpr int O_COL = 2 * BN;
    static constexpr int THREADS = 224;                // 4 softmax + K producer + MMA + V producer
    static_assert(O_COL + D <= TMEM_COLS, "TMEM columns");
    static_assert(SMEM_BYTES <= 227 * 1024, "shared memory");
    static_assert(BN % 64 == 0 && D % 64 == 0, "tile shape");
};

// PAIR: a cluster of two CTAs takes two adjacent query blocks of one request
// and KV head; both walk the same K/V tiles and each CTA loads half of every
// tile with TMA multicast into both, halving the per-SM K/V traffic.  Without
// PAIR a CTA takes a request whose rows fit one query block.
template <int D, int G, bool PAIR>
__global__ void __launch_bounds__(224, 1)
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
    const uint32_t p_smem = sbase + C::OFF_P;
    // barriers (each waited by one party in order, never two phases behind)
    const uint32_t bar_q = sbase + C::OFF_BAR;
    const uint32_t bar_k_full = bar_q + 8;                          // [NSTAGE]
    const uint32_t bar_k_empty = bar_k_full + 8 * C::NSTAGE;        // [NSTAGE]
    const uint32_t bar_v_full = bar_k_empty + 8 * C::NSTAGE;        // [NSTAGE]
    const uint32_t bar_v_empty = bar_v_full + 8 * C::NSTAGE;        // [NSTAGE]
    const uint32_t bar_s_full = bar_v_empty + 8 * C::NSTAGE;        // [2] S buffer
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
    int r, i0, rows, kend, rot_seed;
    if (PAIR) {
        // Virtual pair p belongs to the last request r with cu[r] / (2 BQ) + r <= p;
        // the two CTAs of a cluster (rank 0, 1) take blocks 2l and 2l + 1.
        const int p = blockIdx.x >> 1;
        const int rank = blockIdx.x & 1;
        int lo = 0, hi = a.num_seqs - 1;
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (a.cu_seqlens_q[mid] / (2 * C::BQ) + mid <= p) lo = mid;
            else hi = mid - 1;
        }
        r = lo;
        const int c0r = a.cu_seqlens_q[r];
        const int nr = a.cu_seqlens_q[r + 1] - c0r;
        const int nblk = (nr + C::BQ - 1) / C::BQ;
        const int npairs = (nblk + 1) / 2;
        const int lp = p - (c0r / (2 * C::BQ) + r);
        if (nblk < 2 || lp < 0 || lp >= npairs) return;   // whole cluster leaves together
        const int lpp = npairs - 1 - lp;                    // heaviest pair first
        const int qb = 2 * lpp + rank;                      // may be past the last block
        const int qb_hi = min(2 * lpp + 1, nblk - 1);       // the pair's heavier block
        i0 = qb * C::BQ;
        rows = qb < nblk ? min(C::BQ, nr - i0) : 0;
        int Nr = a.seq_lens_k[r];
        Nr = max(0, min(Nr, a.max_blocks_per_seq * bs));
        const int i0_hi = qb_hi * C::BQ;
        const int rows_hi = min(C::BQ, nr - i0_hi);
        kend = max(0, a.causal ? min(Nr, Nr - nr + i0_hi + rows_hi) : Nr);
        rot_seed = p;
    } else {
        r = blockIdx.x;
        const int nr = a.cu_seqlens_q[r + 1] - a.cu_seqlens_q[r];
        if (nr <= 1 || nr > C::BQ) return;                 // decode rows / paired launch
        int Nr = a.seq_lens_k[r];
        Nr = max(0, min(Nr, a.max_blocks_per_seq * bs));
        i0 = 0;
        rows = nr;
        kend = max(0, a.causal ? min(Nr, Nr - nr + rows) : Nr);
        rot_seed = blockIdx.x;
    }
    const int c0 = a.cu_seqlens_q[r];
    const int n = a.cu_seqlens_q[r + 1] - c0;
    int N = a.seq_lens_k[r];
    N = max(0, min(N, a.max_blocks_per_seq * bs));
    const int ntiles = (kend + C::BN - 1) / C::BN;
    const int64_t row_base = (int64_t)c0 + i0;
    // The blocks of one request read the same keys: each starts at its own tile
    // and wraps around, so they do not all hit the same L2 lines at once (the
    // online softmax does not depend on the order of the tiles).  Both CTAs of a
    // pair use the same order.
    const int rot = ntiles > 1
        ? (int)(((uint32_t)rot_seed * 2654435761u + (uint32_t)blockIdx.y * 40503u) % ntiles)
        : 0;
    auto tile_of = [&](int j) { const int jt = j + rot; return jt >= ntiles ? jt - ntiles : jt; };
    constexpr uint16_t kPairMask = 0x3;

    // ---------------------------------------------------------------- setup
    if (tid == 0) {
        mbar_init(bar_q, 1);
        for (int s = 0; s < C::NSTAGE; ++s) {
            mbar_init(bar_k_full + 8 * s, 1);
            mbar_init(bar_k_empty + 8 * s, PAIR ? 2 : 1);   // both CTAs release a stage
            mbar_init(bar_v_full + 8 * s, 1);
            mbar_init(bar_v_empty + 8 * s, PAIR ? 2 : 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(bar_s_full + 8 * b, 1);
            mbar_init(bar_s_free + 8 * b, 4);
            mbar_init(bar_p_full + 8 * b, 4);
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
    if (PAIR) cluster_sync();   // the peer's barriers exist before any multicast
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
        // page ids of a tile's boxes: lane u holds box u's page, loaded one tile ahead
        auto pages_of = [&](int j) -> int {
            if (j >= ntiles) return 0;
            const int kt = tile_of(j) * C::BN;
            const int nsub = (min(C::BN, kend - kt) + BR - 1) / BR;
            return lane < nsub ? bt[(kt + lane * BR) / bs] : 0;
        };
        int pg_cur = pages_of(0);
        int issued = 0;
        for (int j = 0; j < ntiles; ++j) {
            const int pg_next = pages_of(j + 1);
            const int st = j % C::NSTAGE;
            const int use = j / C::NSTAGE;
            int bad = 0;
            if (lane == 0 && use > 0)
                bad = !mbar_wait(bar_empty + 8 * st, (use - 1) & 1, a.err, abort_flag);
            if (__shfl_sync(0xffffffffu, bad, 0)) break;
            const int kt = tile_of(j) * C::BN;
            const int cnt = min(C::BN, kend - kt);
            const int nsub = (cnt + BR - 1) / BR;
            if (lane == 0) mbar_arrive_expect_tx(bar_full + 8 * st, nsub * C::KCH * BR * 128);
            __syncwarp();
            const uint32_t dst = stage0 + st * C::KV_TILE;
            // paired: rank 0 loads the first half of the boxes, rank 1 the rest,
            // each multicast to both CTAs (every CTA expects the whole tile)
            const int u_lo = PAIR ? ((blockIdx.x & 1) ? (nsub + 1) / 2 : 0) : 0;
            const int u_hi = PAIR ? ((blockIdx.x & 1) ? nsub : (nsub + 1) / 2) : nsub;
            for (int u = 0; u < nsub; ++u) {
                const int page = __shfl_sync(0xffffffffu, pg_cur, u);
                if (lane == 0 && u >= u_lo && u < u_hi) {
                    const int row0 = page * bs + (kt + u * BR) % bs;
#pragma unroll
                    for (int c = 0; c < C::KCH; ++c) {
                        const uint32_t d = dst + c * C::BN * 128 + u * BR * 128;
                        if (PAIR)
                            tma_load_3d_mc(d, map, c * 64, h, row0, bar_full + 8 * st,
                                           kPairMask, pol_kv);
                        else
                            tma_load_3d(d, map, c * 64, h, row0, bar_full + 8 * st, pol_kv);
                    }
                }
            }
            __syncwarp();
            pg_cur = pg_next;
            issued = j + 1;
        }
        if (lane == 0) {
            if (is_k) mbar_drain(bar_q, 0, kWaitLimitCycles / 8);
            for (int j = max(0, issued - C::NSTAGE); j < issued; ++j)
                mbar_drain(bar_full + 8 * (j % C::NSTAGE), (j / C::NSTAGE) & 1,
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
                const int stp = jj % C::NSTAGE;
                mbar_wait(bar_p_full + 8 * pb, (jj >> 1) & 1, a.err, abort_flag);
                mbar_wait(bar_v_full + 8 * stp, (jj / C::NSTAGE) & 1, a.err, abort_flag);
                tc_fence_after();
                const uint32_t vs = v_smem + stp * C::KV_TILE;
                const uint32_t ps = p_smem + pb * C::P_BYTES;
#pragma unroll
                for (int kk = 0; kk < C::BN / 16; ++kk) {
                    const uint64_t ad =
                        smem_desc_sw128(ps + (kk >> 2) * 128 * 128 + (kk & 3) * 32, 16, 1024);
                    // V as MN-major B: atoms of 64 d x 8 keys; LBO steps d-chunks, SBO
                    // steps 8-key groups; one k-step is 16 keys
                    const uint64_t bd = smem_desc_sw128(vs + kk * 16 * 128, C::BN * 128, 1024);
                    tc_mma_bf16(tmem + C::O_COL, ad, bd, IDESC_O, (jj > 0 || kk > 0) ? 1u : 0u);
                }
                tc_commit(bar_o_done + 8 * pb);
                if (PAIR) tc_commit_mc(bar_v_empty + 8 * stp, kPairMask);
                else tc_commit(bar_v_empty + 8 * stp);
            };
            for (int j = 0; j < ntiles; ++j) {
                const int st = j % C::NSTAGE;
                const int sb = j & 1;
                mbar_wait(bar_k_full + 8 * st, (j / C::NSTAGE) & 1, a.err, abort_flag);
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
                if (PAIR) tc_commit_mc(bar_k_empty + 8 * st, kPairMask);
                else tc_commit(bar_k_empty + 8 * st);
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
        const int m = tid;                                // MMA row = TMEM lane
        const int i = m / G, g = m % G;
        const bool row_ok = (m < C::M_USED) && (i < rows);
        const int qi = i0 + i;
        const int lim = min(N - 1, a.causal ? N - n + qi : N - 1);   // last visible key
        // keys up to lim_all are visible to every row of the block
        const int lim_all = min(N - 1, a.causal ? N - n + i0 : N - 1);
        const uint32_t t_lane = tmem + ((uint32_t)(warp * 32) << 16);
        const float qs = a.qscale;
        float m_run = -INFINITY, m_ref = -INFINITY, l = 0.f;
        for (int j = 0; j < ntiles; ++j) {
            const int sb = j & 1;
            const int pb = j & 1;
            const int st = j % C::NSTAGE;
            mbar_wait(bar_s_full + 8 * sb, (j >> 1) & 1, a.err, abort_flag);
            tc_fence_after();
            float s[C::BN];
#pragma unroll
            for (int c = 0; c < C::BN / 32; ++c) tmem_ld32(t_lane + sb * C::BN + 32 * c, s + 32 * c);
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
                for (int c = 0; c < C::BN; ++c)
                    s[c] = (row_ok && kt0 + c <= lim) ? s[c] * qs : -INFINITY;
            }
            const float sc = tmask ? 1.f : qs;
            // row max (8 independent chains) of sc * s, via max(s) or max(-s)
            const bool neg = sc < 0.f;
            float mx[8];
#pragma unroll
            for (int k = 0; k < 8; ++k) mx[k] = neg ? -s[k] : s[k];
#pragma unroll
            for (int c = 8; c < C::BN; c += 8)
#pragma unroll
                for (int k = 0; k < 8; ++k) mx[k] = fmaxf(mx[k], neg ? -s[c + k] : s[c + k]);
#pragma unroll
            for (int k = 4; k > 0; k >>= 1)
#pragma unroll
                for (int q = 0; q < k; ++q) mx[q] = fmaxf(mx[q], mx[q + k]);
            const float tmax = mx[0] == -INFINITY ? -INFINITY : mx[0] * fabsf(sc);
            const float m_new = fmaxf(m_run, tmax);
            m_run = m_new;
            const bool need = (m_new != -INFINITY) && (m_ref == -INFINITY || m_new > m_ref + 8.f);

            // Value rows past the tile's last key may hold anything: zero them
            // before the PV MMA (a zero weight times NaN is still NaN).
            const int cnt = min(C::BN, kend - kt0);
            if (cnt < C::BN) {
                mbar_wait(bar_v_full + 8 * st, (j / C::NSTAGE) & 1, a.err, abort_flag);
                uint8_t *vsp = smem + C::OFF_V + st * C::KV_TILE;
                const int nchunk = (C::BN - cnt) * C::KCH * 8;   // 16-byte pieces to clear
                for (int q = tid; q < nchunk; q += 128) {
                    const int k = cnt + q / (C::KCH * 8);          // key row of the tile
                    const int c = (q >> 3) % C::KCH;               // 128-byte chunk of the row
                    const int off = c * C::BN * 128 + k * 128;
                    *reinterpret_cast<uint4 *>(vsp + off + (q & 7) * 16) = make_uint4(0, 0, 0, 0);
                }
            }
            // O changes only when a row's reference max moves: then PV(j-1) must be done.
            if (j >= 1 && __any_sync(0xffffffffu, need)) {
                mbar_wait(bar_o_done + 8 * ((j - 1) & 1), ((j - 1) >> 1) & 1, a.err, abort_flag);
                tc_fence_after();
                const float f = need ? (m_ref == -INFINITY ? 0.f : exp2f(m_ref - m_new)) : 1.f;
#pragma unroll 1
                for (int c = 0; c < D / 32; ++c) {
                    float o[32];
                    tmem_ld32(t_lane + C::O_COL + 32 * c, o);
                    tmem_wait_ld();
#pragma unroll
                    for (int e = 0; e < 32; ++e) o[e] *= f;
                    tmem_st32(t_lane + C::O_COL + 32 * c, o);
                }
                tmem_wait_st();
            }
            if (need) {
                l *= (m_ref == -INFINITY) ? 0.f : exp2f(m_ref - m_new);
                m_ref = m_new;
            }
            // P buffer pb was last read by PV(j-2)
            if (j >= 2) mbar_wait(bar_o_done + 8 * pb, ((j >> 1) - 1) & 1, a.err, abort_flag);
            // P = 2^(sc * s - m_ref) as bf16 (masked keys: 2^-inf = 0),
            // row m of the K-major 128-byte-swizzled A tile
            const float2 qs2 = make_float2(sc, sc);
            const float mu = (m_ref == -INFINITY) ? 0.f : -m_ref;
            const float2 mu2 = make_float2(mu, mu);
            float2 sum2[4];
#pragma unroll
            for (int k = 0; k < 4; ++k) sum2[k] = make_float2(0.f, 0.f);
            const uint32_t ps = p_smem + pb * C::P_BYTES;
#pragma unroll
            for (int k8 = 0; k8 < C::BN / 8; ++k8) {
                uint32_t w4[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    float2 x = __ffma2_rn(make_float2(s[k8 * 8 + 2 * e], s[k8 * 8 + 2 * e + 1]),
                                          qs2, mu2);
                    x.x = ex2_approx(x.x);
                    x.y = ex2_approx(x.y);
                    sum2[e] = __fadd2_rn(sum2[e], x);
                    w4[e] = pack_bf16x2(x.x, x.y);
                }
                const uint32_t addr = ps + (k8 >> 3) * 128 * 128 + m * 128 +
                                      (((k8 & 7) ^ (m & 7)) << 4);
                sts128(addr, w4[0], w4[1], w4[2], w4[3]);
            }
            const float2 sa = __fadd2_rn(sum2[0], sum2[1]);
            const float2 sbb = __fadd2_rn(sum2[2], sum2[3]);
            l += (sa.x + sa.y) + (sbb.x + sbb.y);
            fence_proxy_async_smem();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar_p_full + 8 * pb);
        }
        // ---- epilogue: out = O / (l + sink term)
        if (ntiles > 0) {
            mbar_wait(bar_o_done + 8 * ((ntiles - 1) & 1), ((ntiles - 1) >> 1) & 1, a.err,
                      abort_flag);
            tc_fence_after();
        }
        float scale_out = 0.f;
        if (l > 0.f) {
            if (a.sinks) {
                const float sk2 = a.sinks[h * G + g] * kLog2e;
                const float M2 = fmaxf(m_ref, sk2);
                const float f = exp2f(m_ref - M2);
                scale_out = f / (l * f + exp2f(sk2 - M2));
            } else {
                scale_out = 1.f / l;
            }
        }
        __nv_bfloat16 *orow = reinterpret_cast<__nv_bfloat16 *>(a.out) +
                              ((row_base + i) * Hq + (int64_t)h * G + g) * D;
#pragma unroll 1
        for (int c = 0; c < D / 32; ++c) {
            float o[32];
            if (ntiles > 0) {
                tmem_ld32(t_lane + C::O_COL + 32 * c, o);
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
    // no CTA of a pair leaves while its peer may still multicast into it or
    // arrive on its barriers
    if (PAIR) cluster_sync();
}

template <int D, int G, bool PAIR>
cudaError_t launch_prefill_tc_t(const CUtensorMap &qmap, const CUtensorMap &kmap,
                                const CUtensorMap &vmap, const TcArgs &a, dim3 grid,
                                cudaStream_t stream) {
    using C = TcCfg<D, G>;
    auto kern = paged_prefill_tc_kernel<D, G, PAIR>;
    static bool configured = false;
    if (!configured) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             C::SMEM_BYTES);
        if (e != cudaSuccess) return e;
        if (PAIR) {
            e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 0);
            if (e != cudaSuccess) return e;
        }
        configured = true;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(C::THREADS);
    cfg.dynamicSmemBytes = C::SMEM_BYTES;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    if (PAIR) {
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = 2;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
    }
    cudaError_t e = cudaLaunchKernelEx(&cfg, kern, qmap, kmap, vmap, a);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

template <int D, bool PAIR>
cudaError_t launch_prefill_tc_group(int group, const CUtensorMap &qmap, const CUtensorMap &kmap,
                                    const CUtensorMap &vmap, const TcArgs &a, dim3 grid,
                                    cudaStream_t stream) {
    switch (group) {
        case 1: return launch_prefill_tc_t<D, 1, PAIR>(qmap, kmap, vmap, a, grid, stream);
        case 2: return launch_prefill_tc_t<D, 2, PAIR>(qmap, kmap, vmap, a, grid, stream);
        case 3: return launch_prefill_tc_t<D, 3, PAIR>(qmap, kmap, vmap, a, grid, stream);
        case 4: return launch_prefill_tc_t<D, 4, PAIR>(qmap, kmap, vmap, a, grid, stream);
        case 5: return launch_prefill_tc_t<D, 5, PAIR>(qmap, kmap, vmap, a, grid, stream);
        case 6: return launch_prefill_tc_t<D, 6, PAIR>(qmap, kmap, vmap, a, grid, stream);
        case 7: return launch_prefill_tc_t<D, 7, PAIR>(qmap, kmap, vmap, a, grid, stream);
        case 8: return launch_prefill_tc_t<D, 8, PAIR>(qmap, kmap, vmap, a, grid, stream);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace pa
