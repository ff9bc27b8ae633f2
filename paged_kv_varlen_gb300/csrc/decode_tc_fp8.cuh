// decode_tc_fp8.cuh -- single-query (decode) requests over the quantised KV
// cache on the 5th-generation tensor cores: bf16 queries and outputs, K and V
// rows stored as E4M3 codes with a float32 scale per (token, KV head) row.
//
// What it computes: the decode attention of decode_tc.cuh (kwkr.cn, "What is
// Paged Attention": the GQA decode section and trick 4) over the dequantised
// rows value(code) * scale -- the quantised cache is this library's reading of
// the TurboQuant helpers named by lqnn.cn (layered architecture, section 5).
//
// GB300 design (persistent: one CTA per SM, 480 threads).  The work plan, the
// item order, the split partials and the softmax are those of the bf16 kernel;
// what changes is how the rows reach the tensor cores:
//  * Warps 4 and 7 stream the K codes, warps 5 and 8 the V codes, by TMA into
//    two rings of 16 KB stages (128 keys x 128 codes, 128-byte swizzle): one
//    box per run of box_rows keys of a page, one box per lane.  A code row is
//    128 bytes, so one box covers all 128 dims of a chunk -- half the boxes of
//    the bf16 kernel per key.
//  * S^T = K . Q^T runs on the codes as they land: an E4M3 x E4M3 MMA
//    (kind::f8f6f4, fp32 accumulation) with the K stage as the A operand.  The
//    queries are split exactly into two E4M3 parts: scaled by a power of two
//    2^e so that the item's largest |q| lies in [128, 256), each value is
//    hi + lo with hi its nearest E4M3 and lo the E4M3 of the remainder -- the
//    sum holds all eight significant bits of a bf16 for values down to 2^-2
//    (and within 2^-10 absolute below).  One MMA of N = 32 (hi rows, then lo
//    rows) gives both products; the softmax adds them.  Every code is an
//    exact E4M3 value, so nothing is lost on the K side.
//  * Warp 14 loads each item's Q^T (bf16, TMA) as soon as its buffer is free
//    and splits it, an item ahead of the S MMAs.
//  * Warps 9-12 turn every tile's V codes into f16 rows of a swizzled shared-
//    memory stage (thread r = key r; the hardware's E4M3 -> f16 conversion is
//    exact, subnormals included), which the PV MMA reads MN-major.  Rows past
//    the tile's last key become zeros (an unwritten slot may hold a NaN code).
//  * Warp 13 streams each key's K and V scale into a ring of tiles by 4-byte
//    cp.async (page ids fetched three tiles ahead, as the producers do); the
//    ring's barrier completes when the copies land.
//  * Warp 6 issues the S MMAs and O^T += V^T . P^T as in the bf16 kernel.
//  * Warps 0-3 (softmax) multiply each key's scores by its K scale and 2^-e.
//    The weights go to the PV MMA as f16: each times its key's V scale over
//    2^(ev - 127), ev the largest biased exponent of the item's V scales so
//    far, so they stay below 2^9 whatever the scales are (O is rescaled when
//    ev grows, and multiplied back by 2^(ev - 127) at the end); the exp-sums
//    take the unscaled weights.  An item's output is written after the next
//    item's first tile, so the softmax never waits for an item's last PV.
//  * Code size is kept down (the retry loop of the barrier waits and the item
//    store out of line): measured with ncu, a 167 KB build of this kernel
//    spent most of its issue stalls waiting for instructions, its seven roles'
//    loops not fitting the instruction cache together.
//  * Every barrier wait is bounded (pa::mbar_wait_ool); nothing spins forever.
#pragma once

#include "decode_tc.cuh"

namespace pa {

template <int D>
struct DtcF8Cfg {
    static constexpr int KS = D / 128;             // 128-dim chunks of a row
    static constexpr int KCH = D / 64;             // 64-dim sub-chunks of the bf16 Q^T
    static constexpr int BN = 128;                 // keys per tile = MMA M
    static constexpr int NP = 16;                  // MMA N: query heads padded to 16
    static constexpr int CSLOT = BN * 128;         // code stage: 128 keys x 128 codes
    static constexpr int VSLOT = BN * 256;         // bf16 V stage: 128 keys x 128 dims
    static constexpr int VSUB = BN * 128;          // one 64-dim sub-chunk of a V stage
    // stages of each code ring and f16 V stages (at D = 128, 4 + 2 measured
    // 3.4 % faster than 3 + 3 on the GQA decode batch)
    static constexpr int NRC = D >= 256 ? 3 : 4;
    static constexpr int NRV = 2;
    static constexpr int NSC = 3;                  // scale stages (tiles)
    static constexpr int Q_BUF = KCH * NP * 128;   // bf16 Q^T: [KCH][16 rows][128 B]
    // E4M3 Q^T: [KS][hi 16 rows, lo 16 rows][128 B]
    static constexpr int Q8_BUF = KS * 2 * NP * 128;
    static constexpr int P_BUF = 2 * NP * 128;
    static constexpr int OFF_KC = 0;
    static constexpr int OFF_VC = NRC * CSLOT;
    static constexpr int OFF_V = 2 * NRC * CSLOT;
    static constexpr int OFF_Q = OFF_V + NRV * VSLOT;   // two bf16 Q^T buffers
    static constexpr int OFF_Q8 = OFF_Q + 2 * Q_BUF;    // two E4M3 Q^T buffers
    static constexpr int OFF_P = OFF_Q8 + 2 * Q8_BUF;   // two P^T buffers
    static constexpr int OFF_SC = OFF_P + 2 * P_BUF;    // float [NSC][2][128]: K, V scales
    static constexpr int OFF_BAR = OFF_SC + NSC * 2 * BN * 4;
    static constexpr int NBAR = 4 * NRC + 2 * NRV + 2 * NSC + 8 * 2;
    static constexpr int OFF_RED = OFF_BAR + NBAR * 8;   // float [2][4][8] max, [2][4][8] sum
    // float [4] 2^-e of item % 4, then int [2][4] tile maxima of the V-scale exponents
    static constexpr int OFF_QX = OFF_RED + 2 * 2 * 4 * 8 * 4;
    static constexpr int PGR = 4;                  // page-id ring of each streaming warp (tiles)
    static constexpr int OFF_PG = OFF_QX + 64;     // int [5 warps][PGR][16] page ids
    static constexpr int OFF_SROW = OFF_PG + 5 * PGR * 16 * 4;   // int [PGR][16] scale rows
    static constexpr int OFF_PREV = OFF_SROW + PGR * 16 * 4;   // the softmax's pending item
    static constexpr int OFF_MISC = OFF_PREV + 256;
    // 4 softmax warps, 2 K and 2 V producer warps, the MMA warp, 4 converter
    // warps, the scale warp, the query warp
    static constexpr int THREADS = 480;
    static constexpr int OFF_LENS = OFF_MISC + 256;
    static constexpr int SMEM_BYTES = OFF_LENS + (2 * THREADS + 4) * 4 + 1024;
    static constexpr int S_COL = 0;                // two S^T buffers of 2 NP columns (hi, lo)
    static constexpr int O_COL = 4 * NP;           // two O^T accumulators of KS * NP columns
    static constexpr int TMEM_COLS = 128;
    static_assert(O_COL + 2 * KS * NP <= TMEM_COLS, "TMEM columns");
    static_assert(SMEM_BYTES <= 227 * 1024, "shared memory");
    static_assert(OFF_V % 1024 == 0 && OFF_Q % 1024 == 0 && OFF_Q8 % 1024 == 0 &&
                      OFF_P % 1024 == 0 && Q_BUF % 1024 == 0 && Q8_BUF % 1024 == 0,
                  "swizzle atoms");
    static_assert(OFF_MISC % 8 == 0 && 64 + 8 * (THREADS / 32) <= 256, "misc records");
};

// Instruction descriptor of kind::f8f6f4 with E4M3 A and B (both K-major),
// fp32 accumulator.
__host__ __device__ constexpr uint32_t idesc_e4m3_f32(int M, int N) {
    return (1u << 4)                          // accumulator format: f32
           | (0u << 7)                        // A format: E4M3
           | (0u << 10)                       // B format: E4M3
           | ((uint32_t)(N >> 3) << 17)
           | ((uint32_t)(M >> 4) << 24);
}

// D[tmem] (+)= A[smem] * B[smem]^T with E4M3 operands, one CTA, issued by a
// single thread (a K step is 32 codes: 32 bytes of a 128-byte row).
__device__ __forceinline__ void tc_mma_e4m3(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                            uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Arrives on `bar` once every cp.async this thread issued so far has landed
// (the arrival counts towards the barrier's expected count).
__device__ __forceinline__ void cp_async_arrive_noinc(uint32_t bar) {
    asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(bar) : "memory");
}

// x (a float holding a bf16 value, scaled so that |x| < 256) as hi + lo, two
// E4M3 codes: hi the nearest E4M3 of x, lo the nearest of x - hi (exact in
// float).  Returns the codes of two such values packed as (hi0, hi1) and
// (lo0, lo1), the first value in the low byte.
__device__ __forceinline__ void split_e4m3x2(float x0, float x1, uint16_t &hi, uint16_t &lo) {
    hi = __nv_cvt_float2_to_fp8x2(make_float2(x0, x1), __NV_SATFINITE, __NV_E4M3);
    const __half2_raw hr = __nv_cvt_fp8x2_to_halfraw2(hi, __NV_E4M3);
    const float2 hv = __half22float2(*reinterpret_cast<const __half2 *>(&hr));
    lo = __nv_cvt_float2_to_fp8x2(make_float2(x0 - hv.x, x1 - hv.y), __NV_SATFINITE, __NV_E4M3);
}

// Four E4M3 codes (bytes of w, lowest first) as four f16 values, exactly (every
// E4M3 value, subnormals included, is an f16): lo = codes 0, 1 and hi = codes
// 2, 3, the lower code in the low half.
__device__ __forceinline__ void e4m3x4_to_f16(uint32_t w, uint32_t &lo, uint32_t &hi) {
    const __half2_raw l =
        __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)(w & 0xFFFFu), __NV_E4M3);
    const __half2_raw h = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)(w >> 16), __NV_E4M3);
    lo = (uint32_t)l.x | ((uint32_t)l.y << 16);
    hi = (uint32_t)h.x | ((uint32_t)h.y << 16);
}

// Instruction descriptor of kind::f16 with f16 A and B, fp32 accumulator.
__host__ __device__ constexpr uint32_t idesc_f16_f32(int M, int N, int a_mn, int b_mn) {
    return (1u << 4)                          // accumulator format: f32
           | (0u << 7)                        // A format: f16
           | (0u << 10)                       // B format: f16
           | ((uint32_t)a_mn << 15) | ((uint32_t)b_mn << 16)
           | ((uint32_t)(N >> 3) << 17)
           | ((uint32_t)(M >> 4) << 24);
}

// dtc_store_item out of line (once per item; keeps the softmax loop small).
template <int D, int G>
static __device__ __noinline__ void dtc_store_item_ool(const DecodeTcArgs &a, const DtcIter &cur,
                                                       const DtcCut &cut, int t,
                                                       const float (&o)[D / 128][8],
                                                       const float (&L)[G],
                                                       const float (&m_ref)[G]) {
    dtc_store_item<D, G>(a, cur, cut, t, o, L, m_ref);
}

template <int D, int G>
__global__ void __launch_bounds__(480, 1)
    paged_decode_tc_fp8_kernel(const __grid_constant__ CUtensorMap qmap,
                               const __grid_constant__ CUtensorMap kmap,
                               const __grid_constant__ CUtensorMap vmap, const DecodeTcArgs a) {
    using C = DtcF8Cfg<D>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = smem_u32(smem);
    const uint32_t kcring = sbase + C::OFF_KC;
    const uint32_t vcring = sbase + C::OFF_VC;
    const uint32_t vring = sbase + C::OFF_V;
    const uint32_t q_smem = sbase + C::OFF_Q;
    const uint32_t q8_smem = sbase + C::OFF_Q8;
    const uint32_t p_smem = sbase + C::OFF_P;
    const uint32_t sc_smem = sbase + C::OFF_SC;
    // barriers (each waited by its parties in order, never two phases behind)
    const uint32_t bar_kc_full = sbase + C::OFF_BAR;           // [NRC] K codes loaded
    const uint32_t bar_kc_empty = bar_kc_full + 8 * C::NRC;    // [NRC] K codes read by S
    const uint32_t bar_vc_full = bar_kc_empty + 8 * C::NRC;    // [NRC] V codes loaded
    const uint32_t bar_vc_empty = bar_vc_full + 8 * C::NRC;    // [NRC] V codes converted
    const uint32_t bar_v_full = bar_vc_empty + 8 * C::NRC;     // [NRV] bf16 V stage written
    const uint32_t bar_v_empty = bar_v_full + 8 * C::NRV;      // [NRV] V stage read by PV
    const uint32_t bar_sc_full = bar_v_empty + 8 * C::NRV;     // [NSC] scales landed
    const uint32_t bar_sc_empty = bar_sc_full + 8 * C::NSC;    // [NSC] scales read
    const uint32_t bar_q_full = bar_sc_empty + 8 * C::NSC;     // [2] bf16 Q^T loaded
    const uint32_t bar_q8_full = bar_q_full + 16;              // [2] E4M3 Q^T parts written
    const uint32_t bar_q_empty = bar_q8_full + 16;             // [2] last S^T of the item done
    const uint32_t bar_s_full = bar_q_empty + 16;              // [2] S^T in TMEM
    const uint32_t bar_s_free = bar_s_full + 16;               // [2] S^T read
    const uint32_t bar_p_full = bar_s_free + 16;               // [2] P^T written
    const uint32_t bar_o_done = bar_p_full + 16;               // [2] PV that read P buffer b done
    const uint32_t bar_o_full = bar_o_done + 16;               // [2] item's last PV done
    const float *scring = reinterpret_cast<const float *>(smem + C::OFF_SC);   // [NSC][2][128]
    float *red_max = reinterpret_cast<float *>(smem + C::OFF_RED);   // [2][4 warps][8]
    float *red_sum = red_max + 64;                                   // [2][4 warps][8]
    float *q_inv = reinterpret_cast<float *>(smem + C::OFF_QX);      // [4] 2^-e of item % 4
    int *red_ev = reinterpret_cast<int *>(smem + C::OFF_QX + 16);    // [2][4 warps]
    int *pgring = reinterpret_cast<int *>(smem + C::OFF_PG);         // [5][PGR][16] page ids
    int *srow = reinterpret_cast<int *>(smem + C::OFF_SROW);         // [PGR][16] first scale rows
    uint8_t *misc = smem + C::OFF_MISC;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(misc);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(misc + 8);
    int *plan_rk = reinterpret_cast<int *>(misc + 16);
    long long *plan_s = reinterpret_cast<long long *>(misc + 32);
    int *plan_j = reinterpret_cast<int *>(misc + 48);
    long long *scratch = reinterpret_cast<long long *>(misc + 64);   // [THREADS / 32]
    int *lens_cu = reinterpret_cast<int *>(smem + C::OFF_LENS);
    int *lens_sl = lens_cu + C::THREADS + 1;
    // the item whose output the softmax writes after the next item's first tile
    struct PendingItem {
        DtcIter it;
        float m_ref[8], L[8];
        int itn;   // index among items with tiles; -1: the item has none
        int ev;    // the V-scale reference exponent (biased); -1: no key
    };
    static_assert(sizeof(PendingItem) <= 256, "pending item record");
    PendingItem *pend = reinterpret_cast<PendingItem *>(smem + C::OFF_PREV);

    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;
    const int S = a.num_seqs;

    // ---------------------------------------------------------------- setup
    pdl_trigger();
    if (tid == 0) {
        for (int s = 0; s < C::NRC; ++s) {
            mbar_init(bar_kc_full + 8 * s, 2);   // an expect-tx arrival per producer warp
            mbar_init(bar_kc_empty + 8 * s, 1);  // the S MMAs' commit
            mbar_init(bar_vc_full + 8 * s, 2);
            mbar_init(bar_vc_empty + 8 * s, 4);  // one arrival per converter warp
        }
        for (int s = 0; s < C::NRV; ++s) {
            mbar_init(bar_v_full + 8 * s, 4);
            mbar_init(bar_v_empty + 8 * s, 1);
        }
        for (int s = 0; s < C::NSC; ++s) {
            mbar_init(bar_sc_full + 8 * s, 32);  // a cp.async arrival per scale-warp lane
            mbar_init(bar_sc_empty + 8 * s, 4);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(bar_q_full + 8 * b, 1);
            mbar_init(bar_q8_full + 8 * b, 1);
            mbar_init(bar_q_empty + 8 * b, 1);
            mbar_init(bar_s_full + 8 * b, 1);
            mbar_init(bar_s_free + 8 * b, 4);
            mbar_init(bar_p_full + 8 * b, 4);
            mbar_init(bar_o_done + 8 * b, 1);
            mbar_init(bar_o_full + 8 * b, 1);
        }
        fence_barrier_init();
        *abort_flag = 0;
        plan_rk[0] = S;
        plan_rk[1] = 0;
        plan_rk[2] = -1;
        plan_rk[3] = 0;
        plan_s[0] = 0;
        plan_s[1] = INT64_MAX;
        plan_j[0] = 0;
        plan_j[1] = 0;
    }
    if (warp == 6) {
        tmem_alloc(smem_u32(tmem_slot), C::TMEM_COLS);
        tmem_relinquish();
    }
    // rows past the G heads of the Q^T and P^T buffers are never written:
    // zero them once so the padded MMA columns stay finite
    for (int i = tid; i < (2 * C::Q_BUF + 2 * C::Q8_BUF + 2 * C::P_BUF) / 16; i += C::THREADS)
        *reinterpret_cast<uint4 *>(smem + C::OFF_Q + 16 * i) = make_uint4(0, 0, 0, 0);
    fence_proxy_async_smem();
    pdl_wait();   // the previous kernel of the stream may write what this one reads

    const DtcPlanSmem ps = {lens_cu, lens_sl, plan_rk, plan_s, plan_j, scratch};
    dtc_plan_share<C::THREADS>(a, ps);
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
    const int bs = a.block_size;
    const int BR = a.box_rows;

    if (warp == 4 || warp == 5 || warp == 7 || warp == 8 || warp == 13) {
        // ============================================================ streaming warps
        // Warps 4 and 7 stream K codes, warps 5 and 8 V codes: warp ph of a
        // ring takes page runs [0, h0) (ph 0) or [h0, nbox) (ph 1) of every
        // stage, one 128-code box per run and lane.  Warp 13 copies each key's
        // K and V scale.  Lanes fetch the page ids of each tile into a shared
        // ring by 4-byte cp.async three tiles ahead, so no load is waited on.
        const bool is_sc = warp == 13;
        const bool is_k = warp == 4 || warp == 7;
        const int ph = warp >= 7 ? 1 : 0;
        const CUtensorMap *map = is_k ? &kmap : &vmap;
        const uint32_t ring0 = is_k ? kcring : vcring;
        const uint32_t bfull = is_k ? bar_kc_full : bar_vc_full;
        const uint32_t bempty = is_k ? bar_kc_empty : bar_vc_empty;
        int *pgr = pgring + (is_sc ? 4 : (is_k ? 0 : 2) + ph) * C::PGR * 16;
        const uint64_t pol = policy_evict_first();
        if (lane == 0 && !is_sc) prefetch_tensormap(map);
        auto fetch_pages = [&](const DtcIter &x, int jj, int t) {
            if (valid(x)) {
                const int kt = x.k0 + jj * C::BN;
                const int nbox = (min(C::BN, x.k1 - kt) + BR - 1) / BR;
                if (lane < nbox)
                    cp_async4(smem_u32(pgr + (t % C::PGR) * 16 + lane),
                              a.block_tables + (int64_t)x.r * a.max_blocks_per_seq +
                                  (kt + lane * BR) / bs);
            }
            cp_async_commit();
        };
        DtcIter cur = it0, la = it0;
        int j = 0, itn = 0, jl = 0, itl = 0;
        while (valid(cur) && cur.ntiles == 0) dtc_next(a, cur, cut);
        while (valid(la) && la.ntiles == 0) dtc_next(a, la, cut);
        for (int t = 0; t < C::PGR - 1; ++t) {
            fetch_pages(la, jl, t);
            if (valid(la)) adv(la, jl, itl);
        }
        int t = 0, issued = 0;
        if (is_sc) {
            // -------- scales: key i of the tile (lanes take i = lane + 32 m) reads
            // row srow[u] + (i mod BR) of the scale arrays, u = i / BR its page run
            const int hkv = a.num_kv_heads;
            int lbr = 0;
            while ((1 << lbr) < BR) ++lbr;   // BR divides 128: a power of two
            while (valid(cur)) {
                fetch_pages(la, jl, t + C::PGR - 1);
                if (valid(la)) adv(la, jl, itl);
                cp_async_wait<C::PGR - 1>();   // tile t's page ids have landed
                __syncwarp();
                const int kt = cur.k0 + j * C::BN;
                const int cnt = min(C::BN, cur.k1 - kt);
                const int nbox = (cnt + BR - 1) / BR;
                int *sr = srow + (t % C::PGR) * 16;
                if (lane < nbox) {
                    const int pg = pgr[(t % C::PGR) * 16 + lane];
                    sr[lane] = (pg >= 0 && pg < a.num_blocks) ? pg * bs + (kt + lane * BR) % bs
                                                               : -1;
                }
                __syncwarp();
                const int sc = t % C::NSC;
                if (t >= C::NSC)
                    mbar_wait_ool(bar_sc_empty + 8 * sc, ((t / C::NSC) - 1) & 1, a.err, abort_flag);
#pragma unroll
                for (int m = 0; m < C::BN / 32; ++m) {
                    const int i = lane + 32 * m;
                    const int row = i < cnt ? sr[i >> lbr] : -1;
                    if (row >= 0) {
                        const int64_t e = ((int64_t)row + (i & (BR - 1))) * hkv + cur.h;
                        cp_async4(sc_smem + ((sc * 2) * C::BN + i) * 4, a.k_scales + e);
                        cp_async4(sc_smem + ((sc * 2 + 1) * C::BN + i) * 4, a.v_scales + e);
                    }
                }
                cp_async_arrive_noinc(bar_sc_full + 8 * sc);
                ++t;
                adv(cur, j, itn);
            }
            cp_async_wait<0>();
        } else {
            while (valid(cur)) {
                fetch_pages(la, jl, t + C::PGR - 1);
                if (valid(la)) adv(la, jl, itl);
                cp_async_wait<C::PGR - 1>();   // tile t's page ids have landed
                __syncwarp();
                int bad = 0;
                const int kt = cur.k0 + j * C::BN;
                const int nbox = (min(C::BN, cur.k1 - kt) + BR - 1) / BR;
                const int *pgt = pgr + (t % C::PGR) * 16;
                const int h0 = (nbox + 1) >> 1;
                const int u0 = ph ? h0 : 0, u1 = ph ? nbox : h0;
                const int u = u0 + lane;   // lane i issues the box of page run u0 + i
                const int row0 = u < u1 ? pgt[u] * bs + (kt + u * BR) % bs : 0;
                for (int c = 0; c < C::KS; ++c) {   // the tile's 128-dim chunks
                    const int idx = t * C::KS + c;
                    const int slot = idx % C::NRC;
                    if (lane == 0 && !bad) {
                        if (idx >= C::NRC)
                            bad = !mbar_wait_ool(bempty + 8 * slot, ((idx / C::NRC) - 1) & 1, a.err,
                                             abort_flag);
                        if (!bad) mbar_arrive_expect_tx(bfull + 8 * slot, (u1 - u0) * BR * 128);
                    }
                    if (__shfl_sync(0xffffffffu, bad, 0)) break;
                    if (u < u1)
                        tma_load_3d(ring0 + slot * C::CSLOT + u * BR * 128, map, c * 128, cur.h,
                                    row0, bfull + 8 * slot, pol);
                    issued = idx + 1;
                }
                if (__shfl_sync(0xffffffffu, bad, 0)) break;
                ++t;
                adv(cur, j, itn);
            }
            cp_async_wait<0>();
            // copies in flight land before the CTA can exit (bounded)
            if (lane == 0) {
                for (int i = max(0, issued - C::NRC); i < issued; ++i)
                    mbar_drain(bfull + 8 * (i % C::NRC), (i / C::NRC) & 1, kWaitLimitCycles / 8);
            }
        }
    } else if (warp == 14) {
        // ============================================================ query warp
        // Loads each item's Q^T (bf16, by TMA: its G heads) as soon as the
        // buffer is free -- the S MMAs of the item before last are done -- then
        // scales it by 2^e so that its largest |q| lies in [128, 256) and
        // splits it into E4M3 hi + lo.  Lane l takes 8-dim chunks l, l + 32, ...
        DtcIter cur = it0;
        while (valid(cur) && cur.ntiles == 0) dtc_next(a, cur, cut);
        int itn = 0;
        constexpr int NCH = G * D / 8;   // 8-dim chunks of the G rows
        auto chunk_addr = [&](int qb, int ch) {
            const int g = ch / (D / 8), d0 = (ch % (D / 8)) * 8;
            return q_smem + qb * C::Q_BUF + (d0 >> 6) * C::NP * 128 + g * 128 +
                   ((((d0 & 63) >> 3) ^ (g & 7)) << 4);
        };
        const uint64_t pol = policy_evict_first();
        if (lane == 0) prefetch_tensormap(&qmap);
        int q_last = -1;   // the last Q^T load issued
        while (valid(cur)) {
            const int qb = itn & 1;
            if (lane == 0) {
                bool ok = true;
                if (itn >= 2)
                    ok = mbar_wait_ool(bar_q_empty + 8 * qb, ((itn >> 1) - 1) & 1, a.err,
                                       abort_flag);
                if (ok) {
                    mbar_arrive_expect_tx(bar_q_full + 8 * qb, C::KCH * G * 128);
#pragma unroll
                    for (int c = 0; c < C::KCH; ++c)
                        tma_load_3d(q_smem + qb * C::Q_BUF + c * C::NP * 128, &qmap, c * 64,
                                    cur.h * G, (int)cur.row, bar_q_full + 8 * qb, pol);
                    q_last = itn;
                }
            }
            __syncwarp();
            mbar_wait_ool(bar_q_full + 8 * qb, (itn >> 1) & 1, a.err, abort_flag);
            constexpr int PER = (NCH + 31) / 32;
            uint4 qv[PER];   // all loads first: the stores below are ordered after them
#pragma unroll
            for (int m = 0; m < PER; ++m)
                qv[m] = lane + 32 * m < NCH ? lds128(chunk_addr(qb, lane + 32 * m))
                                            : make_uint4(0, 0, 0, 0);
            float amax = 0.f;
#pragma unroll
            for (int m = 0; m < PER; ++m) {
                const uint32_t w[4] = {qv[m].x, qv[m].y, qv[m].z, qv[m].w};
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    amax = fmaxf(amax, fmaxf(fabsf(__uint_as_float(w[e] << 16)),
                                             fabsf(__uint_as_float(w[e] & 0xFFFF0000u))));
            }
            amax = warp_max(amax);
            // 2^e with amax * 2^e in [128, 256): biased exponent 261 - E(amax),
            // kept inside the normal range
            const int E = (__float_as_uint(amax) >> 23) & 255;
            const int fe = min(max(261 - E, 1), 254);
            const float f = __uint_as_float((uint32_t)fe << 23);
            if (lane == 0) q_inv[itn & 3] = 1.f / f;
            const uint32_t q8 = q8_smem + qb * C::Q8_BUF;
#pragma unroll
            for (int m = 0; m < PER; ++m) {
                const int ch = lane + 32 * m;
                if (ch >= NCH) break;
                const int g = ch / (D / 8), d0 = (ch % (D / 8)) * 8;
                const uint32_t w[4] = {qv[m].x, qv[m].y, qv[m].z, qv[m].w};
                uint32_t hi[2], lo[2];
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    uint16_t h0, l0, h1, l1;
                    split_e4m3x2(__uint_as_float(w[2 * e] << 16) * f,
                                 __uint_as_float(w[2 * e] & 0xFFFF0000u) * f, h0, l0);
                    split_e4m3x2(__uint_as_float(w[2 * e + 1] << 16) * f,
                                 __uint_as_float(w[2 * e + 1] & 0xFFFF0000u) * f, h1, l1);
                    hi[e] = (uint32_t)h0 | ((uint32_t)h1 << 16);
                    lo[e] = (uint32_t)l0 | ((uint32_t)l1 << 16);
                }
                // 128-dim chunk c: rows g (hi) and 16 + g (lo) of [32 rows][128 B], swizzled
                const int c = d0 >> 7, dd = d0 & 127;
                const uint32_t off =
                    c * 2 * C::NP * 128 + g * 128 + (((dd >> 4) ^ (g & 7)) << 4) + (dd & 15);
                asm volatile("st.shared.v2.u32 [%0], {%1, %2};" ::"r"(q8 + off), "r"(hi[0]),
                             "r"(hi[1])
                             : "memory");
                asm volatile("st.shared.v2.u32 [%0], {%1, %2};" ::"r"(q8 + C::NP * 128 + off),
                             "r"(lo[0]), "r"(lo[1])
                             : "memory");
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar_q8_full + 8 * qb);
            ++itn;
            do dtc_next(a, cur, cut);
            while (valid(cur) && cur.ntiles == 0);
        }
        // a load in flight lands before the CTA can exit (bounded)
        if (lane == 0 && q_last >= 0)
            mbar_drain(bar_q_full + 8 * (q_last & 1), (q_last >> 1) & 1, kWaitLimitCycles / 8);
    } else if (warp >= 9) {
        // ============================================================ converters
        // Thread r (0..127) converts key r's V row of every tile.
        const int r = tid - 9 * 32;
        DtcIter cur = it0;
        while (valid(cur) && cur.ntiles == 0) dtc_next(a, cur, cut);
        int j = 0, itn = 0, gt = 0;
        while (valid(cur)) {
            // ---- V chunks: codes -> f16 rows of a swizzled shared-memory stage;
            // rows past the tile's last key (any code, NaN included) become zeros
            const bool live = r < min(C::BN, cur.k1 - (cur.k0 + j * C::BN));
            for (int c = 0; c < C::KS; ++c) {
                const int idx = gt * C::KS + c;
                const int cs = idx % C::NRC;
                const int vsl = idx % C::NRV;
                mbar_wait_ool(bar_vc_full + 8 * cs, (idx / C::NRC) & 1, a.err, abort_flag);
                if (idx >= C::NRV)
                    mbar_wait_ool(bar_v_empty + 8 * vsl, ((idx / C::NRV) - 1) & 1, a.err,
                                  abort_flag);
                const uint32_t row = vcring + cs * C::CSLOT + r * 128;
                const uint32_t vdst = vring + vsl * C::VSLOT + r * 128;
                // all eight loads first: the stores below are ordered after them
                uint4 vv[8];
#pragma unroll
                for (int q = 0; q < 8; ++q) vv[q] = lds128(row + ((q ^ (r & 7)) << 4));
#pragma unroll
                for (int q = 0; q < 8; ++q) {   // dims 16q .. 16q + 15: 16-byte chunks 2q, 2q + 1
                    uint4 v = vv[q];
                    if (!live) v = make_uint4(0, 0, 0, 0);
                    uint32_t o[8];
                    e4m3x4_to_f16(v.x, o[0], o[1]);
                    e4m3x4_to_f16(v.y, o[2], o[3]);
                    e4m3x4_to_f16(v.z, o[4], o[5]);
                    e4m3x4_to_f16(v.w, o[6], o[7]);
                    const uint32_t sub = vdst + (q >> 2) * C::VSUB;
                    const int c0 = (2 * q) & 7;
                    sts128(sub + ((c0 ^ (r & 7)) << 4), o[0], o[1], o[2], o[3]);
                    sts128(sub + (((c0 + 1) ^ (r & 7)) << 4), o[4], o[5], o[6], o[7]);
                }
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive(bar_vc_empty + 8 * cs);
                    mbar_arrive(bar_v_full + 8 * vsl);
                }
            }
            ++gt;
            adv(cur, j, itn);
        }
    } else if (warp == 6) {
        // ============================================================ MMA issuer
        if (lane == 0) {
            constexpr uint32_t IDESC_S = idesc_e4m3_f32(128, 2 * C::NP);
            constexpr uint32_t IDESC_O = idesc_f16_f32(128, C::NP, 1, 0);
            auto issue_pv = [&](int g_t, int ob, bool first, bool last) {
                const int pb = g_t & 1;
                mbar_wait_ool(bar_p_full + 8 * pb, (g_t >> 1) & 1, a.err, abort_flag);
#pragma unroll
                for (int c = 0; c < C::KS; ++c) {
                    const int idx = g_t * C::KS + c;
                    mbar_wait_ool(bar_v_full + 8 * (idx % C::NRV), (idx / C::NRV) & 1, a.err,
                              abort_flag);
                }
                tc_fence_after();
                const uint32_t ps_ = p_smem + pb * C::P_BUF;
#pragma unroll
                for (int c = 0; c < C::KS; ++c) {
                    const int idx = g_t * C::KS + c;
                    const uint32_t vs = vring + (idx % C::NRV) * C::VSLOT;
                    const uint32_t od = tmem + C::O_COL + (ob * C::KS + c) * C::NP;
#pragma unroll 1
                    for (int kk = 0; kk < C::BN / 16; ++kk) {
                        const uint64_t ad = smem_desc_sw128(vs + kk * 16 * 128, C::VSUB, 1024);
                        const uint64_t bd = smem_desc_sw128(
                            ps_ + (kk >> 2) * C::NP * 128 + (kk & 3) * 32, 16, 1024);
                        tc_mma_bf16(od, ad, bd, IDESC_O, (!first || kk > 0) ? 1u : 0u);
                    }
                }
                tc_commit(bar_o_done + 8 * pb);
#pragma unroll
                for (int c = 0; c < C::KS; ++c)
                    tc_commit(bar_v_empty + 8 * ((g_t * C::KS + c) % C::NRV));
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
                mbar_wait_ool(bar_q8_full + 8 * qb, (itn >> 1) & 1, a.err, abort_flag);
                const uint32_t q8 = q8_smem + qb * C::Q8_BUF;
                for (int j = 0; j < cur.ntiles; ++j) {
                    const int sb = gt & 1;
                    if (gt >= 2)
                        mbar_wait_ool(bar_s_free + 8 * sb, ((gt >> 1) - 1) & 1, a.err, abort_flag);
#pragma unroll
                    for (int c = 0; c < C::KS; ++c) {
                        const int idx = gt * C::KS + c;
                        mbar_wait_ool(bar_kc_full + 8 * (idx % C::NRC), (idx / C::NRC) & 1, a.err,
                                  abort_flag);
                    }
                    tc_fence_after();
                    // [S_hi | S_lo]^T = K . [Q_hi | Q_lo]^T (N = 32): for each
                    // 128-dim chunk, four 32-code steps
#pragma unroll
                    for (int c = 0; c < C::KS; ++c) {
                        const uint32_t ks = kcring + ((gt * C::KS + c) % C::NRC) * C::CSLOT;
#pragma unroll 1
                        for (int kk = 0; kk < 4; ++kk) {
                            const uint64_t ad = smem_desc_sw128(ks + kk * 32, 16, 1024);
                            const uint64_t bd =
                                smem_desc_sw128(q8 + c * 2 * C::NP * 128 + kk * 32, 16, 1024);
                            tc_mma_e4m3(tmem + C::S_COL + sb * 2 * C::NP, ad, bd, IDESC_S,
                                        (c > 0 || kk > 0) ? 1u : 0u);
                        }
                    }
                    tc_commit(bar_s_full + 8 * sb);
#pragma unroll
                    for (int c = 0; c < C::KS; ++c)
                        tc_commit(bar_kc_empty + 8 * ((gt * C::KS + c) % C::NRC));
                    if (j == cur.ntiles - 1) tc_commit(bar_q_empty + 8 * qb);
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
            if (gt > 0)
                mbar_drain(bar_o_done + 8 * ((gt - 1) & 1), ((gt - 1) >> 1) & 1,
                           kWaitLimitCycles / 8);
        }
    } else {
        // ============================================================ softmax
        const int t = tid;   // key of the tile = TMEM lane
        const uint32_t t_lane = tmem + ((uint32_t)(warp * 32) << 16);
        DtcIter cur = it0;
        int gt = 0, itn = 0, ie = 0;
        // An item's output is written after the next item's first tile, so the
        // softmax never waits for an item's last PV (behind that tile's V
        // conversion) before going on: its accumulator stays untouched until
        // the item after next.  The pending item's record (the same for every
        // softmax thread) is written by thread 0 after a barrier all of them
        // pass once they have read the previous record.
        bool pending = false;
        auto finish_prev = [&]() {
            const int pitn = pend->itn;
            const float vback = pend->ev >= 0 ? ldexpf(1.f, pend->ev - 127) : 1.f;
            float o[C::KS][8], Lp[G], mp[G];
#pragma unroll
            for (int g = 0; g < G; ++g) {
                Lp[g] = pend->L[g];
                mp[g] = pend->m_ref[g];
            }
            if (pitn >= 0) {
                mbar_wait_ool(bar_o_full + 8 * (pitn & 1), (pitn >> 1) & 1, a.err, abort_flag);
                tc_fence_after();
#pragma unroll
                for (int c = 0; c < C::KS; ++c)
                    tmem_ld8(t_lane + C::O_COL + ((pitn & 1) * C::KS + c) * C::NP, o[c]);
                tmem_wait_ld();
                tc_fence_before();
#pragma unroll
                for (int c = 0; c < C::KS; ++c)
#pragma unroll
                    for (int e = 0; e < 8; ++e) o[c][e] *= vback;
            } else {
#pragma unroll
                for (int c = 0; c < C::KS; ++c)
#pragma unroll
                    for (int e = 0; e < 8; ++e) o[c][e] = 0.f;
            }
            dtc_store_item_ool<D, G>(a, pend->it, cut, t, o, Lp, mp);
            pending = false;
        };
        while (valid(cur)) {
            const int ob = itn & 1;
            float m_run[G], m_ref[G], l[G];
#pragma unroll
            for (int g = 0; g < G; ++g) {
                m_run[g] = -INFINITY;
                m_ref[g] = -INFINITY;
                l[g] = 0.f;
            }
            float qsc = 0.f;
            // The softmax weights go to the PV MMA as f16 times the key's V
            // scale over 2^(ev - 127), ev the largest biased exponent of the
            // item's V scales so far: at most 2 * 2^8, so never past f16's
            // range whatever the scales; when ev grows, O is rescaled.
            int ev = -1;
            float vmul = 1.f;
            for (int j = 0; j < cur.ntiles; ++j) {
                const int sb = gt & 1;
                mbar_wait_ool(bar_s_full + 8 * sb, (gt >> 1) & 1, a.err, abort_flag);
                tc_fence_after();
                float sv[8], sl[8];
                tmem_ld8(t_lane + C::S_COL + sb * 2 * C::NP, sv);
                tmem_ld8(t_lane + C::S_COL + sb * 2 * C::NP + C::NP, sl);
                tmem_wait_ld();
#pragma unroll
                for (int g = 0; g < 8; ++g) sv[g] += sl[g];
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar_s_free + 8 * sb);
                // the item's 2^-e, written before its Q parts (whose barrier the
                // S MMAs passed)
                if (j == 0) qsc = a.qscale * q_inv[itn & 3];
                // this key's K and V scales
                const int sc = gt % C::NSC;
                mbar_wait_ool(bar_sc_full + 8 * sc, (gt / C::NSC) & 1, a.err, abort_flag);
                const float kscale = scring[(sc * 2) * C::BN + t];
                const float vscale = scring[(sc * 2 + 1) * C::BN + t];
                __syncwarp();
                if (lane == 0) mbar_arrive(bar_sc_empty + 8 * sc);

                const int kt = cur.k0 + j * C::BN;
                const int cnt = min(C::BN, cur.k1 - kt);
                const bool kv = t < cnt;
                const float ksc = qsc * kscale;
                float x[G];
#pragma unroll
                for (int g = 0; g < G; ++g) x[g] = kv ? sv[g] * ksc : -INFINITY;
                float *rm = red_max + (gt & 1) * 32;
#pragma unroll
                for (int g = 0; g < G; ++g) {
                    const float mx = warp_max(x[g]);
                    if (lane == 0) rm[warp * 8 + g] = mx;
                }
                {
                    const int e = __reduce_max_sync(
                        0xffffffffu, kv ? (int)((__float_as_uint(vscale) >> 23) & 255) : 0);
                    if (lane == 0) red_ev[(gt & 1) * 4 + warp] = e;
                }
                named_barrier_sync(1, 128);
                const int* re = red_ev + (gt & 1) * 4;
                const int ev_new = max(ev, max(max(re[0], re[1]), max(re[2], re[3])));
                const bool ev_up = ev_new > ev;
                float mnew[G];
                bool need[G];
                bool any = ev_up;
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
                        if (need[g])
                            f[g] = m_ref[g] == -INFINITY ? 0.f : ex2_approx(m_ref[g] - mnew[g]);
                    if (j >= 1) {   // O^T holds PVs of this item: rescale after the last one
                        const float fv = (ev_up && ev >= 0) ? ldexpf(1.f, ev - ev_new) : 1.f;
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
                            for (int e = 0; e < 8; ++e) o[e] *= f[e] * fv;
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
                    if (ev_up) {
                        ev = ev_new;
                        vmul = ldexpf(1.f, 127 - ev);
                    }
                }
#pragma unroll
                for (int g = 0; g < G; ++g) m_run[g] = mnew[g];

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
                    *reinterpret_cast<__half *>(
                        prow + g * 128 + ((((kc >> 3) ^ g) & 7) << 4) + (kc & 7) * 2) =
                        __float2half_rn(kv ? pg * (vscale * vmul) : 0.f);
                }
                fence_proxy_async_smem();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar_p_full + 8 * pb);
                ++gt;
                if (pending) finish_prev();
            }

            // ---- end of the item: exp-sums over the 128 keys; the output waits
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
            if (pending) {   // an item without tiles: the previous record is read first
                finish_prev();
                named_barrier_sync(1, 128);
            }
            if (t == 0) {
                pend->it = cur;
#pragma unroll
                for (int g = 0; g < G; ++g) {
                    pend->m_ref[g] = m_ref[g];
                    pend->L[g] = L[g];
                }
                pend->itn = cur.ntiles > 0 ? itn : -1;
                pend->ev = ev;
            }
            pending = true;
            if (cur.ntiles > 0) ++itn;
            ++ie;
            dtc_next(a, cur, cut);
        }
        if (pending) {   // thread 0 wrote the record after the last barrier
            named_barrier_sync(1, 128);
            finish_prev();
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
cudaError_t launch_decode_tc_fp8_t(const CUtensorMap &qmap, const CUtensorMap &kmap,
                                   const CUtensorMap &vmap, const DecodeTcArgs &a, int grid,
                                   cudaStream_t stream) {
    using C = DtcF8Cfg<D>;
    auto kern = paged_decode_tc_fp8_kernel<D, G>;
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
cudaError_t launch_decode_tc_fp8_group(int group, const CUtensorMap &qmap,
                                       const CUtensorMap &kmap, const CUtensorMap &vmap,
                                       const DecodeTcArgs &a, int grid, cudaStream_t stream) {
    switch (group) {
        case 1: return launch_decode_tc_fp8_t<D, 1>(qmap, kmap, vmap, a, grid, stream);
        case 2: return launch_decode_tc_fp8_t<D, 2>(qmap, kmap, vmap, a, grid, stream);
        case 3: return launch_decode_tc_fp8_t<D, 3>(qmap, kmap, vmap, a, grid, stream);
        case 4: return launch_decode_tc_fp8_t<D, 4>(qmap, kmap, vmap, a, grid, stream);
        case 5: return launch_decode_tc_fp8_t<D, 5>(qmap, kmap, vmap, a, grid, stream);
        case 6: return launch_decode_tc_fp8_t<D, 6>(qmap, kmap, vmap, a, grid, stream);
        case 7: return launch_decode_tc_fp8_t<D, 7>(qmap, kmap, vmap, a, grid, stream);
        case 8: return launch_decode_tc_fp8_t<D, 8>(qmap, kmap, vmap, a, grid, stream);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace pa
