// decode_kernel.cuh -- paged attention on CUDA cores for one query row at a
// time, all query heads of one KV head per CTA (GQA grouping).
//
// Pages (kwkr.cn, "What is Paged Attention"): the K/V of request r sit in
// pages block_tables[r][j / block_size]; the GQA decode section serves all
// query heads that share a KV head from one read of its pages; trick 1 folds
// log2(e) into the scale so every exponent is exp2 and keeps the running
// (max, sum) in registers; trick 4 cuts long contexts into 256/512-key
// partitions whose partials go to a shared reduce.
//
// GB300 design
//  * One producer warp streams the CTA's pages with TMA (cp.async.bulk.tensor,
//    a 3-D map over [num_blocks*block_size rows, H_kv, D]) into a ring of
//    shared-memory stages, 128-byte swizzled; page ids are prefetched 32
//    sub-boxes ahead in registers and broadcast with warp shuffles.
//  * NW consumer warps each take whole tiles of TK keys.  QK: each key is
//    owned by LPK lanes that read its row (conflict-free thanks to the
//    swizzle) against the pre-scaled fp32 query heads in shared memory
//    (broadcast reads).  Softmax: one max update per tile, exp2 only.  PV:
//    lanes own 16-byte slices of the value rows and accumulate all G heads.
//  * Warp states are merged in shared memory at the end; the CTA writes
//    either split partials (log2-space max, exp-sum, normalised output) or
//    the final row, with the sink logit applied once.
//  * Every barrier wait is bounded (pa::mbar_wait); nothing spins forever.
#pragma once

#include "pa_common.cuh"
#include "pa_internal.h"

namespace pa {

template <typename T, int D, int G>
struct DecodeCfg {
    static constexpr int E = sizeof(T);
    static constexpr int VEC = Elem<T>::kVec;                 // elements per 16-B chunk
    static constexpr int CPR = D * E / 16;                    // 16-B chunks per K/V row
    static constexpr int EPB = 128 / E;                       // elements per 128-B box row
    static constexpr int NBOX = D / EPB;                      // boxes across one row
    static constexpr int TK = decode_tile_keys(E, D);         // keys per tile
    static constexpr int LPK = 32 / TK;                       // lanes per key (QK)
    static constexpr int CPK = CPR / LPK;                     // chunks per lane (QK)
    // PV reads value rows in pieces of PVB bytes: 16, or 8 for 8-bit codes so
    // that a lane's accumulators cover 8 elements as with bf16
    static constexpr int PVB = E == 1 ? 8 : 16;
    static constexpr int VPV = PVB / E;                       // elements per PV piece
    static constexpr int PPR = D * E / PVB;                   // PV pieces per row
    static constexpr int LPR = PPR < 32 ? PPR : 32;           // lanes per row (PV)
    static constexpr int KPS = 32 / LPR;                      // rows per PV step
    static constexpr int CPL = PPR / LPR;                     // pieces per lane (PV)
    static constexpr int NW = 4;                              // consumer warps
    static constexpr int THREADS = (NW + 1) * 32;
    // CTAs per SM the register budget is sized for: large head groups keep more
    // accumulators live and get a larger share of the register file.
    static constexpr int MIN_CTAS = G <= 5 ? 3 : 2;
    static constexpr int GP = (G + 3) & ~3;                   // padded head count
    static constexpr int TILE_BYTES = TK * D * E;             // K (or V) bytes per tile
    static constexpr int STAGE_BYTES = 2 * TILE_BYTES;
    // Ring depth: NSW stages per consumer warp, tile t -> warp t % NW, stage
    // t % NS.  Stage s then always belongs to warp s % NW and has a single
    // consumer that waits on its phases strictly in order, which the
    // parity-based mbarrier wait requires (a waiter two phases ahead would pass
    // early).  Two stages per warp let a warp compute on one tile while the
    // next is in flight.
    static constexpr int NSW = 1;
    static constexpr int NS = NW * NSW;
    static constexpr int OFF_Q = NS * STAGE_BYTES;
    static constexpr int OFF_P = OFF_Q + G * D * 4;
    static constexpr int OFF_BAR = OFF_P + NW * TK * GP * 8;
    static constexpr int OFF_FLAG = OFF_BAR + 2 * NS * 8;
    static constexpr int SMEM_BYTES = OFF_FLAG + 16 + 1024;  // + alignment slack
    // merge scratch (reuses the stage ring once it has drained)
    static constexpr int MERGE_BYTES = NW * G * (D + 2) * 4;
    static_assert(MERGE_BYTES <= NS * STAGE_BYTES, "merge scratch must fit in the ring");
    static_assert(D % EPB == 0 && CPR % LPK == 0 && PPR % LPR == 0, "shape");
    static_assert(LPK <= 4 && TK >= 8, "lane mapping needs 8..32 keys per tile");
    static_assert(SMEM_BYTES <= 227 * 1024, "shared memory");
};

// T: queries and output (fp32 / bf16); KV: the caches (T, or fp8_e4m3 codes
// with a float32 scale per (slot, KV head) row).
template <typename T, int D, int G, typename KV = T>
__global__ void __launch_bounds__(DecodeCfg<KV, D, G>::THREADS, DecodeCfg<KV, D, G>::MIN_CTAS)
    paged_decode_kernel(const __grid_constant__ CUtensorMap kmap,
                        const __grid_constant__ CUtensorMap vmap, const DecodeArgs a) {
    using C = DecodeCfg<KV, D, G>;
    constexpr bool kScaled = Elem<KV>::kScaled;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    float *qs = reinterpret_cast<float *>(smem + C::OFF_Q);
    float *ps = reinterpret_cast<float *>(smem + C::OFF_P);
    const uint32_t ring = smem_u32(smem);
    const uint32_t bar_full = smem_u32(smem + C::OFF_BAR);
    const uint32_t bar_empty = bar_full + C::NS * 8;
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + C::OFF_FLAG);

    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;
    const int h = blockIdx.y;   // kv head
    const int Hq = a.num_q_heads;
    const int bs = a.block_size;

    // ---------------------------------------------------------------- work item
    int r, part = 0;
    int64_t row;
    int k0, k1;
    bool split = false;
    if (a.mode == 0) {
        r = blockIdx.z;
        const int c0 = a.cu_seqlens_q[r];
        if (a.cu_seqlens_q[r + 1] - c0 != 1) return;   // multi-query request: other kernel
        row = c0;
        int N = a.seq_lens_k[r];
        N = max(0, min(N, a.max_blocks_per_seq * bs));
        part = blockIdx.x;
        if (a.partition_size > 0) {
            split = true;
            k0 = part * a.partition_size;
            if (k0 >= N) return;                       // empty partition: never written
            k1 = min(N, k0 + a.partition_size);
        } else {
            if (part > 0) return;
            k0 = 0;
            k1 = N;
        }
    } else {
        row = blockIdx.x;
        r = request_of_row(a.cu_seqlens_q, a.num_seqs, row);
        const int c0 = a.cu_seqlens_q[r];
        const int n = a.cu_seqlens_q[r + 1] - c0;
        if (n <= 1) return;                            // single-query: decode launch
        const int i = static_cast<int>(row - c0);
        int N = a.seq_lens_k[r];
        N = max(0, min(N, a.max_blocks_per_seq * bs));
        int nvis = a.causal ? min(N, N - n + i + 1) : N;
        k0 = 0;
        k1 = max(0, nvis);
    }
    const int ntiles = (k1 - k0 + C::TK - 1) / C::TK;
    const int BR = a.box_rows;                         // rows per TMA box (divides TK)
    const int SUB = C::TK / BR;                        // boxes (pages) per tile per D-box

    // ---------------------------------------------------------------- setup
    {
        const T *qrow = reinterpret_cast<const T *>(a.q) + (row * Hq + (int64_t)h * G) * D;
        for (int idx = tid; idx < G * D; idx += C::THREADS)
            qs[idx] = Elem<T>::load(qrow + idx) * a.qscale;
    }
    if (tid == 0) {
        for (int s = 0; s < C::NS; ++s) {
            mbar_init(bar_full + 8 * s, 1);
            mbar_init(bar_empty + 8 * s, 1);
        }
        fence_barrier_init();
        *abort_flag = 0;
    }
    __syncthreads();

    if (warp == C::NW) {
        // ============================================================ producer
        if (lane == 0) {
            prefetch_tensormap(&kmap);
            prefetch_tensormap(&vmap);
        }
        const uint64_t pol = policy_evict_first();
        const int32_t *bt = a.block_tables + (int64_t)r * a.max_blocks_per_seq;
        const int nsb_total = (k1 - k0 + BR - 1) / BR;
        auto page_of = [&](int gsb) -> int {
            return (gsb < nsb_total) ? bt[(k0 + gsb * BR) / bs] : 0;
        };
        int base = 0;
        int issued = 0;
        int cur = page_of(lane);
        int nxt = page_of(32 + lane);
        const uint32_t box_bytes = BR * 128;
        for (int t = 0; t < ntiles; ++t) {
            const int s = t % C::NS;
            const int use = t / C::NS;
            int stop = 0;
            if (lane == 0 && use > 0)
                stop = !mbar_wait(bar_empty + 8 * s, (use - 1) & 1, a.err, abort_flag);
            if (__shfl_sync(0xffffffffu, stop, 0)) break;   // aborted: issue nothing more
            __syncwarp();
            const int cnt = min(C::TK, k1 - (k0 + t * C::TK));
            const int nsub = (cnt + BR - 1) / BR;
            if (lane == 0) mbar_arrive_expect_tx(bar_full + 8 * s, nsub * C::NBOX * box_bytes * 2);
            __syncwarp();
            const uint32_t sk = ring + s * C::STAGE_BYTES;
            const uint32_t sv = sk + C::TILE_BYTES;
            for (int u = 0; u < nsub; ++u) {
                const int gsb = t * SUB + u;
                if (gsb >= base + 32) {
                    base += 32;
                    cur = nxt;
                    nxt = page_of(base + 32 + lane);
                }
                const int page = __shfl_sync(0xffffffffu, cur, gsb - base);
                if (lane == 0) {
                    const int key = k0 + gsb * BR;
                    const int row0 = page * bs + key % bs;
#pragma unroll
                    for (int b = 0; b < C::NBOX; ++b) {
                        // stage layout [box b][key][128 B]: key rows of a box stay
                        // consecutive, so consumers address a key without dividing
                        const uint32_t off = (b * C::TK + u * BR) * 128;
                        tma_load_3d(sk + off, &kmap, b * C::EPB, h, row0, bar_full + 8 * s, pol);
                        tma_load_3d(sv + off, &vmap, b * C::EPB, h, row0, bar_full + 8 * s, pol);
                    }
                }
            }
            __syncwarp();
            issued = t + 1;
        }
        // Drain: let this CTA's last copy into each stage land (bounded) before
        // the warp exits; immediate when the consumers have already waited.
        if (lane == 0) {
            for (int t = max(0, issued - C::NS); t < issued; ++t)
                mbar_drain(bar_full + 8 * (t % C::NS), (t / C::NS) & 1, kWaitLimitCycles / 8);
        }
        return;
    }

    // ================================================================ consumers
    // Packed fp32x2 arithmetic: pairs of adjacent elements share one FFMA2.
    constexpr int HV = C::VPV / 2;                     // element pairs per PV piece
    float m[G], l[G];
    float2 acc[G][C::CPL * HV];
#pragma unroll
    for (int g = 0; g < G; ++g) {
        m[g] = -INFINITY;
        l[g] = 0.f;
#pragma unroll
        for (int e = 0; e < C::CPL * HV; ++e) acc[g][e] = make_float2(0.f, 0.f);
    }
    // QK lane mapping: quarter-warps share a half so one wavefront reads 8 rows
    const int qk_key = (lane & 7) + 8 * (lane / (8 * C::LPK));
    const int qk_half = (lane >> 3) % C::LPK;
    const uint32_t qk_row = qk_key * 128;
    const int qk_x = qk_key & 7;
    // PV lane mapping: lane owns chunk pv_lane (+ LPR * ci) of rows pv_sub + KPS*k
    const int pv_sub = lane / C::LPR;
    const int pv_lane = lane % C::LPR;
    float2 *psw = reinterpret_cast<float2 *>(ps) + warp * C::TK * C::GP;   // (p, p) pairs

    for (int t = warp; t < ntiles; t += C::NW) {
        const int s = t % C::NS;
        const int use = t / C::NS;
        mbar_wait(bar_full + 8 * s, use & 1, a.err, abort_flag);
        const int cnt = min(C::TK, k1 - (k0 + t * C::TK));
        const uint32_t sk = ring + s * C::STAGE_BYTES;
        const uint32_t sv = sk + C::TILE_BYTES;
        // quantised cache: the scales of this lane's key row (K) and value row (V)
        float kscale = 1.f, vscale = 1.f;
        if constexpr (kScaled) {
            if (qk_key < cnt) {
                const int key = k0 + t * C::TK + qk_key;
                const int page =
                    __ldg(a.block_tables + (int64_t)r * a.max_blocks_per_seq + key / bs);
                const int64_t sidx = ((int64_t)page * bs + key % bs) * a.num_kv_heads + h;
                kscale = __ldg(a.k_scales + sidx);
                vscale = __ldg(a.v_scales + sidx);
            }
        }

        // ---- scores t_j = <q * scale * log2e, k_j> for this lane's key
        float2 sc2[G];
#pragma unroll
        for (int g = 0; g < G; ++g) sc2[g] = make_float2(0.f, 0.f);
#pragma unroll 4
        for (int i = 0; i < C::CPK; ++i) {
            const int c = qk_half * C::CPK + i;
            const uint32_t addr = sk + (c >> 3) * (C::TK * 128) + qk_row + (((c & 7) ^ qk_x) << 4);
            float kf[C::VEC];
            Elem<KV>::unpack(lds128(addr), kf);
#pragma unroll
            for (int g = 0; g < G; ++g) {
                const float4 *qv = reinterpret_cast<const float4 *>(qs + g * D + c * C::VEC);
#pragma unroll
                for (int v4 = 0; v4 < C::VEC / 4; ++v4) {
                    const float4 qq = qv[v4];
                    sc2[g] = __ffma2_rn(make_float2(qq.x, qq.y),
                                        make_float2(kf[4 * v4 + 0], kf[4 * v4 + 1]), sc2[g]);
                    sc2[g] = __ffma2_rn(make_float2(qq.z, qq.w),
                                        make_float2(kf[4 * v4 + 2], kf[4 * v4 + 3]), sc2[g]);
                }
            }
        }
        float sc[G];
#pragma unroll
        for (int g = 0; g < G; ++g) {
            sc[g] = sc2[g].x + sc2[g].y;
            if (C::LPK > 1) sc[g] += __shfl_xor_sync(0xffffffffu, sc[g], 8);
            if (C::LPK > 2) sc[g] += __shfl_xor_sync(0xffffffffu, sc[g], 16);
            if constexpr (kScaled) sc[g] *= kscale;   // <q, code_j> * scale_j
        }
        const bool valid = qk_key < cnt;
        // ---- one online-softmax update per tile (log2 domain)
        float corr[G];
#pragma unroll
        for (int g = 0; g < G; ++g) {
            const float sg = valid ? sc[g] : -INFINITY;
            const float mnew = fmaxf(m[g], warp_max(sg));
            const bool none = (mnew == -INFINITY);
            corr[g] = none ? 1.f : exp2f(m[g] - mnew);
            const float pg = none ? 0.f : exp2f(sg - mnew);
            l[g] = l[g] * corr[g] + (qk_half == 0 ? pg : 0.f);
            m[g] = mnew;
            // the PV weight carries the value row's scale (l counts p alone)
            const float pw = kScaled ? pg * vscale : pg;
            if (qk_half == 0) psw[qk_key * C::GP + g] = make_float2(pw, pw);
        }
#pragma unroll
        for (int g = 0; g < G; ++g) {
            const float2 cc = make_float2(corr[g], corr[g]);
#pragma unroll
            for (int e = 0; e < C::CPL * HV; ++e) acc[g][e] = __fmul2_rn(acc[g][e], cc);
        }
        __syncwarp();

        // ---- acc += p_j * v_j over the valid keys of the tile
        auto pv_row = [&](int j) {
            float2 pj[C::GP];
#pragma unroll
            for (int g2 = 0; g2 < C::GP / 2; ++g2) {
                const float4 pv = reinterpret_cast<const float4 *>(psw + j * C::GP)[g2];
                pj[2 * g2 + 0] = make_float2(pv.x, pv.y);
                pj[2 * g2 + 1] = make_float2(pv.z, pv.w);
            }
            const uint32_t row = sv + j * 128;
            const int jx = j & 7;
#pragma unroll
            for (int ci = 0; ci < C::CPL; ++ci) {
                const int pc = pv_lane + ci * C::LPR;   // PV piece of the row
                const int c = pc * C::PVB / 16;         // its 16-byte chunk
                const uint32_t addr = row + (c >> 3) * (C::TK * 128) + (((c & 7) ^ jx) << 4);
                float vf[C::VPV];
                if constexpr (C::PVB == 16)
                    Elem<KV>::unpack(lds128(addr), vf);
                else
                    Elem<KV>::unpack8(lds64(addr + (pc & 1) * 8), vf);
#pragma unroll
                for (int g = 0; g < G; ++g)
#pragma unroll
                    for (int e = 0; e < HV; ++e)
                        acc[g][ci * HV + e] = __ffma2_rn(
                            pj[g], make_float2(vf[2 * e], vf[2 * e + 1]), acc[g][ci * HV + e]);
            }
        };
        if (cnt == C::TK) {
#pragma unroll
            for (int jj = 0; jj < C::TK / C::KPS; ++jj) pv_row(jj * C::KPS + pv_sub);
        } else {
            for (int j = pv_sub; j < cnt; j += C::KPS) pv_row(j);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(bar_empty + 8 * s);
    }

    // ---------------------------------------------------------------- merge
    // PV sub-groups of a warp share m: sum their accumulators.
#pragma unroll
    for (int o = C::LPR; o < 32; o <<= 1)
#pragma unroll
        for (int g = 0; g < G; ++g)
#pragma unroll
            for (int e = 0; e < C::CPL * HV; ++e) {
                acc[g][e].x += __shfl_xor_sync(0xffffffffu, acc[g][e].x, o);
                acc[g][e].y += __shfl_xor_sync(0xffffffffu, acc[g][e].y, o);
            }
#pragma unroll
    for (int g = 0; g < G; ++g) l[g] = warp_sum(l[g]);

    named_barrier_sync(1, C::NW * 32);   // every consumer is done with the ring
    float *ms = reinterpret_cast<float *>(smem);      // [NW][G]
    float *ls = ms + C::NW * G;                        // [NW][G]
    float *os = ls + C::NW * G;                        // [NW][G][D]
    if (lane == 0) {
#pragma unroll
        for (int g = 0; g < G; ++g) {
            ms[warp * G + g] = m[g];
            ls[warp * G + g] = l[g];
        }
    }
    if (pv_sub == 0) {
#pragma unroll
        for (int g = 0; g < G; ++g)
#pragma unroll
            for (int ci = 0; ci < C::CPL; ++ci)
#pragma unroll
                for (int e = 0; e < HV; ++e) {
                    float *o = os + (warp * G + g) * D + (pv_lane + ci * C::LPR) * C::VPV + 2 * e;
                    o[0] = acc[g][ci * HV + e].x;
                    o[1] = acc[g][ci * HV + e].y;
                }
    }
    named_barrier_sync(1, C::NW * 32);

    for (int idx = tid; idx < G * D; idx += C::NW * 32) {
        const int g = idx / D, d = idx % D;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < C::NW; ++w) M = fmaxf(M, ms[w * G + g]);
        float L = 0.f, O = 0.f;
        if (M != -INFINITY) {
#pragma unroll
            for (int w = 0; w < C::NW; ++w) {
                const float f = exp2f(ms[w * G + g] - M);   // 0 for an idle warp (-inf)
                L += ls[w * G + g] * f;
                O += os[(w * G + g) * D + d] * f;
            }
        }
        const int hq = h * G + g;
        if (split) {
            const int64_t slot = ((int64_t)r * a.max_parts + part) * Hq + hq;
            a.part_o[slot * D + d] = L > 0.f ? O / L : 0.f;
            if (d == 0) {
                a.part_m[slot] = M;
                a.part_l[slot] = L;
            }
        } else {
            float res = 0.f;
            if (L > 0.f) {
                if (a.sinks) {
                    const float sk2 = a.sinks[hq] * kLog2e;
                    const float M2 = fmaxf(M, sk2);
                    const float f = exp2f(M - M2);
                    res = (O * f) / (L * f + exp2f(sk2 - M2));
                } else {
                    res = O / L;
                }
            }
            reinterpret_cast<T *>(a.out)[(row * Hq + hq) * D + d] = Elem<T>::to_store(res);
        }
    }
}

template <typename T, int D, int G, typename KV = T>
cudaError_t launch_decode_t(const CUtensorMap &kmap, const CUtensorMap &vmap, const DecodeArgs &a,
                            dim3 grid, cudaStream_t stream) {
    using C = DecodeCfg<KV, D, G>;
    auto kern = paged_decode_kernel<T, D, G, KV>;
    static bool configured = false;   // benign race: idempotent attribute set
    if (!configured) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             C::SMEM_BYTES);
        if (e != cudaSuccess) return e;
        configured = true;
    }
    kern<<<grid, C::THREADS, C::SMEM_BYTES, stream>>>(kmap, vmap, a);
    return cudaGetLastError();
}

template <typename T, int D, typename KV = T>
cudaError_t launch_decode_group(int group, const CUtensorMap &kmap, const CUtensorMap &vmap,
                                const DecodeArgs &a, dim3 grid, cudaStream_t stream) {
    switch (group) {
        case 1: return launch_decode_t<T, D, 1, KV>(kmap, vmap, a, grid, stream);
        case 2: return launch_decode_t<T, D, 2, KV>(kmap, vmap, a, grid, stream);
        case 3: return launch_decode_t<T, D, 3, KV>(kmap, vmap, a, grid, stream);
        case 4: return launch_decode_t<T, D, 4, KV>(kmap, vmap, a, grid, stream);
        case 5: return launch_decode_t<T, D, 5, KV>(kmap, vmap, a, grid, stream);
        case 6: return launch_decode_t<T, D, 6, KV>(kmap, vmap, a, grid, stream);
        case 7: return launch_decode_t<T, D, 7, KV>(kmap, vmap, a, grid, stream);
        case 8: return launch_decode_t<T, D, 8, KV>(kmap, vmap, a, grid, stream);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace pa
