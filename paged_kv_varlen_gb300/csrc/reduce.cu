// reduce.cu -- the shared split-KV reduce (kwkr.cn trick 4: partials are a
// log2-space (max, exp-sum) pair plus a normalised partial output; one shared
// reduce kernel merges them, and the GQA decode path reuses it).
//
// One CTA per (request, query head).  The partition maxima and exp-sums are
// read in one pass and the weights w_p = l_p * 2^(m_p - M) kept in shared
// memory; then thread (g, c) combines the 16-byte slice c of the head
// dimension over every PG-th partition starting at g, four loads in flight
// (coalesced reads of the [num_seqs, max_parts, Hq, D] partial outputs), and
// the PG partial sums are added through shared memory.
#include "pa_common.cuh"
#include "pa_internal.h"

namespace pa {

constexpr int kReduceThreads = 128;
static_assert(kMaxDecodeCtas % kReduceThreads == 0, "cut-table rounds");

template <typename T, int D>
__global__ void __launch_bounds__(kReduceThreads) split_reduce_kernel(const ReduceArgs a) {
    extern __shared__ float wsh[];   // [2][max_parts + ncut]: weights, then maxima
    constexpr int LANES = D / 4;                 // float4 slices of one head's row
    constexpr int PG = kReduceThreads / LANES;   // partition groups working in parallel
    __shared__ float red[kReduceThreads / 32];
    __shared__ float Msh, densh;
    __shared__ float4 part[PG > 1 ? PG - 1 : 1][LANES];
    __shared__ int xslot[kMaxDecodeCtas];   // extra partials of this (request, head)
    __shared__ int xcount[kMaxDecodeCtas / 32];   // hits per (round, warp)
    const int r = blockIdx.x;
    const int hq = blockIdx.y;
    const int Hq = a.num_q_heads;
    if (!a.meta_before_wait) pdl_wait();   // (launched early: see launch_reduce_t)
    const int c0 = a.cu_seqlens_q[r];
    if (a.cu_seqlens_q[r + 1] - c0 != 1) {
        if (a.meta_before_wait) pdl_wait();   // complete only after the kernel before it
        return;
    }
    const int N = max(0, a.seq_lens_k[r]);
    const int nparts = min((N + a.partition_size - 1) / a.partition_size, a.max_parts);
    const int tid = threadIdx.x;
    const float sk2 = a.sinks ? a.sinks[hq] * kLog2e : -INFINITY;
    if (a.meta_before_wait) pdl_wait();    // the partials come from the previous kernel
    float *msh = wsh + a.max_parts + a.ncut;
    // parts of items cut between decode CTAs: extra partials [nparts, nparts + nx),
    // listed in cut-table order (ballots and per-warp counts, no atomics), so
    // the partials are always summed in the same order: bit-reproducible
    const int g = a.group > 0 ? hq % a.group : 0;
    constexpr int RND = kMaxDecodeCtas / kReduceThreads;
    constexpr int NW = kReduceThreads / 32;
    const int lane = tid & 31, wid = tid >> 5;
    uint32_t bal[RND];
#pragma unroll
    for (int k = 0; k < RND; ++k) {
        const int b = k * kReduceThreads + tid;
        bool hit = false;
        if (b < a.ncut) {
            const int4 e = a.cut_tab[b];
            hit = e.x == r && e.y == hq / a.group;
        }
        bal[k] = __ballot_sync(0xffffffffu, hit);
        if (lane == 0) xcount[k * NW + wid] = __popc(bal[k]);
    }
    __syncthreads();
    int nx = 0;
#pragma unroll
    for (int k = 0; k < RND; ++k) {
        int before = 0;   // hits at lower cut-table indices
#pragma unroll
        for (int q = 0; q < RND * NW; ++q) before += q < k * NW + wid ? xcount[q] : 0;
        if ((bal[k] >> lane) & 1u)
            xslot[before + __popc(bal[k] & ((1u << lane) - 1u))] = k * kReduceThreads + tid;
    }
#pragma unroll
    for (int q = 0; q < RND * NW; ++q) nx += xcount[q];
    __syncthreads();
    const int ntot = nparts + nx;

    // M = max over partitions of m_p, and over the sink logit (m_p and l_p are
    // read together, one pass)
    float mx = -INFINITY;
    for (int p = tid; p < ntot; p += kReduceThreads) {
        float m, l;
        if (p < nparts) {
            const int64_t slot = ((int64_t)r * a.max_parts + p) * Hq + hq;
            m = a.part_m[slot];
            l = a.part_l[slot];
        } else {
            const int64_t xs = (int64_t)xslot[p - nparts] * a.group + g;
            m = a.xpart_m[xs];
            l = a.xpart_l[xs];
        }
        wsh[p] = l;
        msh[p] = m;
        mx = fmaxf(mx, m);
    }
    mx = warp_max(mx);
    if ((tid & 31) == 0) red[tid >> 5] = mx;
    __syncthreads();
    if (tid == 0) {
        float M = sk2;
        for (int w = 0; w < kReduceThreads / 32; ++w) M = fmaxf(M, red[w]);
        Msh = M;
    }
    __syncthreads();
    const float M = Msh;
    float sum = 0.f;
    for (int p = tid; p < ntot; p += kReduceThreads) {
        const float w = wsh[p] * exp2f(msh[p] - M);
        wsh[p] = w;
        sum += w;
    }
    sum = warp_sum(sum);
    __syncthreads();   // red[] reuse; wsh complete
    if ((tid & 31) == 0) red[tid >> 5] = sum;
    __syncthreads();
    if (tid == 0) {
        float s = 0.f;
        for (int w = 0; w < kReduceThreads / 32; ++w) s += red[w];
        if (a.sinks && nparts > 0) s += exp2f(sk2 - M);
        densh = s;
    }
    __syncthreads();
    const float den = densh;

    // O = sum_p w_p o_p / den: thread (g, c) sums the float4 slice c over the
    // partitions p = g, g + PG, ... (loads issued four at a time), then the PG
    // groups are added through shared memory
    const int c = tid % LANES, pg = tid / LANES;
    const float *po = a.part_o + ((int64_t)r * a.max_parts * Hq + hq) * D + c * 4;
    const int64_t pstride = (int64_t)Hq * D;   // floats between partitions
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
    int p = pg;
    for (; p + 3 * PG < nparts; p += 4 * PG) {
        float4 o[4];
#pragma unroll
        for (int u = 0; u < 4; ++u)
            o[u] = *reinterpret_cast<const float4 *>(po + (int64_t)(p + u * PG) * pstride);
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const float w = wsh[p + u * PG];
            acc[0] = fmaf(w, o[u].x, acc[0]);
            acc[1] = fmaf(w, o[u].y, acc[1]);
            acc[2] = fmaf(w, o[u].z, acc[2]);
            acc[3] = fmaf(w, o[u].w, acc[3]);
        }
    }
    for (; p < ntot; p += PG) {
        const float *src = p < nparts
                               ? po + (int64_t)p * pstride
                               : a.xpart_o + ((int64_t)xslot[p - nparts] * a.group + g) * D + c * 4;
        const float4 o = *reinterpret_cast<const float4 *>(src);
        const float w = wsh[p];
        acc[0] = fmaf(w, o.x, acc[0]);
        acc[1] = fmaf(w, o.y, acc[1]);
        acc[2] = fmaf(w, o.z, acc[2]);
        acc[3] = fmaf(w, o.w, acc[3]);
    }
    if (PG > 1) {
        if (pg > 0) part[pg - 1][c] = make_float4(acc[0], acc[1], acc[2], acc[3]);
        __syncthreads();
        if (pg == 0) {
#pragma unroll
            for (int k = 0; k < PG - 1; ++k) {
                const float4 o = part[k][c];
                acc[0] += o.x;
                acc[1] += o.y;
                acc[2] += o.z;
                acc[3] += o.w;
            }
        }
    }
    if (pg == 0) {
        T *out = reinterpret_cast<T *>(a.out) + ((int64_t)c0 * Hq + hq) * D;
#pragma unroll
        for (int e = 0; e < 4; ++e)
            out[c * 4 + e] = Elem<T>::to_store(nparts > 0 ? acc[e] / den : 0.f);
    }
}

template <typename T, int D>
static cudaError_t launch_reduce_t(const ReduceArgs &a, cudaStream_t stream) {
    const size_t smem = 2 * sizeof(float) * (size_t)((a.max_parts > 0 ? a.max_parts : 1) + a.ncut);
    auto kern = split_reduce_kernel<T, D>;
    if (smem > 48 * 1024) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)smem);
        if (e != cudaSuccess) return e;
    }
    // launched while the kernel writing the partials still runs; each CTA
    // waits for it (pdl_wait) before reading them
    return launch_pdl(kern, dim3(a.num_seqs, a.num_q_heads), dim3(kReduceThreads), smem, stream,
                      a);
}

cudaError_t launch_reduce(int elem_bytes, int head_dim, const ReduceArgs &a, cudaStream_t stream) {
    if (a.num_seqs == 0 || a.num_q_heads == 0) return cudaSuccess;
    if (elem_bytes == 4) {
        switch (head_dim) {
            case 64: return launch_reduce_t<float, 64>(a, stream);
            case 128: return launch_reduce_t<float, 128>(a, stream);
            case 256: return launch_reduce_t<float, 256>(a, stream);
        }
    } else {
        switch (head_dim) {
            case 64: return launch_reduce_t<__nv_bfloat16, 64>(a, stream);
            case 128: return launch_reduce_t<__nv_bfloat16, 128>(a, stream);
            case 256: return launch_reduce_t<__nv_bfloat16, 256>(a, stream);
        }
    }
    return cudaErrorInvalidValue;
}

}  // namespace pa
