// prefill_plan.cu -- the claim order of the multi-query kernel's work units.
//
// The multi-query kernel (prefill_tc.cuh) is persistent: its CTAs claim work
// units -- (request, query block, KV head) -- from a counter in the
// workspace.  Units differ in weight by the number of key tiles they read
// (a long prompt's last block reads every key, a verify window a whole
// context), so they are claimed heaviest request first: this kernel counting-
// sorts the requests with two or more query rows by their key tiles
// (descending) and writes, for the k-th request of that order, the number of
// units before it.  A claim c then belongs to the request k with
// P[k] <= c < P[k + 1]; inside a request the heaviest query block comes
// first, all KV heads of a block together.  One CTA, launched before the
// multi-query kernel, which overlaps its setup with it (programmatic
// dependent launch).
#include "pa_common.cuh"
#include "pa_internal.h"

namespace pa {

constexpr int kPlanThreads = 1024;
constexpr int kPlanBuckets = 4096;

// Inclusive scan over the CTA; *total = the CTA's sum (ends with a barrier).
__device__ __forceinline__ int plan_block_scan(int v, int *tmp, int *total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) tmp[warp] = x;
    __syncthreads();
    int before = 0, tot = 0;
#pragma unroll
    for (int w = 0; w < kPlanThreads / 32; ++w) {
        const int t = tmp[w];
        if (w < warp) before += t;
        tot += t;
    }
    __syncthreads();
    *total = tot;
    return x + before;
}

__global__ void __launch_bounds__(kPlanThreads, 1) mq_plan_kernel(const MqPlanArgs a) {
    pdl_trigger();   // the multi-query kernel may start its setup meanwhile
    __shared__ int hist[kPlanBuckets];   // requests per bucket, then next free position
    __shared__ int tmp[kPlanThreads / 32];
    const int tid = threadIdx.x;
    const int S = a.num_seqs;
    int *hdr = a.plan;                    // [0] claim counter, [1] requests, [2] units
    int *order = hdr + kPlanHeader;       // [S]
    int *P = order + S;                   // [S + 1]
    auto bucket_of = [&](int r, int *units) -> int {
        const int c0 = a.cu_seqlens_q[r];
        const int n = a.cu_seqlens_q[r + 1] - c0;
        if (n < 2) return -1;             // decode rows: the decode kernel's
        const int N = max(0, min(a.seq_lens_k[r], a.max_keys));
        *units = ((n + a.block_rows - 1) / a.block_rows) * a.num_kv_heads;
        // heaviest first: bucket 0 holds the most key tiles
        return kPlanBuckets - 1 - min((N + a.tile_keys - 1) / a.tile_keys, kPlanBuckets - 1);
    };
    for (int i = tid; i < kPlanBuckets; i += kPlanThreads) hist[i] = 0;
    __syncthreads();
    for (int r = tid; r < S; r += kPlanThreads) {
        int u;
        const int b = bucket_of(r, &u);
        if (b >= 0) atomicAdd(&hist[b], 1);
    }
    __syncthreads();
    // exclusive scan of the histogram, four buckets per thread
    constexpr int PER = kPlanBuckets / kPlanThreads;
    int loc[PER], sum = 0;
#pragma unroll
    for (int q = 0; q < PER; ++q) {
        loc[q] = hist[tid * PER + q];
        sum += loc[q];
    }
    int count;
    const int incl = plan_block_scan(sum, tmp, &count);
    int run = incl - sum;
#pragma unroll
    for (int q = 0; q < PER; ++q) {
        hist[tid * PER + q] = run;
        run += loc[q];
    }
    __syncthreads();
    // requests into their positions (the order inside a bucket does not
    // matter: every unit's result is independent of which CTA computes it)
    for (int r = tid; r < S; r += kPlanThreads) {
        int u;
        const int b = bucket_of(r, &u);
        if (b >= 0) order[atomicAdd(&hist[b], 1)] = r;
    }
    __syncthreads();   // (global writes of this CTA are visible to it after the barrier)
    // units before each request of the order
    int carry = 0;
    for (int base = 0; base < count; base += kPlanThreads) {
        const int k = base + tid;
        int u = 0;
        if (k < count) bucket_of(order[k], &u);
        int tot;
        const int inc = plan_block_scan(u, tmp, &tot);
        if (k < count) P[k] = carry + inc - u;
        carry += tot;
    }
    if (tid == 0) {
        P[count] = carry;
        hdr[0] = 0;
        hdr[1] = count;
        hdr[2] = carry;
    }
}

cudaError_t launch_mq_plan(const MqPlanArgs &a, cudaStream_t stream) {
    mq_plan_kernel<<<1, kPlanThreads, 0, stream>>>(a);
    return cudaGetLastError();
}

}  // namespace pa
