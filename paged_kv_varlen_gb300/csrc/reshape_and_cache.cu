// reshape_and_cache.cu -- scatter this step's K/V rows into the page pool
// (kwkr.cn kernel table: reshape_and_cache writes projected K/V into the
// paged cache).
//
// A token's row [H_kv, D] is contiguous both in the source and at its slot
// (the pool is [num_blocks, block_size, H_kv, D], so slot s starts at
// s * H_kv * D elements).  One warp copies one token's K and V rows with
// 16-byte loads and stores when every address allows it, else with 4- or
// 2-byte words.  The copy is a plain bit copy.
#include "pa_common.cuh"
#include "pa_internal.h"

namespace pa {

constexpr int kScatterWarps = 8;

template <typename W>
__global__ void __launch_bounds__(kScatterWarps * 32)
    scatter_rows_kernel(const uint8_t *__restrict__ key, const uint8_t *__restrict__ value,
                        int64_t stride_bytes, uint8_t *__restrict__ kc, uint8_t *__restrict__ vc,
                        const int64_t *__restrict__ slots, int64_t num_tokens, int64_t row_bytes,
                        int64_t num_slots) {
    pdl_trigger();   // the attention kernel may start its setup meanwhile
    const int64_t t = (int64_t)blockIdx.x * kScatterWarps + (threadIdx.x >> 5);
    if (t >= num_tokens) return;
    const int lane = threadIdx.x & 31;
    const int64_t slot = slots[t];
    if (slot < 0 || slot >= num_slots) return;   // padding token / outside the pool
    const int64_t nw = row_bytes / (int64_t)sizeof(W);
    const W *ks = reinterpret_cast<const W *>(key + t * stride_bytes);
    const W *vs = reinterpret_cast<const W *>(value + t * stride_bytes);
    W *kd = reinterpret_cast<W *>(kc + slot * row_bytes);
    W *vd = reinterpret_cast<W *>(vc + slot * row_bytes);
    for (int64_t i = lane; i < nw; i += 32) {
        const W kv = __ldg(ks + i);
        const W vv = __ldg(vs + i);
        kd[i] = kv;
        vd[i] = vv;
    }
}

cudaError_t launch_reshape_and_cache(const void *key, const void *value, int64_t stride_bytes,
                                     void *key_cache, void *value_cache, const int64_t *slots,
                                     int64_t num_tokens, int64_t row_bytes, int64_t num_slots,
                                     cudaStream_t stream) {
    if (num_tokens == 0) return cudaSuccess;
    const uintptr_t align = reinterpret_cast<uintptr_t>(key) | reinterpret_cast<uintptr_t>(value) |
                            reinterpret_cast<uintptr_t>(key_cache) |
                            reinterpret_cast<uintptr_t>(value_cache) | (uintptr_t)stride_bytes |
                            (uintptr_t)row_bytes;
    const dim3 grid((unsigned)((num_tokens + kScatterWarps - 1) / kScatterWarps));
    const dim3 block(kScatterWarps * 32);
    auto k8 = reinterpret_cast<const uint8_t *>(key);
    auto v8 = reinterpret_cast<const uint8_t *>(value);
    auto kc = reinterpret_cast<uint8_t *>(key_cache);
    auto vc = reinterpret_cast<uint8_t *>(value_cache);
    if ((align & 15) == 0)
        scatter_rows_kernel<uint4><<<grid, block, 0, stream>>>(k8, v8, stride_bytes, kc, vc, slots,
                                                               num_tokens, row_bytes, num_slots);
    else if ((align & 3) == 0)
        scatter_rows_kernel<uint32_t><<<grid, block, 0, stream>>>(
            k8, v8, stride_bytes, kc, vc, slots, num_tokens, row_bytes, num_slots);
    else
        scatter_rows_kernel<uint16_t><<<grid, block, 0, stream>>>(
            k8, v8, stride_bytes, kc, vc, slots, num_tokens, row_bytes, num_slots);
    return cudaGetLastError();
}

}  // namespace pa
