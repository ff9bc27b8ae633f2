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

namespace pa {

// ---------------------------------------------------------------- quantised cache
// reshape_and_cache into the quantised KV cache (TurboQuant helpers, lqnn.cn
// section 5; the format is this library's reading: 8-bit E4M3 codes and one
// float32 scale per (token, KV head) row):
//   amax = max_d |x_d|, inv = 448 / amax, code_d = E4M3(x_d * inv) (round to
//   nearest even, saturating), scale = amax / 448; a row of zeros gets codes 0
//   and scale 0.
// One warp per (token, KV head); each lane converts D / 32 elements of the K
// row, then of the V row.  Negative slots and slots past the pool are skipped.
constexpr int kQuantWarps = 8;

template <typename T, int D>
__global__ void __launch_bounds__(kQuantWarps * 32)
    quantize_kv_fp8_kernel(const T *__restrict__ key, const T *__restrict__ value, int64_t stride,
                           uint8_t *__restrict__ kc, uint8_t *__restrict__ vc,
                           float *__restrict__ ks, float *__restrict__ vs,
                           const int64_t *__restrict__ slots, int64_t num_tokens, int num_kv_heads,
                           int64_t num_slots) {
    constexpr int PER = D / 32;   // elements per lane
    const int64_t pair = (int64_t)blockIdx.x * kQuantWarps + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    const int64_t t = pair / num_kv_heads;
    const int h = (int)(pair % num_kv_heads);
    if (t >= num_tokens) return;
    const int64_t slot = slots[t];
    if (slot < 0 || slot >= num_slots) return;   // padding token / outside the pool
    const int64_t row = slot * num_kv_heads + h;
#pragma unroll
    for (int which = 0; which < 2; ++which) {
        const T *src = (which ? value : key) + t * stride + (int64_t)h * D + lane * PER;
        float x[PER];
        float amax = 0.f;
#pragma unroll
        for (int i = 0; i < PER; ++i) {
            x[i] = Elem<T>::load(src + i);
            amax = fmaxf(amax, fabsf(x[i]));
        }
        amax = warp_max(amax);
        uint8_t code[PER];
        if (amax == 0.f) {
#pragma unroll
            for (int i = 0; i < PER; ++i) code[i] = 0;
        } else {
            const float inv = __fdiv_rn(448.f, amax);
#pragma unroll
            for (int i = 0; i < PER; ++i)
                code[i] = __nv_cvt_float_to_fp8(__fmul_rn(x[i], inv), __NV_SATFINITE, __NV_E4M3);
        }
        uint8_t *dst = (which ? vc : kc) + row * D + lane * PER;
        if constexpr (PER == 4) {
            *reinterpret_cast<uint32_t *>(dst) = (uint32_t)code[0] | ((uint32_t)code[1] << 8) |
                                                 ((uint32_t)code[2] << 16) |
                                                 ((uint32_t)code[3] << 24);
        } else {
#pragma unroll
            for (int i = 0; i < PER; i += 4)
                *reinterpret_cast<uint32_t *>(dst + i) =
                    (uint32_t)code[i] | ((uint32_t)code[i + 1] << 8) |
                    ((uint32_t)code[i + 2] << 16) | ((uint32_t)code[i + 3] << 24);
        }
        if (lane == 0) (which ? vs : ks)[row] = amax == 0.f ? 0.f : __fdiv_rn(amax, 448.f);
    }
}

template <typename T>
static cudaError_t launch_quantize_t(const void *key, const void *value, int64_t stride,
                                     uint8_t *kc, uint8_t *vc, float *ks, float *vs,
                                     const int64_t *slots, int64_t num_tokens, int num_kv_heads,
                                     int head_dim, int64_t num_slots, cudaStream_t stream) {
    const int64_t pairs = num_tokens * num_kv_heads;
    const dim3 grid((unsigned)((pairs + kQuantWarps - 1) / kQuantWarps));
    const dim3 block(kQuantWarps * 32);
    auto k = reinterpret_cast<const T *>(key);
    auto v = reinterpret_cast<const T *>(value);
    if (head_dim == 128)
        quantize_kv_fp8_kernel<T, 128><<<grid, block, 0, stream>>>(
            k, v, stride, kc, vc, ks, vs, slots, num_tokens, num_kv_heads, num_slots);
    else
        quantize_kv_fp8_kernel<T, 256><<<grid, block, 0, stream>>>(
            k, v, stride, kc, vc, ks, vs, slots, num_tokens, num_kv_heads, num_slots);
    return cudaGetLastError();
}

cudaError_t launch_quantize_kv_fp8(const void *key, const void *value, int64_t stride,
                                   int elem_bytes, uint8_t *key_codes, uint8_t *value_codes,
                                   float *key_scales, float *value_scales, const int64_t *slots,
                                   int64_t num_tokens, int num_kv_heads, int head_dim,
                                   int64_t num_slots, cudaStream_t stream) {
    if (num_tokens == 0) return cudaSuccess;
    if (elem_bytes == 4)
        return launch_quantize_t<float>(key, value, stride, key_codes, value_codes, key_scales,
                                        value_scales, slots, num_tokens, num_kv_heads, head_dim,
                                        num_slots, stream);
    return launch_quantize_t<__nv_bfloat16>(key, value, stride, key_codes, value_codes,
                                            key_scales, value_scales, slots, num_tokens,
                                            num_kv_heads, head_dim, num_slots, stream);
}

}  // namespace pa
