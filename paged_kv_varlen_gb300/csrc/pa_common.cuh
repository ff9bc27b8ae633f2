// pa_common.cuh -- device helpers shared by the sm_103a kernels: mbarrier and
// TMA (cp.async.bulk.tensor) wrappers written as inline PTX, bounded waits,
// bf16 unpacking.  Every wait on an mbarrier gives up after a fixed number of
// cycles and reports it through the library's device error word instead of
// spinning forever.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace pa {

// About one second at 2 GHz: far beyond any legitimate pipeline stall.
constexpr long long kWaitLimitCycles = 2000000000LL;

// Kernels report an abandoned bounded wait through the library's device error
// word (passed by pointer; read and cleared by pa_device_error()).
__device__ __forceinline__ void report_error(int *err, int code) {
    if (err) atomicExch(err, code);
}

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ---------------------------------------------------------------- mbarrier
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_barrier_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// Waits for the phase with the given parity to complete.  Bounded: after
// kWaitLimitCycles it reports error 1 through the device error word, raises
// the CTA's abort flag and returns false.  Once the flag is up (this CTA) or
// the error word is set (any CTA), waits return false at once, so a broken
// pipeline ends quickly instead of timing out wait after wait.  Callers carry
// on after a false return so every barrier still gets its arrivals.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, int *err,
                                          volatile int *abort_flag) {
    if (mbar_try_wait(bar, parity)) return true;
    if (*abort_flag) return false;
    const long long t0 = clock64();
    for (uint32_t it = 1;; ++it) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((it & 1023) == 0) {
            if (*abort_flag || (err && *reinterpret_cast<volatile int *>(err))) {
                *abort_flag = 1;
                return false;
            }
            if (clock64() - t0 > kWaitLimitCycles) {
                report_error(err, 1);
                *abort_flag = 1;
                return false;
            }
        }
    }
}

// mbar_wait with the retry loop out of line (one shared copy per kernel), for
// kernels whose many wait sites would otherwise each carry a copy of it.
static __device__ __noinline__ bool mbar_wait_slow(uint32_t bar, uint32_t parity, int *err,
                                                  volatile int *abort_flag) {
    return mbar_wait(bar, parity, err, abort_flag);
}
__device__ __forceinline__ bool mbar_wait_ool(uint32_t bar, uint32_t parity, int *err,
                                              volatile int *abort_flag) {
    if (mbar_try_wait(bar, parity)) return true;
    return mbar_wait_slow(bar, parity, err, abort_flag);
}

// Bounded wait that ignores the abort flag (used to drain copies in flight
// before a CTA exits); gives up silently after `limit` cycles.
__device__ __forceinline__ void mbar_drain(uint32_t bar, uint32_t parity, long long limit) {
    const long long t0 = clock64();
    while (!mbar_try_wait(bar, parity))
        if (clock64() - t0 > limit) return;
}

// ---------------------------------------------------------------- dependent launch
// Programmatic dependent launch: a kernel launched with programmatic stream
// serialization may start while the kernel before it in the stream runs;
// pdl_wait() blocks the calling thread until that kernel has completed and
// its memory writes are visible (at once when there is none, or when it was
// launched without the attribute).  pdl_trigger() lets the next kernel start.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ---------------------------------------------------------------- cp.async
// 4-byte asynchronous global -> shared copy (through L1).
__device__ __forceinline__ void cp_async4(uint32_t dst, const void *src) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
    asm volatile("cp.async.commit_group;" ::: "memory");
}
// Waits until at most N of this thread's committed groups are still in flight.
template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// ---------------------------------------------------------------- TMA
__device__ __forceinline__ uint64_t policy_evict_first() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

__device__ __forceinline__ uint64_t policy_evict_last() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

// Brings the 128-byte line holding `p` into L2 (no register result).
__device__ __forceinline__ void prefetch_l2(const void *p) {
    asm volatile("prefetch.global.L2 [%0];" ::"l"(reinterpret_cast<uint64_t>(p)) : "memory");
}

__device__ __forceinline__ void prefetch_tensormap(const void *map) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// 3-D tiled TMA load of one box into shared memory, completing on `bar`.
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const void *map, int x, int y, int z,
                                            uint32_t bar, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        ".L2::cache_hint [%0], [%1, {%2, %3, %4}], [%5], %6;" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(bar), "l"(policy)
        : "memory");
}

// ---------------------------------------------------------------- smem access
__device__ __forceinline__ uint4 lds128(uint32_t addr) {
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "r"(addr));
    return v;
}

__device__ __forceinline__ uint2 lds64(uint32_t addr) {
    uint2 v;
    asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(addr));
    return v;
}

__device__ __forceinline__ void named_barrier_sync(int id, int nthreads) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// ---------------------------------------------------------------- element types
// A 16-byte chunk of K/V holds 8 bf16 or 4 float values; unpack to float.
template <typename T> struct Elem;

template <> struct Elem<float> {
    static constexpr int kVec = 4;
    static constexpr bool kScaled = false;
    static __device__ __forceinline__ void unpack(const uint4 &u, float *f) {
        f[0] = __uint_as_float(u.x);
        f[1] = __uint_as_float(u.y);
        f[2] = __uint_as_float(u.z);
        f[3] = __uint_as_float(u.w);
    }
    static __device__ __forceinline__ float load(const float *p) { return *p; }
    static __device__ __forceinline__ float to_store(float x) { return x; }
};

template <> struct Elem<__nv_bfloat16> {
    static constexpr int kVec = 8;
    static constexpr bool kScaled = false;
    // A bf16 value is the upper half of the float32 with the same bits.
    static __device__ __forceinline__ void unpack(const uint4 &u, float *f) {
        f[0] = __uint_as_float(u.x << 16);
        f[1] = __uint_as_float(u.x & 0xffff0000u);
        f[2] = __uint_as_float(u.y << 16);
        f[3] = __uint_as_float(u.y & 0xffff0000u);
        f[4] = __uint_as_float(u.z << 16);
        f[5] = __uint_as_float(u.z & 0xffff0000u);
        f[6] = __uint_as_float(u.w << 16);
        f[7] = __uint_as_float(u.w & 0xffff0000u);
    }
    static __device__ __forceinline__ float load(const __nv_bfloat16 *p) {
        return __bfloat162float(*p);
    }
    static __device__ __forceinline__ __nv_bfloat16 to_store(float x) {
        return __float2bfloat16_rn(x);
    }
};

// An 8-bit float of the quantised KV cache (E4M3: 1 sign, 4 exponent and 3
// mantissa bits, max 448); its rows carry a float32 scale per (token, KV head).
struct fp8_e4m3 {
    uint8_t bits;
};

template <> struct Elem<fp8_e4m3> {
    static constexpr int kVec = 16;
    static constexpr bool kScaled = true;
    // 16 codes -> 16 floats (an E4M3 value is exact in half precision)
    static __device__ __forceinline__ void unpack(const uint4 &u, float *f) {
        const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                const __half2_raw h = __nv_cvt_fp8x2_to_halfraw2(
                    static_cast<__nv_fp8x2_storage_t>((w[i] >> (16 * j)) & 0xffffu), __NV_E4M3);
                const float2 v = __half22float2(*reinterpret_cast<const __half2 *>(&h));
                f[4 * i + 2 * j] = v.x;
                f[4 * i + 2 * j + 1] = v.y;
            }
        }
    }
    // 8 codes -> 8 floats
    static __device__ __forceinline__ void unpack8(const uint2 &u, float *f) {
        const uint32_t w[2] = {u.x, u.y};
#pragma unroll
        for (int i = 0; i < 2; ++i) {
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                const __half2_raw h = __nv_cvt_fp8x2_to_halfraw2(
                    static_cast<__nv_fp8x2_storage_t>((w[i] >> (16 * j)) & 0xffffu), __NV_E4M3);
                const float2 v = __half22float2(*reinterpret_cast<const __half2 *>(&h));
                f[4 * i + 2 * j] = v.x;
                f[4 * i + 2 * j + 1] = v.y;
            }
        }
    }
};

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// Request that owns packed query row `row`: the last r with cu[r] <= row
// (binary search over cu_seqlens_q, as one block does for its own rows).
__device__ __forceinline__ int request_of_row(const int32_t *cu, int num_seqs, int64_t row) {
    int lo = 0, hi = num_seqs - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (cu[mid] <= row) lo = mid;
        else hi = mid - 1;
    }
    return lo;
}

}  // namespace pa
