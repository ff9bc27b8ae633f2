// Instantiations of the paged decode kernels for bf16 queries over the
// quantised cache (E4M3 codes + a float32 scale per row) with head_dim 256
// (query-head groups 1..8); see decode_kernel.cuh.
#include "decode_kernel.cuh"

namespace pa {

cudaError_t launch_decode_fp8kv_d256(int group, const CUtensorMap &kmap, const CUtensorMap &vmap,
                                    const DecodeArgs &a, dim3 grid, cudaStream_t stream) {
    return launch_decode_group<__nv_bfloat16, 256, fp8_e4m3>(group, kmap, vmap, a, grid, stream);
}

}  // namespace pa
