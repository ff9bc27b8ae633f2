// Instantiations of the paged decode kernels for bf16 K/V with head_dim 64
// (query-head groups 1..8); see decode_kernel.cuh.
#include "decode_kernel.cuh"

namespace pa {

cudaError_t launch_decode_bf16_d64(int group, const CUtensorMap &kmap, const CUtensorMap &vmap,
                                   const DecodeArgs &a, dim3 grid, cudaStream_t stream) {
    return launch_decode_group<__nv_bfloat16, 64>(group, kmap, vmap, a, grid, stream);
}


}  // namespace pa
