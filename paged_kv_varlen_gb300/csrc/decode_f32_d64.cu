// Instantiations of the paged decode kernels for f32 K/V with head_dim 64
// (query-head groups 1..8); see decode_kernel.cuh.
#include "decode_kernel.cuh"

namespace pa {

cudaError_t launch_decode_f32_d64(int group, const CUtensorMap &kmap, const CUtensorMap &vmap,
                                   const DecodeArgs &a, dim3 grid, cudaStream_t stream) {
    return launch_decode_group<float, 64>(group, kmap, vmap, a, grid, stream);
}


}  // namespace pa
