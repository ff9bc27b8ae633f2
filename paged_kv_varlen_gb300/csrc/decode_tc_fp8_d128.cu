// Instantiations of the tensor-core decode kernel over the quantised KV cache
// for head_dim 128 (query-head groups 1..8); see decode_tc_fp8.cuh.
#include "decode_tc_fp8.cuh"

namespace pa {

cudaError_t launch_decode_tc_fp8_d128(int group, const CUtensorMap &qmap, const CUtensorMap &kmap,
                                     const CUtensorMap &vmap, const DecodeTcArgs &a, int grid,
                                     cudaStream_t stream) {
    return launch_decode_tc_fp8_group<128>(group, qmap, kmap, vmap, a, grid, stream);
}

}  // namespace pa
