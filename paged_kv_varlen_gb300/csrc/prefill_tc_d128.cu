// Instantiations of the tensor-core multi-query-row kernel for head_dim 128
// (query-head groups 1..8); see prefill_tc.cuh.
#include "prefill_tc.cuh"

namespace pa {

cudaError_t launch_prefill_tc_d128(int group, const CUtensorMap &qmap, const CUtensorMap &kmap,
                                  const CUtensorMap &vmap, const TcArgs &a, int grid,
                                  cudaStream_t stream) {
    return launch_prefill_tc_group<128>(group, qmap, kmap, vmap, a, grid, stream);
}

}  // namespace pa
