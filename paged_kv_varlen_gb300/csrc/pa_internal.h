// pa_internal.h -- host-side structures shared between the C-ABI layer
// (pa_api.cu) and the kernel translation units.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <utility>

#include "pa.h"

namespace pa {

constexpr float kLog2e = 1.4426950408889634f;   // log2(e)

// Arguments of the paged decode / multi-row kernel (CUDA cores).
struct DecodeArgs {
    void *out;                 // [total_q, Hq, D]
    const void *q;             // [total_q, Hq, D]
    const int32_t *cu_seqlens_q;
    const int32_t *seq_lens_k;
    const int32_t *block_tables;
    int max_blocks_per_seq;
    int num_seqs;
    int num_q_heads;
    int num_kv_heads;
    int block_size;
    float qscale;              // scale * log2(e)
    const float *sinks;        // [Hq] or nullptr
    int causal;
    // mode 0: grid (max_parts, Hkv, num_seqs); single-query requests only.
    // mode 1: grid (total_q, Hkv); rows of multi-query requests only.
    int mode;
    int partition_size;        // mode 0: > 0 writes split partials, 0 = whole range
    int max_parts;
    float *part_o;             // [num_seqs, max_parts, Hq, D]
    float *part_m;             // [num_seqs, max_parts, Hq]
    float *part_l;             // [num_seqs, max_parts, Hq]
    int64_t total_q;
    int *err;                  // device error word
    int box_rows;              // rows per TMA box: divides both kernels' tile lengths
    // quantised cache only: float32 scale of each (slot, KV head)'s K and V row,
    // [num_blocks * block_size, H_kv]; nullptr for bf16 / fp32 caches
    const float *k_scales;
    const float *v_scales;
};

// Arguments of the tensor-core kernel for multi-query rows (bf16).
struct TcArgs {
    void *out;                 // [total_q, Hq, D] bf16
    const int32_t *cu_seqlens_q;
    const int32_t *seq_lens_k;
    const int32_t *block_tables;
    int max_blocks_per_seq;
    int num_seqs;
    int num_q_heads;
    int num_kv_heads;
    int block_size;
    float qscale;              // scale * log2(e)
    const float *sinks;        // [Hq] or nullptr
    int causal;
    int box_rows;              // rows per K/V TMA box (divides the V sub-tile and the block size)
    int *err;                  // device error word
    int *plan;                 // claim counter, order and unit prefix (mq_plan_kernel)
    int test_skip_first_k;     // 1: skip the K loads of each CTA's first tile (failure-path test)
    int64_t total_q;           // packed query rows (bounds of the output writes)
};

// The plan of the multi-query kernel's work units (prefill_plan.cu): in the
// workspace, [kPlanHeader] header ints (claim counter, requests, units), then
// order[num_seqs], then P[num_seqs + 1].
constexpr int kPlanHeader = 4;
__host__ __device__ constexpr size_t plan_bytes(int num_seqs) {
    return (size_t)(kPlanHeader + 2 * (size_t)num_seqs + 1) * sizeof(int);
}
struct MqPlanArgs {
    const int32_t *cu_seqlens_q;
    const int32_t *seq_lens_k;
    int num_seqs;
    int num_kv_heads;
    int block_rows;            // query rows per unit (128 / group)
    int tile_keys;             // keys per K/V tile
    int max_keys;              // max_blocks_per_seq * block_size
    int *plan;
};
cudaError_t launch_mq_plan(const MqPlanArgs &a, cudaStream_t stream);

// Arguments of the tensor-core kernel for single-query (decode) requests (bf16).
struct DecodeTcArgs {
    void *out;                 // [total_q, Hq, D] bf16
    const int32_t *cu_seqlens_q;
    const int32_t *seq_lens_k;
    const int32_t *block_tables;
    int max_blocks_per_seq;
    int num_seqs;
    int num_q_heads;
    int num_kv_heads;
    int block_size;
    float qscale;              // scale * log2(e)
    const float *sinks;        // [Hq] or nullptr
    int partition_size;        // > 0: split partials; 0: whole range, final output
    int max_parts;
    float *part_o;             // [num_seqs, max_parts, Hq, D]
    float *part_m;             // [num_seqs, max_parts, Hq]
    float *part_l;             // [num_seqs, max_parts, Hq]
    int box_rows;              // rows per K/V TMA box: divides 128, the block and partition sizes
    int *err;                  // device error word
    // split items cut at a CTA's share end: that CTA's partial of the item's
    // first part, [grid][G] (o: x D), and the table [grid] of (request, KV
    // head, partition, 0) of the cut item, request -1 when none
    float *xpart_o;
    float *xpart_m;
    float *xpart_l;
    int4 *cut_tab;
    // 1: the previous kernel of the stream is the scatter of this step's K/V
    // rows (it writes nothing else the kernel reads): only the K/V loads wait
    // for it.  0: the whole kernel waits for the previous kernel first.
    int after_scatter;
    // quantised cache only: float32 scale of each (slot, KV head)'s K and V
    // row, [num_blocks * block_size, H_kv], and the pool's pages (page ids at
    // or past it give a zero scale); nullptr / 0 for a bf16 cache
    const float *k_scales;
    const float *v_scales;
    int64_t num_blocks;
    // weight of an item's fixed cost in the work plan, in units of a fifth of
    // a key tile (an item weighs 5 per tile plus this): what one item costs
    // beyond its tiles on the kernel in question, measured
    int item_cost;
};

// Keys per K/V tile of the multi-query kernel, keys of one V sub-tile (the
// rows a TMA box may span) and query rows per work unit.
__host__ __device__ constexpr int tc_tile_keys(int head_dim) { return 128; }
__host__ __device__ constexpr int tc_vsub_keys(int head_dim) { return 8192 / head_dim; }
__host__ __device__ constexpr int tc_block_rows(int group) { return 128 / group; }

struct ReduceArgs {
    void *out;
    const float *part_o;
    const float *part_m;
    const float *part_l;
    const int32_t *cu_seqlens_q;
    const int32_t *seq_lens_k;
    int num_seqs;
    int max_parts;
    int partition_size;
    int num_q_heads;
    const float *sinks;
    int meta_before_wait;      // 1: cu_seqlens_q / seq_lens_k / sinks are read before
                               // waiting on the previous kernel (it does not write them)
    // extra partials of items cut between decode CTAs (ncut = 0: none)
    const float *xpart_o;      // [ncut][group][D]
    const float *xpart_m;      // [ncut][group]
    const float *xpart_l;
    const int4 *cut_tab;       // [ncut]: (request, KV head, partition, 0), request -1: none
    int ncut;
    int group;                 // query heads per KV head
};

// CTAs of the tensor-core decode kernel at most (one extra partial slot each).
constexpr int kMaxDecodeCtas = 256;

// Launches `kern` with programmatic stream serialization: it may start while
// the previous kernel of the stream runs and waits for it with pdl_wait().
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t stream, Args &&...args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

// Per (dtype, head_dim) launchers; `group` = Hq / Hkv in 1..8.
// Each returns the launch error (cudaSuccess if launched).
#define PA_DECLARE_DECODE(NAME) \
    cudaError_t NAME(int group, const CUtensorMap &kmap, const CUtensorMap &vmap, \
                     const DecodeArgs &a, dim3 grid, cudaStream_t stream);
PA_DECLARE_DECODE(launch_decode_f32_d64)
PA_DECLARE_DECODE(launch_decode_f32_d128)
PA_DECLARE_DECODE(launch_decode_f32_d256)
PA_DECLARE_DECODE(launch_decode_bf16_d64)
PA_DECLARE_DECODE(launch_decode_bf16_d128)
PA_DECLARE_DECODE(launch_decode_bf16_d256)
// bf16 queries over the quantised (E4M3 + scale) cache, head_dim 128 / 256
PA_DECLARE_DECODE(launch_decode_fp8kv_d128)
PA_DECLARE_DECODE(launch_decode_fp8kv_d256)
#undef PA_DECLARE_DECODE


// Keys per tile of the decode kernel: 16 KB of K+V per tile (32 rows of
// 256 B, 16 rows of 512 B, 8 rows of 1024 B), between 8 and 32 keys (one to
// four lanes per key in the QK step).
__host__ __device__ constexpr int decode_tile_keys(int elem_bytes, int head_dim) {
    return 8192 / (head_dim * elem_bytes) > 32 ? 32
           : (8192 / (head_dim * elem_bytes) < 8 ? 8 : 8192 / (head_dim * elem_bytes));
}

// gcd of the tile length and the block size: the rows one TMA box copies, so
// that a box never crosses a page boundary.
__host__ __device__ constexpr int gcd_int(int a, int b) { return b == 0 ? a : gcd_int(b, a % b); }

// Message returned by pa_last_error_string() on this thread.
void set_last_error(const char *msg);

// Host-side argument checks of pa_varlen_attention (no device call); sets the
// message of pa_last_error_string() on failure.
pa_status check_attention_args(const void *out, const void *q, const void *key_cache,
                               const void *value_cache, const int32_t *cu_seqlens_q,
                               const int32_t *seq_lens_k, const int32_t *block_tables,
                               int max_blocks_per_seq, int num_seqs, int64_t total_q,
                               int max_seqlen_q, int max_seqlen_k, int num_q_heads,
                               int num_kv_heads, int head_dim, int block_size, int64_t num_blocks,
                               const float *sinks, int partition_size, pa_dtype dtype);

// Tensor-core kernel for multi-query rows, per head_dim (bf16 only):
// persistent, `grid` CTAs (at most one per SM) claim the work units of the
// plan written by mq_plan_kernel (launched just before it on the stream).
#define PA_DECLARE_TC(NAME) \
    cudaError_t NAME(int group, const CUtensorMap &qmap, const CUtensorMap &kmap, \
                     const CUtensorMap &vmap, const TcArgs &a, int grid, cudaStream_t stream);
PA_DECLARE_TC(launch_prefill_tc_d64)
PA_DECLARE_TC(launch_prefill_tc_d128)
PA_DECLARE_TC(launch_prefill_tc_d256)
#undef PA_DECLARE_TC

// Tensor-core kernel for single-query requests, per head_dim (bf16; 128 and
// 256): persistent, grid.x CTAs (at most one per SM) share the batch's work.
#define PA_DECLARE_DTC(NAME) \
    cudaError_t NAME(int group, const CUtensorMap &qmap, const CUtensorMap &kmap, \
                     const CUtensorMap &vmap, const DecodeTcArgs &a, int grid, \
                     cudaStream_t stream);
PA_DECLARE_DTC(launch_decode_tc_d128)
PA_DECLARE_DTC(launch_decode_tc_d256)
// the same over the quantised cache (E4M3 codes + float32 row scales)
PA_DECLARE_DTC(launch_decode_tc_fp8_d128)
PA_DECLARE_DTC(launch_decode_tc_fp8_d256)
#undef PA_DECLARE_DTC

cudaError_t launch_reduce(int elem_bytes, int head_dim, const ReduceArgs &a, cudaStream_t stream);
// Partitions per request the reduce takes (its weights and maxima live in
// shared memory: 8 bytes per partition).
constexpr int kMaxReduceParts = 12288;

cudaError_t launch_reshape_and_cache(const void *key, const void *value, int64_t stride_bytes,
                                     void *key_cache, void *value_cache, const int64_t *slots,
                                     int64_t num_tokens, int64_t row_bytes, int64_t num_slots,
                                     cudaStream_t stream);

// reshape_and_cache into the quantised cache (E4M3 codes + a float32 scale per
// row); key / value are bf16 (elem_bytes 2) or float32 (4), stride in elements.
cudaError_t launch_quantize_kv_fp8(const void *key, const void *value, int64_t stride,
                                   int elem_bytes, uint8_t *key_codes, uint8_t *value_codes,
                                   float *key_scales, float *value_scales, const int64_t *slots,
                                   int64_t num_tokens, int num_kv_heads, int head_dim,
                                   int64_t num_slots, cudaStream_t stream);

}  // namespace pa
