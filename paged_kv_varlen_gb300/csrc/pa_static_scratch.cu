// pa_static_scratch.cu -- pa_varlen_attention_static_scratch: the attention
// call for callers that cannot allocate device memory.  The split-KV partials
// go to a fixed array that is part of the library's own device image, so the
// call needs no workspace and allocates nothing.
#include <cstdio>
#include <mutex>

#include "pa.h"
#include "pa_internal.h"

#define PA_API extern "C" __attribute__((visibility("default")))

namespace pa {
namespace {

// The scratch itself.  It is loaded with the library's device code and stays
// resident on every GPU that uses the library until the process exits.
static __device__ __align__(256) unsigned char g_static_scratch[PA_STATIC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
void *g_scratch_ptr[kMaxDevices];
bool g_scratch_ready[kMaxDevices];
std::mutex g_scratch_mu;

// Device address of the scratch on the current device.  In host code the
// array's name only stands for the symbol, never for a usable address, so the
// address is looked up once per device (with that device current) and cached.
pa_status scratch_address(void **out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        set_last_error("static scratch: no current CUDA device");
        return PA_ERR_CUDA;
    }
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    if (!g_scratch_ready[dev]) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_static_scratch);
        if (e != cudaSuccess) {
            char msg[200];
            snprintf(msg, sizeof msg, "static scratch: cudaGetSymbolAddress failed: %s",
                     cudaGetErrorString(e));
            set_last_error(msg);
            return PA_ERR_CUDA;
        }
        g_scratch_ptr[dev] = p;
        g_scratch_ready[dev] = true;
    }
    *out = g_scratch_ptr[dev];
    return PA_OK;
}

}  // namespace
}  // namespace pa

using namespace pa;

PA_API pa_status pa_varlen_attention_static_scratch(
    void *out, const void *q, const void *key_cache, const void *value_cache,
    const int32_t *cu_seqlens_q, const int32_t *seq_lens_k, const int32_t *block_tables,
    int max_blocks_per_seq, int num_seqs, int64_t total_q, int max_seqlen_q, int max_seqlen_k,
    int num_q_heads, int num_kv_heads, int head_dim, int block_size, int64_t num_blocks,
    float scale, const float *sinks, int causal, int partition_size, pa_dtype dtype,
    void *stream) {
    // the attention call's own argument checks come first, so a bad argument
    // gets the same status (and message) as from pa_varlen_attention
    pa_status st = check_attention_args(out, q, key_cache, value_cache, cu_seqlens_q, seq_lens_k,
                                        block_tables, max_blocks_per_seq, num_seqs, total_q,
                                        max_seqlen_q, max_seqlen_k, num_q_heads, num_kv_heads,
                                        head_dim, block_size, num_blocks, sinks, partition_size,
                                        dtype);
    if (st != PA_OK || total_q == 0) return st;
    // A split plan that needs more than the array holds is refused by the
    // attention call's workspace check, before any launch, with the bytes it
    // needed in pa_last_error_string().
    void *scratch = nullptr;
    st = scratch_address(&scratch);
    if (st != PA_OK) return st;
    return pa_varlen_attention(out, q, key_cache, value_cache, cu_seqlens_q, seq_lens_k,
                               block_tables, max_blocks_per_seq, num_seqs, total_q, max_seqlen_q,
                               max_seqlen_k, num_q_heads, num_kv_heads, head_dim, block_size,
                               num_blocks, scale, sinks, causal, partition_size, scratch,
                               PA_STATIC_SCRATCH_BYTES, dtype, stream);
}
