// pa_api.cu -- the C ABI (include/pa.h): host-side argument checks, the
// split-KV plan, TMA tensor maps over the page pool, and the launch sequence
// of one attention call.  Everything here is host code except the device
// error word.
#include <algorithm>
#include <atomic>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>

#include "pa.h"
#include "pa_internal.h"

#define PA_API extern "C" __attribute__((visibility("default")))

namespace pa {
namespace {

// The device error word of this library: one int per device that loads it,
// read and cleared by pa_device_error().
__device__ int g_error_word;

thread_local char g_last_error[256] = "no error";

// Set by pa_test_expire_next_wait(): the next multi-query launch skips the K
// loads of each CTA's first tile.
std::atomic<int> g_expire_next_wait{0};

pa_status cuda_fail(cudaError_t e, const char *where) {
    snprintf(g_last_error, sizeof g_last_error, "%s: %s (%s)", where, cudaGetErrorName(e),
             cudaGetErrorString(e));
    return PA_ERR_CUDA;
}

constexpr int kMaxDevices = 64;

struct DeviceInfo {
    int sm_count = 0;
    int *err = nullptr;
    bool ready = false;
};
DeviceInfo g_dev[kMaxDevices];
std::mutex g_dev_mu;

// SM count and error-word address of the current device (looked up once).
pa_status device_info(DeviceInfo *out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    if (dev < 0 || dev >= kMaxDevices) return PA_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_dev_mu);
    DeviceInfo &d = g_dev[dev];
    if (!d.ready) {
        e = cudaDeviceGetAttribute(&d.sm_count, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceGetAttribute");
        e = cudaGetSymbolAddress(reinterpret_cast<void **>(&d.err), g_error_word);
        if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress");
        d.ready = true;
    }
    *out = d;
    return PA_OK;
}

// cuTensorMapEncodeTiled through the runtime's driver entry point (no libcuda
// link dependency).
typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                  const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                  const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

// A 3-D map over one cache: x = element within a head row (D), y = KV head,
// z = token row of the pool (page * block_size + slot).  Boxes are 128 bytes
// wide (one swizzle span) and `box_rows` rows tall, 128-byte swizzled.
pa_status make_cache_map(CUtensorMap *map, const void *cache, pa_dtype dtype, int head_dim,
                         int num_kv_heads, int64_t pool_rows, int box_rows) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) {
        snprintf(g_last_error, sizeof g_last_error, "cuTensorMapEncodeTiled unavailable");
        return PA_ERR_CUDA;
    }
    const int e = dtype == PA_F32 ? 4 : 2;
    cuuint64_t dims[3] = {(cuuint64_t)head_dim, (cuuint64_t)num_kv_heads, (cuuint64_t)pool_rows};
    cuuint64_t strides[2] = {(cuuint64_t)head_dim * e, (cuuint64_t)head_dim * num_kv_heads * e};
    cuuint32_t box[3] = {(cuuint32_t)(128 / e), 1, (cuuint32_t)box_rows};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = fn(map, dtype == PA_F32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32
                                         : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                    3, const_cast<void *>(cache), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) {
        snprintf(g_last_error, sizeof g_last_error, "cuTensorMapEncodeTiled failed (%d)", (int)r);
        return PA_ERR_CUDA;
    }
    return PA_OK;
}

// A 3-D map over the packed bf16 queries: x = element of a head row (D),
// y = query head, z = packed query row.  A box is one 128-byte chunk of the
// `group` heads of one KV head for `rows` consecutive query rows, i.e. one
// MMA row per (query row, head), 128-byte swizzled.
pa_status make_query_map(CUtensorMap *map, const void *q, int head_dim, int num_q_heads,
                         int64_t total_q, int group, int rows) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) {
        snprintf(g_last_error, sizeof g_last_error, "cuTensorMapEncodeTiled unavailable");
        return PA_ERR_CUDA;
    }
    cuuint64_t dims[3] = {(cuuint64_t)head_dim, (cuuint64_t)num_q_heads, (cuuint64_t)total_q};
    cuuint64_t strides[2] = {(cuuint64_t)head_dim * 2, (cuuint64_t)head_dim * num_q_heads * 2};
    cuuint32_t box[3] = {64, (cuuint32_t)group, (cuuint32_t)rows};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(q), dims,
                    strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) {
        snprintf(g_last_error, sizeof g_last_error, "cuTensorMapEncodeTiled (queries) failed (%d)",
                 (int)r);
        return PA_ERR_CUDA;
    }
    return PA_OK;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

// Split-KV workspace layout: part_o, part_m, part_l, then the extra partials
// of items cut between decode CTAs (xpart_o, xpart_m, xpart_l: one slot of up
// to 8 query heads per CTA) and their table.
struct SplitLayout {
    size_t o_bytes, ml_bytes, xo_bytes, xml_bytes, tab_bytes, total;
};

SplitLayout split_layout(int num_seqs, int max_parts, int num_q_heads, int head_dim) {
    SplitLayout L;
    const size_t units = (size_t)num_seqs * max_parts * num_q_heads;
    L.o_bytes = align256(units * head_dim * sizeof(float));
    L.ml_bytes = align256(units * sizeof(float));
    const size_t xunits = (size_t)kMaxDecodeCtas * 8;
    L.xo_bytes = align256(xunits * head_dim * sizeof(float));
    L.xml_bytes = align256(xunits * sizeof(float));
    L.tab_bytes = align256((size_t)kMaxDecodeCtas * sizeof(int4));
    L.total = L.o_bytes + 2 * L.ml_bytes + L.xo_bytes + 2 * L.xml_bytes + L.tab_bytes;
    return L;
}

int ceil_div(int64_t a, int64_t b) { return (int)((a + b - 1) / b); }

// The launches of one attention call, from its sizes alone (host arithmetic;
// the calls below launch exactly this).
struct LaunchPlan {
    bool quantised = false;    // pa_varlen_attention_fp8kv
    int partition_size = 0;    // split-KV partition used, 0: none
    int max_parts = 1;         // partitions per request
    bool tc_decode = false;    // single-query rows on a persistent tensor-core kernel
    int decode_grid[3] = {0, 0, 0};
    bool mq = false;           // rows of multi-query requests
    bool mq_tc = false;        // ... on the persistent tensor-core kernel
    int mq_grid[3] = {0, 0, 0};
    bool reduce = false;
    int reduce_grid[2] = {0, 0};
    size_t workspace = 0;      // bytes the call needs
    int head_dim = 0, group = 0;
    pa_dtype dtype = PA_BF16;
};

LaunchPlan plan_attention(int num_seqs, int64_t total_q, int max_seqlen_q, int max_seqlen_k,
                          int num_q_heads, int num_kv_heads, int head_dim, int partition_size,
                          pa_dtype dtype, bool quantised, int sm_count) {
    LaunchPlan L;
    L.quantised = quantised;
    L.head_dim = head_dim;
    L.group = num_q_heads / num_kv_heads;
    L.dtype = dtype;
    const int sms = sm_count > 0 ? sm_count : 148;
    const int P = pa_choose_partition_size(num_seqs, num_kv_heads, max_seqlen_k, partition_size,
                                           sms);
    L.partition_size = P;
    L.max_parts = (P > 0 && max_seqlen_k > 0) ? ceil_div(max_seqlen_k, P) : 1;
    L.tc_decode = quantised || (dtype == PA_BF16 && (head_dim == 128 || head_dim == 256));
    if (L.tc_decode) {
        const int64_t items_max = (int64_t)num_seqs * num_kv_heads * L.max_parts;
        L.decode_grid[0] = (int)std::min<int64_t>(std::min<int64_t>(sms, kMaxDecodeCtas),
                                                  items_max);
        L.decode_grid[1] = L.decode_grid[2] = 1;
    } else {
        L.decode_grid[0] = L.max_parts;
        L.decode_grid[1] = num_kv_heads;
        L.decode_grid[2] = num_seqs;
    }
    L.mq = max_seqlen_q > 1;
    L.mq_tc = L.mq && dtype == PA_BF16 && !quantised;
    if (L.mq_tc) {
        const int bq = tc_block_rows(L.group);
        const int64_t units_max = (total_q / bq + num_seqs) * (int64_t)num_kv_heads;
        L.mq_grid[0] = (int)std::min<int64_t>(sms, units_max);
        L.mq_grid[1] = L.mq_grid[2] = 1;
    } else if (L.mq) {
        L.mq_grid[0] = (int)total_q;
        L.mq_grid[1] = num_kv_heads;
        L.mq_grid[2] = 1;
    }
    L.reduce = P > 0;
    if (L.reduce) {
        L.reduce_grid[0] = num_seqs;
        L.reduce_grid[1] = num_q_heads;
    }
    if (L.mq_tc || P > 0)
        L.workspace = align256(plan_bytes(num_seqs)) +
                      (P > 0 ? split_layout(num_seqs, L.max_parts, num_q_heads, head_dim).total
                             : 0);
    return L;
}

// One line, key=value, of a plan (what pa_describe_plan and pa_last_plan return).
void format_plan(const LaunchPlan &L, char *buf, size_t n) {
    const char *dec = L.quantised   ? "paged_decode_tc_fp8"
                      : L.tc_decode ? "paged_decode_tc"
                                    : "paged_decode";
    const char *mq = !L.mq ? "none" : L.mq_tc ? "paged_prefill_tc" : "paged_decode_rows";
    snprintf(buf, n,
             "dtype=%s cache=%s head_dim=%d group=%d partition=%d max_parts=%d "
             "decode_kernel=%s decode_grid=%dx%dx%d mq_kernel=%s mq_grid=%dx%dx%d "
             "reduce=%s reduce_grid=%dx%d workspace=%zu",
             L.dtype == PA_F32 ? "f32" : "bf16", L.quantised ? "e4m3" : "plain", L.head_dim,
             L.group, L.partition_size, L.max_parts, dec, L.decode_grid[0], L.decode_grid[1],
             L.decode_grid[2], mq, L.mq_grid[0], L.mq_grid[1], L.mq_grid[2],
             L.reduce ? "split_reduce" : "none", L.reduce_grid[0], L.reduce_grid[1], L.workspace);
}

thread_local char g_last_plan[512] = "none";

// Records the plan of the call being launched; with PA_DEBUG=1 in the
// environment, also prints it to stderr.
void record_plan(const LaunchPlan &L) {
    static const bool debug = [] {
        const char *v = getenv("PA_DEBUG");
        return v && v[0] && strcmp(v, "0") != 0;
    }();
    format_plan(L, g_last_plan, sizeof g_last_plan);
    if (debug) fprintf(stderr, "pa: %s\n", g_last_plan);
}

// This step's K/V rows for pa_scatter_and_attend (one per query row).
struct StepScatter {
    const void *key;
    const void *value;
    int64_t stride;                 // elements between tokens
    const int64_t *slot_mapping;
};

}  // namespace

// Lets other translation units of the library report a message through
// pa_last_error_string().
void set_last_error(const char *msg) { snprintf(g_last_error, sizeof g_last_error, "%s", msg); }

}  // namespace pa

using namespace pa;

PA_API const char *pa_status_string(pa_status s) {
    switch (s) {
        case PA_OK: return "PA_OK";
        case PA_ERR_INVALID_ARG: return "PA_ERR_INVALID_ARG";
        case PA_ERR_UNSUPPORTED: return "PA_ERR_UNSUPPORTED";
        case PA_ERR_WORKSPACE: return "PA_ERR_WORKSPACE";
        case PA_ERR_CUDA: return "PA_ERR_CUDA";
    }
    return "PA_ERR_UNKNOWN";
}

PA_API const char *pa_last_error_string(void) { return g_last_error; }

PA_API pa_status pa_describe_plan(int num_seqs, int64_t total_q, int max_seqlen_q,
                                  int max_seqlen_k, int num_q_heads, int num_kv_heads,
                                  int head_dim, int partition_size, pa_dtype dtype, int quantised,
                                  int sm_count, char *buf, size_t buf_len) {
    if (!buf || buf_len == 0) return PA_ERR_INVALID_ARG;
    buf[0] = 0;
    if ((dtype != PA_F32 && dtype != PA_BF16) || num_seqs <= 0 || total_q <= 0 ||
        max_seqlen_q < 0 || max_seqlen_k < 0 || num_q_heads <= 0 || num_kv_heads <= 0 ||
        num_q_heads % num_kv_heads != 0 || head_dim <= 0 || partition_size < -1 ||
        (quantised && dtype != PA_BF16)) {
        snprintf(g_last_error, sizeof g_last_error, "pa_describe_plan: invalid sizes");
        return PA_ERR_INVALID_ARG;
    }
    format_plan(plan_attention(num_seqs, total_q, max_seqlen_q, max_seqlen_k, num_q_heads,
                               num_kv_heads, head_dim, partition_size, dtype, quantised != 0,
                               sm_count),
                buf, buf_len);
    return PA_OK;
}

PA_API const char *pa_last_plan(void) { return g_last_plan; }

PA_API const char *pa_build_info(void) {
    return "libpa paged varlen attention; sm_103a; kernels: reshape_and_cache, "
           "paged_decode_tc (tcgen05/TMEM, persistent), paged_decode_tc_fp8 (E4M3 cache, "
           "tcgen05), paged_decode (TMA ring, CUDA cores), "
           "paged_prefill_tc (tcgen05/TMEM), split_reduce";
}

PA_API int pa_choose_partition_size(int num_seqs, int num_kv_heads, int max_seqlen_k,
                                    int partition_size, int sm_count) {
    if (partition_size < 0) return 0;
    if (partition_size > 0) return partition_size;
    if (max_seqlen_k <= 512) return 0;
    // Work budget: keep every SM busy with several partitions.  Long
    // partitions first (fewer partials to write and reduce, less per-partition
    // overhead), shorter when the batch is too small to fill the GPU (the
    // page's 512-then-256 order, with 1024 ahead of it for large batches).
    const int64_t units = (int64_t)num_seqs * num_kv_heads;
    const int64_t want = (int64_t)4 * (sm_count > 0 ? sm_count : 148);
    if (units >= want && max_seqlen_k <= 2048) return 0;
    if (units * (max_seqlen_k / 1024) >= 2 * want) return 1024;
    if (units * (max_seqlen_k / 512) >= want) return 512;
    return 256;
}

PA_API size_t pa_varlen_attention_workspace_size(int num_seqs, int max_seqlen_k,
                                                 int num_q_heads, int head_dim,
                                                 int partition_size) {
    if (num_seqs <= 0 || num_q_heads <= 0 || head_dim <= 0) return 0;
    size_t n = align256(plan_bytes(num_seqs));   // the multi-query kernel's unit plan
    if (partition_size < 0) return n;
    const int P = partition_size > 0 ? partition_size : 256;  // auto picks 0, 256, 512 or 1024
    const int max_parts = max_seqlen_k > 0 ? ceil_div(max_seqlen_k, P) : 1;
    return n + split_layout(num_seqs, max_parts, num_q_heads, head_dim).total;
}

PA_API pa_status pa_reshape_and_cache(const void *key, const void *value, int64_t kv_token_stride,
                                      void *key_cache, void *value_cache,
                                      const int64_t *slot_mapping, int64_t num_tokens,
                                      int num_kv_heads, int head_dim, int block_size,
                                      int64_t num_blocks, pa_dtype dtype, void *stream) {
    if (dtype != PA_F32 && dtype != PA_BF16) return PA_ERR_INVALID_ARG;
    if (num_tokens < 0 || num_kv_heads <= 0 || head_dim <= 0 || block_size <= 0 ||
        num_blocks <= 0)
        return PA_ERR_INVALID_ARG;
    if (kv_token_stride < (int64_t)num_kv_heads * head_dim) return PA_ERR_INVALID_ARG;
    if (num_tokens == 0) return PA_OK;
    if (!key || !value || !key_cache || !value_cache || !slot_mapping) return PA_ERR_INVALID_ARG;
    const int64_t e = dtype == PA_F32 ? 4 : 2;
    if (((reinterpret_cast<uintptr_t>(key) | reinterpret_cast<uintptr_t>(value) |
          reinterpret_cast<uintptr_t>(key_cache) | reinterpret_cast<uintptr_t>(value_cache)) %
         e) != 0)
        return PA_ERR_INVALID_ARG;
    if (num_tokens > (int64_t)0x7fffffff * 8) return PA_ERR_UNSUPPORTED;
    cudaError_t err = launch_reshape_and_cache(
        key, value, kv_token_stride * e, key_cache, value_cache, slot_mapping, num_tokens,
        (int64_t)num_kv_heads * head_dim * e, num_blocks * block_size,
        static_cast<cudaStream_t>(stream));
    if (err != cudaSuccess) return cuda_fail(err, "reshape_and_cache launch");
    return PA_OK;
}

namespace pa {

// Host-side argument checks of pa_varlen_attention (and of every call built on
// it); each failure names its reason in pa_last_error_string().
pa_status check_attention_args(const void *out, const void *q, const void *key_cache,
                               const void *value_cache, const int32_t *cu_seqlens_q,
                               const int32_t *seq_lens_k, const int32_t *block_tables,
                               int max_blocks_per_seq, int num_seqs, int64_t total_q,
                               int max_seqlen_q, int max_seqlen_k, int num_q_heads,
                               int num_kv_heads, int head_dim, int block_size, int64_t num_blocks,
                               const float *sinks, int partition_size, pa_dtype dtype) {
    auto fail = [](pa_status st, const char *why) {
        snprintf(g_last_error, sizeof g_last_error, "%s", why);
        return st;
    };
    if (dtype != PA_F32 && dtype != PA_BF16) return fail(PA_ERR_INVALID_ARG, "unknown dtype");
    if (num_seqs < 0 || total_q < 0 || max_seqlen_q < 0 || max_seqlen_k < 0)
        return fail(PA_ERR_INVALID_ARG, "negative size");
    if (total_q == 0) return PA_OK;
    if (num_seqs == 0) return fail(PA_ERR_INVALID_ARG, "query rows but no request");
    if (!out || !q || !key_cache || !value_cache || !cu_seqlens_q || !seq_lens_k || !block_tables)
        return fail(PA_ERR_INVALID_ARG, "null pointer");
    if (num_q_heads <= 0 || num_kv_heads <= 0 || num_q_heads % num_kv_heads != 0)
        return fail(PA_ERR_INVALID_ARG, "num_q_heads must be a positive multiple of num_kv_heads");
    if (max_blocks_per_seq <= 0 || num_blocks <= 0 || block_size <= 0)
        return fail(PA_ERR_INVALID_ARG, "block table and pool sizes must be positive");
    if (partition_size < -1 || (partition_size > 0 && partition_size % 32 != 0))
        return fail(PA_ERR_INVALID_ARG,
                    "partition_size must be -1, 0 or a positive multiple of 32");
    if (num_q_heads / num_kv_heads > 8)
        return fail(PA_ERR_UNSUPPORTED, "more than 8 query heads per KV head");
    if (head_dim != 64 && head_dim != 128 && head_dim != 256)
        return fail(PA_ERR_UNSUPPORTED, "head_dim must be 64, 128 or 256");
    if (block_size % 8 != 0 || block_size > 1024)
        return fail(PA_ERR_UNSUPPORTED, "block_size must be a multiple of 8 up to 1024");
    if (num_seqs > 65535 || num_kv_heads > 65535)
        return fail(PA_ERR_UNSUPPORTED, "more than 65535 requests or KV heads");
    if (num_blocks * block_size > 0x7fffffffLL ||
        (int64_t)max_blocks_per_seq * block_size > 0x7fffffffLL || total_q > 0x7fffffffLL)
        return fail(PA_ERR_UNSUPPORTED, "pool, block table or batch beyond 2^31 rows");
    if (!aligned16(out) || !aligned16(q) || !aligned16(key_cache) || !aligned16(value_cache))
        return fail(PA_ERR_INVALID_ARG, "q, out and the caches must be 16-byte aligned");
    if (sinks && (reinterpret_cast<uintptr_t>(sinks) & 3))
        return fail(PA_ERR_INVALID_ARG, "sinks must be 4-byte aligned");
    return PA_OK;
}

}  // namespace pa

// The attention call; with `fs`, this step's K/V rows are scattered first --
// inside the tensor-core decode kernel when it runs, else by the scatter kernel.
static pa_status attention_impl(void *out, const void *q, const void *key_cache,
                                const void *value_cache, const int32_t *cu_seqlens_q,
                                const int32_t *seq_lens_k, const int32_t *block_tables,
                                int max_blocks_per_seq, int num_seqs, int64_t total_q,
                                int max_seqlen_q, int max_seqlen_k, int num_q_heads,
                                int num_kv_heads, int head_dim, int block_size, int64_t num_blocks,
                                float scale, const float *sinks, int causal, int partition_size,
                                void *workspace, size_t workspace_bytes, pa_dtype dtype,
                                void *stream, const StepScatter *fs) {
    // ---- host-side checks (nothing is launched if one fails)
    pa_status st = check_attention_args(out, q, key_cache, value_cache, cu_seqlens_q, seq_lens_k,
                                        block_tables, max_blocks_per_seq, num_seqs, total_q,
                                        max_seqlen_q, max_seqlen_k, num_q_heads, num_kv_heads,
                                        head_dim, block_size, num_blocks, sinks, partition_size,
                                        dtype);
    if (st != PA_OK) return st;
    if (total_q == 0) return PA_OK;
    const int group = num_q_heads / num_kv_heads;

    DeviceInfo dev;
    st = device_info(&dev);
    if (st != PA_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);

    // ---- split plan and workspace
    const LaunchPlan plan = plan_attention(num_seqs, total_q, max_seqlen_q, max_seqlen_k,
                                           num_q_heads, num_kv_heads, head_dim, partition_size,
                                           dtype, false, dev.sm_count);
    const int P = plan.partition_size;
    const int max_parts = plan.max_parts;
    float *part_o = nullptr, *part_m = nullptr, *part_l = nullptr;
    float *xpart_o = nullptr, *xpart_m = nullptr, *xpart_l = nullptr;
    int4 *cut_tab = nullptr;
    if (P > 0 && max_parts > kMaxReduceParts) {
        snprintf(g_last_error, sizeof g_last_error,
                 "%d split-KV partitions per request, at most %d", max_parts, kMaxReduceParts);
        return PA_ERR_UNSUPPORTED;
    }
    // the workspace: the multi-query kernel's unit plan, then the split partials
    const bool mq_tc = plan.mq_tc;
    const size_t plan_sz = align256(plan_bytes(num_seqs));
    int *unit_plan = nullptr;
    if (mq_tc || P > 0) {
        const size_t need = plan.workspace;
        if (!workspace || workspace_bytes < need || !aligned16(workspace)) {
            snprintf(g_last_error, sizeof g_last_error,
                     "this call needs %zu bytes of 16-byte aligned workspace (split-KV "
                     "partition %d, %d partitions per request); %zu given%s",
                     need, P, max_parts, workspace ? workspace_bytes : (size_t)0,
                     workspace && !aligned16(workspace) ? " (misaligned)" : "");
            return PA_ERR_WORKSPACE;
        }
        unit_plan = static_cast<int *>(workspace);
    }
    if (P > 0) {
        const SplitLayout L = split_layout(num_seqs, max_parts, num_q_heads, head_dim);
        char *w = static_cast<char *>(workspace) + plan_sz;
        part_o = reinterpret_cast<float *>(w);
        part_m = reinterpret_cast<float *>(w + L.o_bytes);
        part_l = reinterpret_cast<float *>(w + L.o_bytes + L.ml_bytes);
        w += L.o_bytes + 2 * L.ml_bytes;
        xpart_o = reinterpret_cast<float *>(w);
        xpart_m = reinterpret_cast<float *>(w + L.xo_bytes);
        xpart_l = reinterpret_cast<float *>(w + L.xo_bytes + L.xml_bytes);
        cut_tab = reinterpret_cast<int4 *>(w + L.xo_bytes + 2 * L.xml_bytes);
    }

    // ---- tensor maps over the two caches
    const int e = dtype == PA_F32 ? 4 : 2;
    // TMA box height: divides the kernel's tile length and the block size, so a
    // box never crosses a page
    const int box_rows = gcd_int(decode_tile_keys(e, head_dim), block_size);
    CUtensorMap kmap, vmap;
    st = make_cache_map(&kmap, key_cache, dtype, head_dim, num_kv_heads, num_blocks * block_size,
                        box_rows);
    if (st != PA_OK) return st;
    st = make_cache_map(&vmap, value_cache, dtype, head_dim, num_kv_heads,
                        num_blocks * block_size, box_rows);
    if (st != PA_OK) return st;

    DecodeArgs a;
    memset(&a, 0, sizeof a);
    a.out = out;
    a.q = q;
    a.cu_seqlens_q = cu_seqlens_q;
    a.seq_lens_k = seq_lens_k;
    a.block_tables = block_tables;
    a.max_blocks_per_seq = max_blocks_per_seq;
    a.num_seqs = num_seqs;
    a.num_q_heads = num_q_heads;
    a.num_kv_heads = num_kv_heads;
    a.block_size = block_size;
    a.qscale = scale * kLog2e;
    a.sinks = sinks;
    a.causal = causal ? 1 : 0;
    a.partition_size = P;
    a.max_parts = max_parts;
    a.part_o = part_o;
    a.part_m = part_m;
    a.part_l = part_l;
    a.total_q = total_q;
    a.err = dev.err;
    a.box_rows = box_rows;

    auto launch = [&](dim3 grid) -> cudaError_t {
        if (dtype == PA_F32) {
            switch (head_dim) {
                case 64: return launch_decode_f32_d64(group, kmap, vmap, a, grid, s);
                case 128: return launch_decode_f32_d128(group, kmap, vmap, a, grid, s);
                default: return launch_decode_f32_d256(group, kmap, vmap, a, grid, s);
            }
        }
        switch (head_dim) {
            case 64: return launch_decode_bf16_d64(group, kmap, vmap, a, grid, s);
            case 128: return launch_decode_bf16_d128(group, kmap, vmap, a, grid, s);
            default: return launch_decode_bf16_d256(group, kmap, vmap, a, grid, s);
        }
    };

    // 0) this step's K/V rows (pa_scatter_and_attend): the scatter kernel; the
    //    tensor-core decode kernel launched next overlaps it (programmatic
    //    dependent launch) and only its K/V loads wait for it
    const bool tc_decode = plan.tc_decode;
    int dtc_grid = 0;   // CTAs of the tensor-core decode kernel (0: not launched)
    cudaError_t ce;
    record_plan(plan);
    if (fs) {
        const int64_t eb = dtype == PA_F32 ? 4 : 2;
        ce = launch_reshape_and_cache(fs->key, fs->value, fs->stride * eb, const_cast<void *>(key_cache),
                                      const_cast<void *>(value_cache), fs->slot_mapping, total_q,
                                      (int64_t)num_kv_heads * head_dim * eb,
                                      num_blocks * block_size, s);
        if (ce != cudaSuccess) return cuda_fail(ce, "reshape_and_cache launch");
    }
    // 1) single-query requests (decode).  bf16 at head_dim 128 / 256: the
    //    persistent tensor-core kernel, one CTA per SM sharing the batch's
    //    (request, KV head, partition) items; otherwise the CUDA-core kernel,
    //    one CTA per (partition, KV head, request).
    if (tc_decode) {
        // box rows divide the 128-key tile, the block size and the partition
        const int dbox = gcd_int(gcd_int(128, block_size), P > 0 ? P : 128);
        CUtensorMap qmap_d, kmap_d, vmap_d;
        st = make_query_map(&qmap_d, q, head_dim, num_q_heads, total_q, group, 1);
        if (st != PA_OK) return st;
        st = make_cache_map(&kmap_d, key_cache, dtype, head_dim, num_kv_heads,
                            num_blocks * block_size, dbox);
        if (st != PA_OK) return st;
        st = make_cache_map(&vmap_d, value_cache, dtype, head_dim, num_kv_heads,
                            num_blocks * block_size, dbox);
        if (st != PA_OK) return st;
        DecodeTcArgs da;
        memset(&da, 0, sizeof da);
        da.out = out;
        da.cu_seqlens_q = cu_seqlens_q;
        da.seq_lens_k = seq_lens_k;
        da.block_tables = block_tables;
        da.max_blocks_per_seq = max_blocks_per_seq;
        da.num_seqs = num_seqs;
        da.num_q_heads = num_q_heads;
        da.num_kv_heads = num_kv_heads;
        da.block_size = block_size;
        da.qscale = scale * kLog2e;
        da.sinks = sinks;
        da.partition_size = P;
        da.max_parts = max_parts;
        da.part_o = part_o;
        da.part_m = part_m;
        da.part_l = part_l;
        da.box_rows = dbox;
        da.err = dev.err;
        da.after_scatter = fs != nullptr ? 1 : 0;
        da.item_cost = 3;   // ~0.6 tile (the bf16 kernel's Q load, pipeline turn, epilogue)
        da.xpart_o = xpart_o;
        da.xpart_m = xpart_m;
        da.xpart_l = xpart_l;
        da.cut_tab = cut_tab;
        const int grid = plan.decode_grid[0];
        dtc_grid = grid;
        ce = head_dim == 128 ? launch_decode_tc_d128(group, qmap_d, kmap_d, vmap_d, da, grid, s)
                             : launch_decode_tc_d256(group, qmap_d, kmap_d, vmap_d, da, grid, s);
        if (ce != cudaSuccess) return cuda_fail(ce, "paged_decode_tc launch");
    } else {
        a.mode = 0;
        ce = launch(dim3(plan.decode_grid[0], plan.decode_grid[1], plan.decode_grid[2]));
        if (ce != cudaSuccess) return cuda_fail(ce, "paged_decode launch");
    }
    // 2) rows of multi-query requests (verify windows, prefill chunks): bf16 on
    //    the tensor cores, float32 on the CUDA-core row kernel
    if (mq_tc) {
        const int bq = tc_block_rows(group);
        // TMA box rows: divide the V sub-tile and the block size, so a box never
        // crosses a page
        const int tc_box = gcd_int(tc_vsub_keys(head_dim), block_size);
        CUtensorMap qmap, kmap_tc, vmap_tc;
        st = make_query_map(&qmap, q, head_dim, num_q_heads, total_q, group, bq);
        if (st != PA_OK) return st;
        st = make_cache_map(&kmap_tc, key_cache, dtype, head_dim, num_kv_heads,
                            num_blocks * block_size, tc_box);
        if (st != PA_OK) return st;
        st = make_cache_map(&vmap_tc, value_cache, dtype, head_dim, num_kv_heads,
                            num_blocks * block_size, tc_box);
        if (st != PA_OK) return st;
        // 1) the claim order of the work units (one CTA)
        MqPlanArgs pl;
        pl.cu_seqlens_q = cu_seqlens_q;
        pl.seq_lens_k = seq_lens_k;
        pl.num_seqs = num_seqs;
        pl.num_kv_heads = num_kv_heads;
        pl.block_rows = bq;
        pl.tile_keys = tc_tile_keys(head_dim);
        pl.max_keys = max_blocks_per_seq * block_size;
        pl.plan = unit_plan;
        ce = launch_mq_plan(pl, s);
        if (ce != cudaSuccess) return cuda_fail(ce, "mq_plan launch");
        // 2) the persistent multi-query kernel: at most one CTA per SM, no more
        //    than there are units
        TcArgs ta;
        ta.out = out;
        ta.cu_seqlens_q = cu_seqlens_q;
        ta.seq_lens_k = seq_lens_k;
        ta.block_tables = block_tables;
        ta.max_blocks_per_seq = max_blocks_per_seq;
        ta.num_seqs = num_seqs;
        ta.num_q_heads = num_q_heads;
        ta.num_kv_heads = num_kv_heads;
        ta.block_size = block_size;
        ta.qscale = scale * kLog2e;
        ta.sinks = sinks;
        ta.causal = causal ? 1 : 0;
        ta.box_rows = tc_box;
        ta.err = dev.err;
        ta.plan = unit_plan;
        ta.test_skip_first_k = g_expire_next_wait.exchange(0);
        ta.total_q = total_q;
        const int grid = plan.mq_grid[0];
        switch (head_dim) {
            case 64: ce = launch_prefill_tc_d64(group, qmap, kmap_tc, vmap_tc, ta, grid, s); break;
            case 128: ce = launch_prefill_tc_d128(group, qmap, kmap_tc, vmap_tc, ta, grid, s); break;
            default: ce = launch_prefill_tc_d256(group, qmap, kmap_tc, vmap_tc, ta, grid, s); break;
        }
        if (ce != cudaSuccess) return cuda_fail(ce, "paged_prefill_tc launch");
    } else if (max_seqlen_q > 1) {
        a.mode = 1;
        ce = launch(dim3((unsigned)plan.mq_grid[0], plan.mq_grid[1], 1));
        if (ce != cudaSuccess) return cuda_fail(ce, "paged_rows launch");
    }
    // 3) merge the split partials of the single-query requests
    if (P > 0) {
        ReduceArgs ra;
        ra.out = out;
        ra.part_o = part_o;
        ra.part_m = part_m;
        ra.part_l = part_l;
        ra.cu_seqlens_q = cu_seqlens_q;
        ra.seq_lens_k = seq_lens_k;
        ra.num_seqs = num_seqs;
        ra.max_parts = max_parts;
        ra.partition_size = P;
        ra.num_q_heads = num_q_heads;
        ra.sinks = sinks;
        ra.meta_before_wait = 1;   // the kernels before it write only out / partials
        ra.xpart_o = xpart_o;
        ra.xpart_m = xpart_m;
        ra.xpart_l = xpart_l;
        ra.cut_tab = cut_tab;
        ra.ncut = dtc_grid;   // 0 unless the tensor-core decode kernel ran
        ra.group = group;
        ce = launch_reduce(e, head_dim, ra, s);
        if (ce != cudaSuccess) return cuda_fail(ce, "split_reduce launch");
    }
    return PA_OK;
}

PA_API pa_status pa_varlen_attention(void *out, const void *q, const void *key_cache,
                                     const void *value_cache, const int32_t *cu_seqlens_q,
                                     const int32_t *seq_lens_k, const int32_t *block_tables,
                                     int max_blocks_per_seq, int num_seqs, int64_t total_q,
                                     int max_seqlen_q, int max_seqlen_k, int num_q_heads,
                                     int num_kv_heads, int head_dim, int block_size,
                                     int64_t num_blocks, float scale, const float *sinks,
                                     int causal, int partition_size, void *workspace,
                                     size_t workspace_bytes, pa_dtype dtype, void *stream) {
    return attention_impl(out, q, key_cache, value_cache, cu_seqlens_q, seq_lens_k, block_tables,
                          max_blocks_per_seq, num_seqs, total_q, max_seqlen_q, max_seqlen_k,
                          num_q_heads, num_kv_heads, head_dim, block_size, num_blocks, scale,
                          sinks, causal, partition_size, workspace, workspace_bytes, dtype,
                          stream, nullptr);
}

PA_API pa_status pa_scatter_and_attend(const void *key, const void *value, int64_t kv_token_stride,
                                       const int64_t *slot_mapping, int64_t num_tokens, void *out,
                                       const void *q, void *key_cache, void *value_cache,
                                       const int32_t *cu_seqlens_q, const int32_t *seq_lens_k,
                                       const int32_t *block_tables, int max_blocks_per_seq,
                                       int num_seqs, int64_t total_q, int max_seqlen_q,
                                       int max_seqlen_k, int num_q_heads, int num_kv_heads,
                                       int head_dim, int block_size, int64_t num_blocks,
                                       float scale, const float *sinks, int causal,
                                       int partition_size, void *workspace,
                                       size_t workspace_bytes, pa_dtype dtype, void *stream) {
    if (dtype != PA_F32 && dtype != PA_BF16) return PA_ERR_INVALID_ARG;
    if (num_tokens != total_q || num_tokens < 0) return PA_ERR_INVALID_ARG;
    if (num_kv_heads <= 0 || head_dim <= 0 ||
        kv_token_stride < (int64_t)num_kv_heads * head_dim)
        return PA_ERR_INVALID_ARG;
    if (num_tokens > 0 && (!key || !value || !slot_mapping)) return PA_ERR_INVALID_ARG;
    const uintptr_t e = dtype == PA_F32 ? 4 : 2;
    if (((reinterpret_cast<uintptr_t>(key) | reinterpret_cast<uintptr_t>(value)) % e) != 0)
        return PA_ERR_INVALID_ARG;
    const StepScatter fs = {key, value, kv_token_stride, slot_mapping};
    return attention_impl(out, q, key_cache, value_cache, cu_seqlens_q, seq_lens_k, block_tables,
                          max_blocks_per_seq, num_seqs, total_q, max_seqlen_q, max_seqlen_k,
                          num_q_heads, num_kv_heads, head_dim, block_size, num_blocks, scale,
                          sinks, causal, partition_size, workspace, workspace_bytes, dtype,
                          stream, &fs);
}

PA_API pa_status pa_split_kv_reduce(void *out, const float *part_out, const float *part_max,
                                    const float *part_sum, const int32_t *cu_seqlens_q,
                                    const int32_t *seq_lens_k, int num_seqs, int max_parts,
                                    int partition_size, int num_q_heads, int head_dim,
                                    const float *sinks, pa_dtype dtype, void *stream) {
    if (dtype != PA_F32 && dtype != PA_BF16) return PA_ERR_INVALID_ARG;
    if (num_seqs < 0 || max_parts <= 0 || partition_size <= 0 || num_q_heads <= 0)
        return PA_ERR_INVALID_ARG;
    if (head_dim != 64 && head_dim != 128 && head_dim != 256) return PA_ERR_UNSUPPORTED;
    if (num_seqs == 0) return PA_OK;
    if (num_seqs > 0x7fffffff || num_q_heads > 65535) return PA_ERR_UNSUPPORTED;
    if (max_parts > kMaxReduceParts) return PA_ERR_UNSUPPORTED;
    if (!out || !part_out || !part_max || !part_sum || !cu_seqlens_q || !seq_lens_k)
        return PA_ERR_INVALID_ARG;
    if (!aligned16(part_out) || (reinterpret_cast<uintptr_t>(out) & 3)) return PA_ERR_INVALID_ARG;
    ReduceArgs ra;
    ra.out = out;
    ra.part_o = part_out;
    ra.part_m = part_max;
    ra.part_l = part_sum;
    ra.cu_seqlens_q = cu_seqlens_q;
    ra.seq_lens_k = seq_lens_k;
    ra.num_seqs = num_seqs;
    ra.max_parts = max_parts;
    ra.partition_size = partition_size;
    ra.num_q_heads = num_q_heads;
    ra.sinks = sinks;
    ra.meta_before_wait = 0;   // the previous kernel may have written anything
    ra.xpart_o = nullptr;
    ra.xpart_m = nullptr;
    ra.xpart_l = nullptr;
    ra.cut_tab = nullptr;
    ra.ncut = 0;
    ra.group = 1;
    cudaError_t ce = launch_reduce(dtype == PA_F32 ? 4 : 2, head_dim, ra,
                                   static_cast<cudaStream_t>(stream));
    if (ce != cudaSuccess) return cuda_fail(ce, "split_reduce launch");
    return PA_OK;
}

PA_API void pa_test_expire_next_wait(void) { g_expire_next_wait.store(1); }

PA_API pa_status pa_device_error(int *code) {
    if (!code) return PA_ERR_INVALID_ARG;
    DeviceInfo dev;
    pa_status st = device_info(&dev);
    if (st != PA_OK) return st;
    cudaError_t e = cudaDeviceSynchronize();
    if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceSynchronize");
    e = cudaMemcpy(code, dev.err, sizeof(int), cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return cuda_fail(e, "read device error word");
    const int zero = 0;
    e = cudaMemcpy(dev.err, &zero, sizeof(int), cudaMemcpyHostToDevice);
    if (e != cudaSuccess) return cuda_fail(e, "clear device error word");
    return PA_OK;
}

// ---------------------------------------------------------------- quantised KV cache
namespace pa {

// A 3-D map over an 8-bit code cache: as make_cache_map, one byte per element,
// boxes 128 codes wide.
static pa_status make_code_map(CUtensorMap *map, const void *codes, int head_dim,
                               int num_kv_heads, int64_t pool_rows, int box_rows) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) {
        snprintf(g_last_error, sizeof g_last_error, "cuTensorMapEncodeTiled unavailable");
        return PA_ERR_CUDA;
    }
    cuuint64_t dims[3] = {(cuuint64_t)head_dim, (cuuint64_t)num_kv_heads, (cuuint64_t)pool_rows};
    cuuint64_t strides[2] = {(cuuint64_t)head_dim, (cuuint64_t)head_dim * num_kv_heads};
    cuuint32_t box[3] = {128, 1, (cuuint32_t)box_rows};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void *>(codes), dims,
                    strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) {
        snprintf(g_last_error, sizeof g_last_error, "cuTensorMapEncodeTiled (codes) failed (%d)",
                 (int)r);
        return PA_ERR_CUDA;
    }
    return PA_OK;
}

}  // namespace pa

PA_API pa_status pa_reshape_and_cache_fp8(const void *key, const void *value,
                                          int64_t kv_token_stride, void *key_codes,
                                          void *value_codes, float *key_scales,
                                          float *value_scales, const int64_t *slot_mapping,
                                          int64_t num_tokens, int num_kv_heads, int head_dim,
                                          int block_size, int64_t num_blocks, pa_dtype dtype,
                                          void *stream) {
    auto fail = [](const char *why) {
        set_last_error(why);
        return PA_ERR_INVALID_ARG;
    };
    if (dtype != PA_F32 && dtype != PA_BF16) return fail("unknown dtype");
    if (num_tokens < 0 || num_kv_heads <= 0 || block_size <= 0 || num_blocks <= 0)
        return fail("negative or empty size");
    if (head_dim != 128 && head_dim != 256) {
        set_last_error("the quantised cache takes head_dim 128 or 256");
        return PA_ERR_UNSUPPORTED;
    }
    if (kv_token_stride < (int64_t)num_kv_heads * head_dim)
        return fail("kv_token_stride shorter than a token's row");
    if (num_tokens == 0) return PA_OK;
    if (!key || !value || !key_codes || !value_codes || !key_scales || !value_scales ||
        !slot_mapping)
        return fail("null pointer");
    const int e = dtype == PA_F32 ? 4 : 2;
    if (((reinterpret_cast<uintptr_t>(key) | reinterpret_cast<uintptr_t>(value)) % (e * 4)) ||
        ((kv_token_stride * e) % (e * 4)) ||
        ((reinterpret_cast<uintptr_t>(key_codes) | reinterpret_cast<uintptr_t>(value_codes) |
          reinterpret_cast<uintptr_t>(key_scales) | reinterpret_cast<uintptr_t>(value_scales)) &
         3))
        return fail("rows must start on 4-element boundaries, codes and scales 4-byte aligned");
    if (num_tokens * num_kv_heads > (int64_t)0x7fffffff * 8) {
        set_last_error("too many (token, KV head) rows");
        return PA_ERR_UNSUPPORTED;
    }
    cudaError_t err = launch_quantize_kv_fp8(
        key, value, kv_token_stride, e, static_cast<uint8_t *>(key_codes),
        static_cast<uint8_t *>(value_codes), key_scales, value_scales, slot_mapping, num_tokens,
        num_kv_heads, head_dim, num_blocks * block_size, static_cast<cudaStream_t>(stream));
    if (err != cudaSuccess) return cuda_fail(err, "quantize_kv_fp8 launch");
    return PA_OK;
}

PA_API pa_status pa_varlen_attention_fp8kv(
    void *out, const void *q, const void *key_codes, const void *value_codes,
    const float *key_scales, const float *value_scales, const int32_t *cu_seqlens_q,
    const int32_t *seq_lens_k, const int32_t *block_tables, int max_blocks_per_seq, int num_seqs,
    int64_t total_q, int max_seqlen_q, int max_seqlen_k, int num_q_heads, int num_kv_heads,
    int head_dim, int block_size, int64_t num_blocks, float scale, const float *sinks, int causal,
    int partition_size, void *workspace, size_t workspace_bytes, pa_dtype dtype, void *stream) {
    // the attention call's checks (q and out in `dtype`, the code caches 16-byte aligned)
    pa_status st = check_attention_args(out, q, key_codes, value_codes, cu_seqlens_q, seq_lens_k,
                                        block_tables, max_blocks_per_seq, num_seqs, total_q,
                                        max_seqlen_q, max_seqlen_k, num_q_heads, num_kv_heads,
                                        head_dim, block_size, num_blocks, sinks, partition_size,
                                        dtype);
    if (st != PA_OK) return st;
    if (dtype != PA_BF16) {
        set_last_error("the quantised cache takes bf16 queries and output");
        return PA_ERR_UNSUPPORTED;
    }
    if (head_dim != 128 && head_dim != 256) {
        set_last_error("the quantised cache takes head_dim 128 or 256");
        return PA_ERR_UNSUPPORTED;
    }
    if (!key_scales || !value_scales ||
        ((reinterpret_cast<uintptr_t>(key_scales) | reinterpret_cast<uintptr_t>(value_scales)) &
         3)) {
        set_last_error("key_scales / value_scales missing or not 4-byte aligned");
        return PA_ERR_INVALID_ARG;
    }
    if (total_q == 0) return PA_OK;
    const int group = num_q_heads / num_kv_heads;
    DeviceInfo dev;
    st = device_info(&dev);
    if (st != PA_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);

    // split plan and workspace: the same layout as pa_varlen_attention's
    const LaunchPlan plan = plan_attention(num_seqs, total_q, max_seqlen_q, max_seqlen_k,
                                           num_q_heads, num_kv_heads, head_dim, partition_size,
                                           dtype, true, dev.sm_count);
    const int P = plan.partition_size;
    const int max_parts = plan.max_parts;
    if (P > 0 && max_parts > kMaxReduceParts) {
        snprintf(g_last_error, sizeof g_last_error,
                 "%d split-KV partitions per request, at most %d", max_parts, kMaxReduceParts);
        return PA_ERR_UNSUPPORTED;
    }
    float *part_o = nullptr, *part_m = nullptr, *part_l = nullptr;
    float *xpart_o = nullptr, *xpart_m = nullptr, *xpart_l = nullptr;
    int4 *cut_tab = nullptr;
    if (P > 0) {
        const size_t plan_sz = align256(plan_bytes(num_seqs));
        const SplitLayout L = split_layout(num_seqs, max_parts, num_q_heads, head_dim);
        const size_t need = plan.workspace;
        if (!workspace || workspace_bytes < need || !aligned16(workspace)) {
            snprintf(g_last_error, sizeof g_last_error,
                     "this call needs %zu bytes of 16-byte aligned workspace (split-KV "
                     "partition %d, %d partitions per request); %zu given%s",
                     need, P, max_parts, workspace ? workspace_bytes : (size_t)0,
                     workspace && !aligned16(workspace) ? " (misaligned)" : "");
            return PA_ERR_WORKSPACE;
        }
        char *w = static_cast<char *>(workspace) + plan_sz;
        part_o = reinterpret_cast<float *>(w);
        part_m = reinterpret_cast<float *>(w + L.o_bytes);
        part_l = reinterpret_cast<float *>(w + L.o_bytes + L.ml_bytes);
        w += L.o_bytes + 2 * L.ml_bytes;
        xpart_o = reinterpret_cast<float *>(w);
        xpart_m = reinterpret_cast<float *>(w + L.xo_bytes);
        xpart_l = reinterpret_cast<float *>(w + L.xo_bytes + L.xml_bytes);
        cut_tab = reinterpret_cast<int4 *>(w + L.xo_bytes + 2 * L.xml_bytes);
    }

    const int box_rows = gcd_int(decode_tile_keys(1, head_dim), block_size);
    CUtensorMap kmap, vmap;
    st = make_code_map(&kmap, key_codes, head_dim, num_kv_heads, num_blocks * block_size,
                       box_rows);
    if (st != PA_OK) return st;
    st = make_code_map(&vmap, value_codes, head_dim, num_kv_heads, num_blocks * block_size,
                       box_rows);
    if (st != PA_OK) return st;

    DecodeArgs a;
    memset(&a, 0, sizeof a);
    a.out = out;
    a.q = q;
    a.cu_seqlens_q = cu_seqlens_q;
    a.seq_lens_k = seq_lens_k;
    a.block_tables = block_tables;
    a.max_blocks_per_seq = max_blocks_per_seq;
    a.num_seqs = num_seqs;
    a.num_q_heads = num_q_heads;
    a.num_kv_heads = num_kv_heads;
    a.block_size = block_size;
    a.qscale = scale * kLog2e;
    a.sinks = sinks;
    a.causal = causal ? 1 : 0;
    a.partition_size = P;
    a.max_parts = max_parts;
    a.part_o = part_o;
    a.part_m = part_m;
    a.part_l = part_l;
    a.total_q = total_q;
    a.err = dev.err;
    a.box_rows = box_rows;
    a.k_scales = key_scales;
    a.v_scales = value_scales;
    auto launch = [&](dim3 grid) -> cudaError_t {
        return head_dim == 128 ? launch_decode_fp8kv_d128(group, kmap, vmap, a, grid, s)
                               : launch_decode_fp8kv_d256(group, kmap, vmap, a, grid, s);
    };
    // single-query rows: the persistent tensor-core kernel, one CTA per SM
    // sharing the batch's (request, KV head, partition) items
    const int dbox = gcd_int(gcd_int(128, block_size), P > 0 ? P : 128);
    CUtensorMap qmap_d, kmap_d, vmap_d;
    st = make_query_map(&qmap_d, q, head_dim, num_q_heads, total_q, group, 1);
    if (st != PA_OK) return st;
    st = make_code_map(&kmap_d, key_codes, head_dim, num_kv_heads, num_blocks * block_size, dbox);
    if (st != PA_OK) return st;
    st = make_code_map(&vmap_d, value_codes, head_dim, num_kv_heads, num_blocks * block_size,
                       dbox);
    if (st != PA_OK) return st;
    DecodeTcArgs da;
    memset(&da, 0, sizeof da);
    da.out = out;
    da.cu_seqlens_q = cu_seqlens_q;
    da.seq_lens_k = seq_lens_k;
    da.block_tables = block_tables;
    da.max_blocks_per_seq = max_blocks_per_seq;
    da.num_seqs = num_seqs;
    da.num_q_heads = num_q_heads;
    da.num_kv_heads = num_kv_heads;
    da.block_size = block_size;
    da.qscale = scale * kLog2e;
    da.sinks = sinks;
    da.partition_size = P;
    da.max_parts = max_parts;
    da.part_o = part_o;
    da.part_m = part_m;
    da.part_l = part_l;
    da.box_rows = dbox;
    da.err = dev.err;
    da.after_scatter = 0;
    da.xpart_o = xpart_o;
    da.xpart_m = xpart_m;
    da.xpart_l = xpart_l;
    da.cut_tab = cut_tab;
    da.k_scales = key_scales;
    da.v_scales = value_scales;
    da.num_blocks = num_blocks;
    // an item costs ~5 tiles beyond its keys here (Q split, deferred output,
    // the roles' item changes; per-CTA times fitted on the GQA decode batch)
    da.item_cost = 25;
    const int grid = plan.decode_grid[0];
    record_plan(plan);
    cudaError_t ce =
        head_dim == 128 ? launch_decode_tc_fp8_d128(group, qmap_d, kmap_d, vmap_d, da, grid, s)
                        : launch_decode_tc_fp8_d256(group, qmap_d, kmap_d, vmap_d, da, grid, s);
    if (ce != cudaSuccess) return cuda_fail(ce, "paged_decode_tc (quantised) launch");
    // rows of multi-query requests: one CTA per (row, KV head)
    if (max_seqlen_q > 1) {
        a.mode = 1;
        ce = launch(dim3((unsigned)plan.mq_grid[0], plan.mq_grid[1], 1));
        if (ce != cudaSuccess) return cuda_fail(ce, "paged_rows (quantised) launch");
    }
    if (P > 0) {
        ReduceArgs ra;
        memset(&ra, 0, sizeof ra);
        ra.out = out;
        ra.part_o = part_o;
        ra.part_m = part_m;
        ra.part_l = part_l;
        ra.cu_seqlens_q = cu_seqlens_q;
        ra.seq_lens_k = seq_lens_k;
        ra.num_seqs = num_seqs;
        ra.max_parts = max_parts;
        ra.partition_size = P;
        ra.num_q_heads = num_q_heads;
        ra.sinks = sinks;
        ra.meta_before_wait = 1;   // the kernels before it write only out / partials
        ra.xpart_o = xpart_o;
        ra.xpart_m = xpart_m;
        ra.xpart_l = xpart_l;
        ra.cut_tab = cut_tab;
        ra.ncut = grid;
        ra.group = group;
        ce = launch_reduce(2, head_dim, ra, s);
        if (ce != cudaSuccess) return cuda_fail(ce, "split_reduce launch");
    }
    return PA_OK;
}
