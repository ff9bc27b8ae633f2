/*
 * pa.h -- C ABI of the paged varlen attention library (libpa.so, sm_103a).
 *
 * Three calls make up the hot path of one model step's attention layer:
 *
 *   pa_reshape_and_cache   write this step's K/V rows into their cache pages
 *   pa_varlen_attention    attention for packed query rows over paged K/V
 *   pa_split_kv_reduce     merge split-KV partial results
 *
 * and pa_scatter_and_attend runs the first two as one call (the decode kernel
 * overlapping the scatter).
 *
 * Sources: "vllm-metal ... Paged Attention kernels" (kwkr.cn) -- section
 * "What is Paged Attention" (pages + block tables), the kernel table
 * (reshape_and_cache, sinks), the GQA decode section (query heads sharing a KV
 * head) and trick 4 (split-KV partitions with a shared log2-space reduce);
 * "vLLM releases vllm-metal" (aisignalhub.me), section "packed queries and
 * paged KV" (packed [total_q, H, D] queries, cu_seqlens boundaries, one mixed
 * step of decode, speculative-verify and prefill rows).
 *
 * Conventions for every call
 *  - Pointers marked "device" must point to memory of the current CUDA
 *    device; the caller owns all of it.  The library never allocates device
 *    memory and keeps no pointer after a call returns.
 *  - `stream` is a cudaStream_t passed as void* (NULL = the legacy default
 *    stream).  Every call is asynchronous on that stream; host-side argument
 *    checks happen before any launch, and a failed check launches nothing.
 *  - Element type: q, caches and out share one pa_dtype.  Metadata is int32,
 *    except slot_mapping (int64).  Sinks and split partials are float32.
 *  - Tensors are dense, row-major (last index fastest), 16-byte aligned.
 *  - No exception crosses the ABI; calls are thread-safe.
 *  - On PA_ERR_CUDA, pa_last_error_string() describes the CUDA error.
 */
#ifndef PA_H_
#define PA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum pa_status {
    PA_OK = 0,
    PA_ERR_INVALID_ARG = 1,  /* null pointer, bad size, misaligned pointer */
    PA_ERR_UNSUPPORTED = 2,  /* shape outside the compiled kernels' range */
    PA_ERR_WORKSPACE = 3,    /* workspace missing or smaller than required */
    PA_ERR_CUDA = 4          /* a CUDA call or kernel launch failed */
} pa_status;

typedef enum pa_dtype { PA_F32 = 0, PA_BF16 = 1 } pa_dtype;

/* Human-readable name of a status code (static string). */
const char *pa_status_string(pa_status status);

/* Description of the last CUDA error seen by this thread (static buffer). */
const char *pa_last_error_string(void);

/* Build identification: target architecture and library version. */
const char *pa_build_info(void);

/*
 * Launch plans (the kwkr.cn hands-on section's dispatch diagnostics: which
 * kernel served the call and with which partition size).
 *
 * pa_describe_plan -- host only, no device call: writes into buf (buf_len
 * bytes, NUL-terminated, truncated if short) the launches that
 * pa_varlen_attention (quantised = 0) or pa_varlen_attention_fp8kv
 * (quantised = 1) makes for these sizes on a GPU of sm_count SMs, as one
 * line of key=value pairs: dtype, cache (plain / e4m3), head_dim, group,
 * partition (split-KV partition used, 0 = none), max_parts, decode_kernel
 * and decode_grid (single-query rows), mq_kernel and mq_grid (rows of
 * multi-query requests; none when max_seqlen_q <= 1), reduce and
 * reduce_grid, workspace (bytes the call needs; 0 = none).  Returns
 * PA_ERR_INVALID_ARG for a null buffer or impossible sizes.
 *
 * pa_last_plan -- the same line for the last attention call this thread
 * launched ("none" before the first); static per-thread buffer.  With the
 * environment variable PA_DEBUG set (not "0") every attention call also
 * prints its line to stderr, prefixed "pa: ".
 */
pa_status pa_describe_plan(int num_seqs, int64_t total_q, int max_seqlen_q, int max_seqlen_k,
                           int num_q_heads, int num_kv_heads, int head_dim, int partition_size,
                           pa_dtype dtype, int quantised, int sm_count, char *buf,
                           size_t buf_len);
const char *pa_last_plan(void);

/*
 * pa_reshape_and_cache -- scatter this step's K/V rows into the page pool.
 * (kwkr.cn kernel table: reshape_and_cache writes projected K/V into the
 * paged cache.)
 *
 *   key, value     device, [num_tokens, H_kv, D] rows; token t starts at
 *                  element t * kv_token_stride (>= H_kv * D), so K and V may
 *                  be views into a fused QKV projection.
 *   key_cache,     device, [num_blocks, block_size, H_kv, D], contiguous.
 *   value_cache
 *   slot_mapping   device, [num_tokens] int64: slot = page * block_size +
 *                  offset.  A negative slot marks a padding token: skipped.
 *                  A slot >= num_blocks * block_size is skipped as well (it
 *                  cannot be checked on the host without a device sync).
 *
 * Postcondition: cache[slot / bs][slot % bs][h][:] == key[t][h][:] bit for
 * bit for every token with a valid slot; every other slot keeps its bytes.
 * Two tokens with the same slot: one of them wins (unspecified which).
 * Errors: PA_ERR_INVALID_ARG (null pointer with num_tokens > 0, sizes <= 0,
 * kv_token_stride < H_kv * D), PA_ERR_CUDA (launch failure).
 */
pa_status pa_reshape_and_cache(const void *key, const void *value, int64_t kv_token_stride,
                               void *key_cache, void *value_cache,
                               const int64_t *slot_mapping, int64_t num_tokens,
                               int num_kv_heads, int head_dim, int block_size,
                               int64_t num_blocks, pa_dtype dtype, void *stream);

/*
 * pa_varlen_attention -- attention for packed query rows over paged K/V.
 * (aisignalhub.me "packed queries and paged KV"; kwkr.cn "What is Paged
 * Attention", GQA decode section, trick 4.)
 *
 * Request r owns query rows cu_seqlens_q[r] .. cu_seqlens_q[r+1]-1 (n rows)
 * and N = seq_lens_k[r] keys; key j lives in page block_tables[r][j / bs],
 * slot j % bs.  N counts this step's tokens, which must already be in the
 * cache (pa_reshape_and_cache first).  Query head h reads KV head
 * h / (H_q / H_kv).  Row i of the request sees key j iff j < N and, when
 * causal, j <= N - n + i (the query rows are the last n positions).
 *   out[row][h] = sum_j e^{s_j - M} V[j] / (sum_j e^{s_j - M} + e^{sink_h - M})
 * with s_j = scale * <q[row][h], K[j]>, the sink term only when sinks != NULL
 * (a logit with no value vector, counted once), and zeros for a row that
 * sees no key.
 *
 *   out            device, [total_q, H_q, D] (written entirely)
 *   q              device, [total_q, H_q, D]
 *   key_cache,     device, [num_blocks, block_size, H_kv, D]
 *   value_cache
 *   cu_seqlens_q   device, [num_seqs + 1] int32, nondecreasing, [0] = 0,
 *                  [num_seqs] = total_q
 *   seq_lens_k     device, [num_seqs] int32, 0 <= N <= max_seqlen_k and
 *                  N <= max_blocks_per_seq * block_size
 *   block_tables   device, [num_seqs, max_blocks_per_seq] int32; entries past
 *                  a request's last page are never read.  Page ids outside
 *                  [0, num_blocks) read as zeros (no fault).
 *   max_seqlen_q,  host upper bounds of n and N (no device sync is made).
 *   max_seqlen_k
 *   sinks          device, [H_q] float32, or NULL for no sinks
 *   partition_size 0 = chosen by the library from the SM count, -1 = never
 *                  split, or a positive multiple of 32 (e.g. 256 or 512):
 *                  the split-KV partition length for single-query requests.
 *   workspace      device scratch of at least
 *                  pa_varlen_attention_workspace_size(...) bytes (NULL only
 *                  when that size is 0).  Contents need no initialisation.
 *
 * Supported: dtype F32 or BF16; head_dim 64, 128 or 256; H_q a multiple of
 * H_kv with H_q / H_kv <= 8; block_size a multiple of 8 (<= 1024); num_seqs
 * <= 65535; with split-KV, at most 12288 partitions per request
 * (ceil(max_seqlen_k / partition_size)).  Single-query rows (decode) run on a bandwidth kernel with
 * split-KV; multi-query rows (speculative verify, prefill) run on the
 * multi-row kernel.
 * Errors: PA_ERR_INVALID_ARG, PA_ERR_UNSUPPORTED, PA_ERR_WORKSPACE,
 * PA_ERR_CUDA.
 */
pa_status pa_varlen_attention(void *out, const void *q, const void *key_cache,
                              const void *value_cache, const int32_t *cu_seqlens_q,
                              const int32_t *seq_lens_k, const int32_t *block_tables,
                              int max_blocks_per_seq, int num_seqs, int64_t total_q,
                              int max_seqlen_q, int max_seqlen_k, int num_q_heads,
                              int num_kv_heads, int head_dim, int block_size,
                              int64_t num_blocks, float scale, const float *sinks, int causal,
                              int partition_size, void *workspace, size_t workspace_bytes,
                              pa_dtype dtype, void *stream);

/*
 * Bytes of workspace pa_varlen_attention needs for these sizes (host only;
 * no device call).  With partition_size 0 the bound covers every partition
 * length the library may choose.  Returns 0 when no split is possible.
 */
size_t pa_varlen_attention_workspace_size(int num_seqs, int max_seqlen_k, int num_q_heads,
                                          int head_dim, int partition_size);

/*
 * Partition length pa_varlen_attention uses for these sizes on a GPU with
 * `sm_count` SMs (host only): 0 = no split, else 1024, 512 or 256 (or the
 * forced value).  The library calls this with the current device's SM count.
 */
int pa_choose_partition_size(int num_seqs, int num_kv_heads, int max_seqlen_k,
                             int partition_size, int sm_count);

/*
 * pa_scatter_and_attend -- one model step in one call: pa_reshape_and_cache of
 * this step's K/V rows, then pa_varlen_attention.  (kwkr.cn kernel table: the
 * scatter runs before the attention kernel that reads the new rows.)
 *
 *   key, value, kv_token_stride, slot_mapping, num_tokens: as for
 *       pa_reshape_and_cache, with num_tokens == total_q (token t carries
 *       query row t's K and V: one step's packed tokens).
 *   every other argument: as for pa_varlen_attention (key_cache and
 *       value_cache are written).
 *
 * Result: exactly the two calls in order.  The kernels overlap: with bf16
 * caches at head_dim 128 or 256 the decode kernel is launched while the
 * scatter runs (programmatic dependent launch) and sets up its work plan,
 * page ids and pipeline meanwhile; only its K/V loads wait for the scatter.
 * Errors: those of both calls; PA_ERR_INVALID_ARG if num_tokens != total_q.
 */
pa_status pa_scatter_and_attend(const void *key, const void *value, int64_t kv_token_stride,
                                const int64_t *slot_mapping, int64_t num_tokens, void *out,
                                const void *q, void *key_cache, void *value_cache,
                                const int32_t *cu_seqlens_q, const int32_t *seq_lens_k,
                                const int32_t *block_tables, int max_blocks_per_seq, int num_seqs,
                                int64_t total_q, int max_seqlen_q, int max_seqlen_k,
                                int num_q_heads, int num_kv_heads, int head_dim, int block_size,
                                int64_t num_blocks, float scale, const float *sinks, int causal,
                                int partition_size, void *workspace, size_t workspace_bytes,
                                pa_dtype dtype, void *stream);

/*
 * The quantised KV cache (the layered-architecture page, lqnn.cn section 5,
 * lists TurboQuant helpers for the KV cache without a format; this library's
 * reading): each token's K row and V row of one KV head is stored as D 8-bit
 * floats E4M3 (1 sign bit, 4 exponent bits with bias 7, 3 mantissa bits, no
 * infinity, largest 448) plus one float32 scale:
 *   amax  = max_d |x_d|,  inv = 448 / amax  (float32 division),
 *   code  = E4M3(x_d * inv)  (float32 product, round to nearest even,
 *                             saturating at 448),
 *   scale = amax / 448  (float32 division); a row of zeros: codes 0, scale 0.
 * The row stands for value(code_d) * scale.  Layouts: codes
 * [num_blocks, block_size, H_kv, D] uint8 (the bf16 cache's layout, one byte
 * per element), scales [num_blocks, block_size, H_kv] float32.  head_dim 128
 * or 256.
 *
 * pa_reshape_and_cache_fp8 -- reshape_and_cache into the quantised cache: for
 * each token t with slot s = slot_mapping[t] >= 0 (and < num_blocks *
 * block_size; others are skipped), quantises key[t] and value[t] ([H_kv, D]
 * rows, bf16 or float32 per `dtype`, token stride kv_token_stride elements)
 * into the codes and scales of slot s.  Key and value rows start on 4-element
 * boundaries; codes and scales are 4-byte aligned.  Returns PA_OK,
 * PA_ERR_INVALID_ARG, PA_ERR_UNSUPPORTED (head_dim), PA_ERR_CUDA.
 */
pa_status pa_reshape_and_cache_fp8(const void *key, const void *value, int64_t kv_token_stride,
                                   void *key_codes, void *value_codes, float *key_scales,
                                   float *value_scales, const int64_t *slot_mapping,
                                   int64_t num_tokens, int num_kv_heads, int head_dim,
                                   int block_size, int64_t num_blocks, pa_dtype dtype,
                                   void *stream);

/*
 * pa_varlen_attention_fp8kv -- pa_varlen_attention over the quantised cache:
 * the same packed rows, masking, sinks, split-KV plan, workspace (sized by
 * pa_varlen_attention_workspace_size) and result, with every key and value
 * row taken as value(code) * scale.  q and out are bf16 (`dtype` must be
 * PA_BF16).  Single-query rows run on the tensor cores (a persistent kernel:
 * QK^T as an E4M3 MMA on the codes with the queries split exactly into two
 * E4M3 parts, PV in f16 from V codes converted exactly, fp32 accumulation;
 * split over partitions and merged by the shared reduce); multi-query rows on
 * the CUDA cores in float32, one CTA per row and KV head.  Returns the
 * statuses of pa_varlen_attention, and PA_ERR_UNSUPPORTED for another dtype
 * or head_dim.
 */
pa_status pa_varlen_attention_fp8kv(
    void *out, const void *q, const void *key_codes, const void *value_codes,
    const float *key_scales, const float *value_scales, const int32_t *cu_seqlens_q,
    const int32_t *seq_lens_k, const int32_t *block_tables, int max_blocks_per_seq, int num_seqs,
    int64_t total_q, int max_seqlen_q, int max_seqlen_k, int num_q_heads, int num_kv_heads,
    int head_dim, int block_size, int64_t num_blocks, float scale, const float *sinks, int causal,
    int partition_size, void *workspace, size_t workspace_bytes, pa_dtype dtype, void *stream);

/*
 * pa_split_kv_reduce -- the shared reduce of split-KV partials.
 * (kwkr.cn trick 4: partials are a log2-space (max, exp-sum) pair plus a
 * normalised partial output, merged by one shared reduce kernel.)
 *
 * For every request r with exactly one query row and every head h, with
 * nparts = ceil(seq_lens_k[r] / partition_size):
 *   M   = max(max_p m_p, sink_h * log2(e))       (sink only if sinks != NULL)
 *   w_p = l_p * 2^(m_p - M)
 *   out[cu_seqlens_q[r]][h] = sum_p w_p o_p / (sum_p w_p + 2^(sink_h log2 e - M))
 * and zeros when nparts == 0.  Rows of other requests are not touched.
 *
 *   part_out  device float32 [num_seqs, max_parts, H_q, D]: o_p (normalised)
 *   part_max  device float32 [num_seqs, max_parts, H_q]: m_p, log2 domain
 *             (a reference for the partition's scale * <q, k> * log2(e):
 *             their max, or a value at most 8 below it, so that every
 *             2^(t_j - m_p) stays finite)
 *   part_sum  device float32 [num_seqs, max_parts, H_q]: l_p = sum of
 *             2^(t_j - m_p) over the partition
 *   out       device [total_q, H_q, D] in `dtype`
 * Errors: PA_ERR_INVALID_ARG, PA_ERR_UNSUPPORTED (head_dim, or max_parts >
 * 12288: the weights live in shared memory), PA_ERR_CUDA.
 */
pa_status pa_split_kv_reduce(void *out, const float *part_out, const float *part_max,
                             const float *part_sum, const int32_t *cu_seqlens_q,
                             const int32_t *seq_lens_k, int num_seqs, int max_parts,
                             int partition_size, int num_q_heads, int head_dim,
                             const float *sinks, pa_dtype dtype, void *stream);

/* Bytes of the fixed device scratch behind pa_varlen_attention_static_scratch. */
#define PA_STATIC_SCRATCH_BYTES (16u << 20)

/*
 * pa_varlen_attention_static_scratch -- pa_varlen_attention for callers that
 * cannot allocate device memory.  (The pages have no counterpart: it exists
 * for callers such as a host framework that owns every device allocation, a
 * serving loop that must never stall or synchronise on cudaMalloc/cudaFree,
 * or a plugin with no allocator at all; they cannot pass a workspace.)
 *
 * Same arguments and results as pa_varlen_attention, minus the workspace.
 * The split-KV partials live in a scratch array of PA_STATIC_SCRATCH_BYTES
 * (16 MiB) compiled into the library as device memory: every GPU that loads
 * the library holds it until the process exits.  The call itself allocates
 * nothing (no cudaMalloc, no cudaFree, no allocating library routine).
 *  - The first call on a device looks up the array's device address
 *    (cudaGetSymbolAddress) and caches it; make that first call before any
 *    stream capture.
 *  - A call whose split plan needs more than PA_STATIC_SCRATCH_BYTES returns
 *    PA_ERR_WORKSPACE without launching anything (pa_last_error_string() says
 *    how many bytes it needed); use pa_varlen_attention with a workspace, a
 *    longer partition_size, or partition_size = -1 instead.
 *  - All calls share the one array and it keeps the last call's contents.
 *    Nothing in it needs to start at zero (a call reads only partials it has
 *    written), but calls that overlap on the GPU -- on two streams, or from
 *    two threads -- race on it: order them on one stream.
 */
pa_status pa_varlen_attention_static_scratch(
    void *out, const void *q, const void *key_cache, const void *value_cache,
    const int32_t *cu_seqlens_q, const int32_t *seq_lens_k, const int32_t *block_tables,
    int max_blocks_per_seq, int num_seqs, int64_t total_q, int max_seqlen_q, int max_seqlen_k,
    int num_q_heads, int num_kv_heads, int head_dim, int block_size, int64_t num_blocks,
    float scale, const float *sinks, int causal, int partition_size, pa_dtype dtype,
    void *stream);

/*
 * Reads and clears the library's device-side error word for the current
 * device (synchronises the device).  Nonzero means a kernel gave up: 1 = a
 * bounded wait ran out (a pipeline barrier that never completed), 3 = the
 * multi-query kernel met a work unit outside the batch (an inconsistent plan)
 * and skipped it; the output is then unreliable.  Returns PA_OK, or
 * PA_ERR_CUDA if the read failed.
 */
pa_status pa_device_error(int *code);

/*
 * pa_test_expire_next_wait -- test hook of the failure path; not for
 * production use.  (The pages have no counterpart: it exists so that a test
 * can watch a bounded wait run out.)  The next attention call of this process
 * that launches the multi-query (tensor-core) kernel makes each of its CTAs
 * skip the K loads of its first key tile.  The MMA warp's bounded wait for
 * that tile gives up after about one second of GPU time; the kernel then sets
 * the device error word, lets every other wait return at once, drains its
 * copies and tensor-core work in flight and returns, without a trap or fault.
 * Its output is unreliable; pa_device_error() reports a nonzero code, and the
 * calls after it run normally.
 */
void pa_test_expire_next_wait(void);

#ifdef __cplusplus
}
#endif

#endif /* PA_H_ */
