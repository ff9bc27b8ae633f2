/*
 * pa_oracle.c -- TEST INFRASTRUCTURE, NOT THE PRODUCT.
 *
 * A plain, slow, fp64 CPU definition of what unified paged varlen attention
 * computes.  Only the test suite, the package smoke check and the benchmark's
 * CPU-baseline leg may load this library; the CUDA path never calls it and
 * shares no code, header or table with it.
 *
 * Sources (web pages on the vllm-metal plugin):
 *  - "vllm-metal ... Paged Attention kernels" (kwkr.cn), section "What is Paged
 *    Attention": K/V live in fixed-size pages; block_tables map a request's
 *    logical block to a physical page.
 *  - same page, kernel table: reshape_and_cache scatters projected K/V rows
 *    into the paged cache; the decode kernel supports attention sinks.
 *  - same page, GQA decode section: 4-8 query heads share one KV head.
 *  - same page, trick 4 (split-KV): the KV range is cut into 256/512-token
 *    partitions whose partials are a log2-space (max, exp-sum) pair plus a
 *    normalised partial output, merged by a shared reduce.
 *  - "vLLM releases vllm-metal" (aisignalhub.me), section "packed queries and
 *    paged KV": every scheduled query token is packed into [total_q, H, D] and
 *    cu_seqlens marks request boundaries.
 *  - "vllm-metal unified memory" (pptc.cn), section 3 (lazy KV allocation):
 *    the kernel masks every slot past the sequence length, so unwritten memory
 *    never reaches the output.
 *
 * Readings where the pages are silent (each also listed in the design notes):
 *  - causal rows are bottom-right aligned: row i of a request with n query rows
 *    and N keys sees keys j <= N - n + i;
 *  - query head h uses KV head h / (H_q / H_kv);
 *  - a sink is a logit in the post-scale domain with no value vector, added
 *    once to the softmax denominator;
 *  - a row that sees no key outputs zeros;
 *  - a negative slot in slot_mapping is a padding token and is skipped.
 *
 * dtype codes: 0 = float32, 1 = bfloat16 (stored as uint16 bit patterns),
 * 2 = float64 (a dequantised 8-bit cache, see the quantised KV section).
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_F32 0
#define ORACLE_BF16 1
#define ORACLE_F64 2

static double elem(const void *base, int64_t idx, int dtype) {
    if (dtype == ORACLE_F32) return (double)((const float *)base)[idx];
    if (dtype == ORACLE_F64) return ((const double *)base)[idx];
    /* a bf16 value is the top half of the float32 with the same bits */
    uint32_t u = (uint32_t)((const uint16_t *)base)[idx] << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* ------------------------------------------------------------------------- */
/* reshape_and_cache: a plain byte copy of each token's [H_kv, D] row into the */
/* slot slot_mapping[t] = page * block_size + offset.                          */
/* Returns 0, or -1 if a slot lies outside the pool.                          */
/* ------------------------------------------------------------------------- */
int oracle_reshape_and_cache(const void *key, const void *value, int64_t kv_token_stride,
                             void *key_cache, void *value_cache, const int64_t *slot_mapping,
                             int64_t num_tokens, int num_kv_heads, int head_dim, int block_size,
                             int64_t num_blocks, int elem_bytes) {
    const int64_t row_elems = (int64_t)num_kv_heads * head_dim;
    const int64_t row_bytes = row_elems * elem_bytes;
    for (int64_t t = 0; t < num_tokens; ++t) {
        int64_t slot = slot_mapping[t];
        if (slot < 0) continue; /* padding token */
        if (slot >= num_blocks * block_size) return -1;
        int64_t page = slot / block_size, off = slot % block_size;
        int64_t dst = (page * block_size + off) * row_bytes;
        int64_t src = t * kv_token_stride * elem_bytes;
        memcpy((char *)key_cache + dst, (const char *)key + src, (size_t)row_bytes);
        memcpy((char *)value_cache + dst, (const char *)value + src, (size_t)row_bytes);
    }
    return 0;
}

/* ------------------------------------------------------------------------- */
/* Attention, one (query row, query head) at a time.                          */
/* ------------------------------------------------------------------------- */
typedef struct {
    double *out;            /* [n_sel, H_q, D] */
    const int64_t *rows;    /* [n_sel] global query rows */
    int64_t n_sel;
    const void *q, *key_cache, *value_cache;
    int dtype;              /* of q */
    int kv_dtype;           /* of the caches */
    const int32_t *cu_seqlens_q, *seq_lens_k, *block_tables;
    int max_blocks_per_seq, num_seqs;
    int num_q_heads, num_kv_heads, head_dim, block_size;
    int64_t num_blocks;
    double scale;
    const double *sinks;    /* [H_q] or NULL */
    int causal;
    int nthreads, tid;
    int error;
} attn_job;

/* Request that owns global query row `row` (plain linear scan). */
static int request_of_row(const int32_t *cu, int num_seqs, int64_t row) {
    for (int r = 0; r < num_seqs; ++r)
        if (row >= cu[r] && row < cu[r + 1]) return r;
    return -1;
}

/* Gathers key/value row j of request r for kv head g: the page is
 * block_tables[r][j / block_size], the slot inside it j % block_size. */
static int64_t kv_offset(const attn_job *a, int r, int64_t j, int g) {
    int32_t page = a->block_tables[(int64_t)r * a->max_blocks_per_seq + j / a->block_size];
    if (page < 0 || page >= a->num_blocks) return -1;
    int64_t slot = (int64_t)page * a->block_size + j % a->block_size;
    return (slot * a->num_kv_heads + g) * a->head_dim;
}

static int attend_one(const attn_job *a, int64_t sel, int h, double *s_buf) {
    const int64_t row = a->rows[sel];
    const int D = a->head_dim;
    double *o = a->out + (sel * a->num_q_heads + h) * D;
    for (int d = 0; d < D; ++d) o[d] = 0.0;

    int r = request_of_row(a->cu_seqlens_q, a->num_seqs, row);
    if (r < 0) return -2;
    const int64_t n = a->cu_seqlens_q[r + 1] - a->cu_seqlens_q[r];
    const int64_t i = row - a->cu_seqlens_q[r];
    const int64_t N = a->seq_lens_k[r];
    if (N > (int64_t)a->max_blocks_per_seq * a->block_size) return -3;
    const int g = h / (a->num_q_heads / a->num_kv_heads);

    /* visible keys: j < N and, if causal, j <= N - n + i */
    int64_t last = N - 1;
    if (a->causal && N - n + i < last) last = N - n + i;
    const int64_t nvis = last + 1 > 0 ? last + 1 : 0;

    const int64_t qoff = (row * a->num_q_heads + h) * D;
    double m = -INFINITY;
    for (int64_t j = 0; j < nvis; ++j) {
        int64_t ko = kv_offset(a, r, j, g);
        if (ko < 0) return -1;
        double dot = 0.0;
        for (int d = 0; d < D; ++d)
            dot += elem(a->q, qoff + d, a->dtype) * elem(a->key_cache, ko + d, a->kv_dtype);
        s_buf[j] = a->scale * dot;
        if (s_buf[j] > m) m = s_buf[j];
    }
    if (nvis == 0) return 0; /* no visible key: zeros, with or without a sink */
    const double sink = a->sinks ? a->sinks[h] : -INFINITY;
    if (sink > m) m = sink;

    double den = 0.0;
    for (int64_t j = 0; j < nvis; ++j) {
        double p = exp(s_buf[j] - m);
        den += p;
        int64_t vo = kv_offset(a, r, j, g);
        for (int d = 0; d < D; ++d) o[d] += p * elem(a->value_cache, vo + d, a->kv_dtype);
    }
    if (a->sinks) den += exp(sink - m);
    for (int d = 0; d < D; ++d) o[d] /= den;
    return 0;
}

static void *attn_worker(void *arg) {
    attn_job *a = (attn_job *)arg;
    int64_t max_n = 1;
    for (int r = 0; r < a->num_seqs; ++r)
        if (a->seq_lens_k[r] > max_n) max_n = a->seq_lens_k[r];
    double *s_buf = (double *)malloc(sizeof(double) * (size_t)max_n);
    if (!s_buf) { a->error = -4; return NULL; }
    const int64_t units = a->n_sel * a->num_q_heads;
    for (int64_t u = a->tid; u < units; u += a->nthreads) {
        int rc = attend_one(a, u / a->num_q_heads, (int)(u % a->num_q_heads), s_buf);
        if (rc && !a->error) a->error = rc;
    }
    free(s_buf);
    return NULL;
}

/*
 * out[sel][h][:] = softmax over the visible keys of request r(row) of
 * scale * <q[row][h], K_r[j]>, applied to V_r, with the sink logit (if any)
 * added once to the denominator.  Computes the rows listed in `rows` only.
 * Returns 0; -1 bad page id; -2 row outside cu_seqlens_q; -3 seq_len larger
 * than the block table; -4 out of memory.
 */
int oracle_paged_attention_kv(double *out, const int64_t *rows, int64_t n_sel, const void *q,
                              const void *key_cache, const void *value_cache, int dtype,
                              int kv_dtype, const int32_t *cu_seqlens_q,
                              const int32_t *seq_lens_k, const int32_t *block_tables,
                              int max_blocks_per_seq, int num_seqs, int num_q_heads,
                              int num_kv_heads, int head_dim, int block_size, int64_t num_blocks,
                              double scale, const double *sinks, int causal, int nthreads) {
    if (nthreads < 1) nthreads = 1;
    if (num_kv_heads <= 0 || num_q_heads % num_kv_heads) return -2;
    attn_job *jobs = (attn_job *)calloc((size_t)nthreads, sizeof(attn_job));
    pthread_t *th = (pthread_t *)calloc((size_t)nthreads, sizeof(pthread_t));
    if (!jobs || !th) { free(jobs); free(th); return -4; }
    for (int t = 0; t < nthreads; ++t) {
        attn_job *a = &jobs[t];
        a->out = out; a->rows = rows; a->n_sel = n_sel; a->q = q;
        a->key_cache = key_cache; a->value_cache = value_cache; a->dtype = dtype;
        a->kv_dtype = kv_dtype;
        a->cu_seqlens_q = cu_seqlens_q; a->seq_lens_k = seq_lens_k;
        a->block_tables = block_tables; a->max_blocks_per_seq = max_blocks_per_seq;
        a->num_seqs = num_seqs; a->num_q_heads = num_q_heads; a->num_kv_heads = num_kv_heads;
        a->head_dim = head_dim; a->block_size = block_size; a->num_blocks = num_blocks;
        a->scale = scale; a->sinks = sinks; a->causal = causal;
        a->nthreads = nthreads; a->tid = t; a->error = 0;
    }
    char *started = (char *)calloc((size_t)nthreads, 1);
    for (int t = 1; t < nthreads; ++t)
        started[t] = pthread_create(&th[t], NULL, attn_worker, &jobs[t]) == 0;
    attn_worker(&jobs[0]);
    for (int t = 1; t < nthreads; ++t) {
        if (started[t]) pthread_join(th[t], NULL);
        else attn_worker(&jobs[t]); /* could not start a thread: do its units here */
    }
    int rc = 0;
    for (int t = 0; t < nthreads; ++t)
        if (jobs[t].error && !rc) rc = jobs[t].error;
    free(started); free(jobs); free(th);
    return rc;
}

/* The same, with the caches in the dtype of q. */
int oracle_paged_attention(double *out, const int64_t *rows, int64_t n_sel, const void *q,
                           const void *key_cache, const void *value_cache, int dtype,
                           const int32_t *cu_seqlens_q, const int32_t *seq_lens_k,
                           const int32_t *block_tables, int max_blocks_per_seq, int num_seqs,
                           int num_q_heads, int num_kv_heads, int head_dim, int block_size,
                           int64_t num_blocks, double scale, const double *sinks, int causal,
                           int nthreads) {
    return oracle_paged_attention_kv(out, rows, n_sel, q, key_cache, value_cache, dtype, dtype,
                                     cu_seqlens_q, seq_lens_k, block_tables, max_blocks_per_seq,
                                     num_seqs, num_q_heads, num_kv_heads, head_dim, block_size,
                                     num_blocks, scale, sinks, causal, nthreads);
}

/* ------------------------------------------------------------------------- */
/* Split-KV, as the split-KV trick describes it, for single-query requests:   */
/* partition p covers keys [p*P, min(N, (p+1)*P)); its partial is the         */
/* log2-space max m_p of t_j = s_j * log2(e), the sum l_p of 2^(t_j - m_p),   */
/* and the normalised output o_p = sum_j 2^(t_j - m_p) v_j / l_p.  Partitions */
/* with no key are not produced.                                              */
/* Layout: part_o [S][max_parts][H_q][D], part_m / part_l [S][max_parts][H_q]. */
/* Requests whose query length is not 1 are skipped.                          */
/* ------------------------------------------------------------------------- */
int oracle_split_partials(double *part_o, double *part_m, double *part_l, int max_parts,
                          int partition_size, const void *q, const void *key_cache,
                          const void *value_cache, int dtype, const int32_t *cu_seqlens_q,
                          const int32_t *seq_lens_k, const int32_t *block_tables,
                          int max_blocks_per_seq, int num_seqs, int num_q_heads,
                          int num_kv_heads, int head_dim, int block_size, int64_t num_blocks,
                          double scale) {
    const double log2e = 1.0 / log(2.0);
    attn_job a;
    memset(&a, 0, sizeof a);
    a.key_cache = key_cache; a.value_cache = value_cache; a.dtype = dtype;
    a.block_tables = block_tables; a.max_blocks_per_seq = max_blocks_per_seq;
    a.num_kv_heads = num_kv_heads; a.head_dim = head_dim; a.block_size = block_size;
    a.num_blocks = num_blocks;
    const int D = head_dim, G = num_q_heads / num_kv_heads;
    for (int r = 0; r < num_seqs; ++r) {
        if (cu_seqlens_q[r + 1] - cu_seqlens_q[r] != 1) continue;
        const int64_t row = cu_seqlens_q[r];
        const int64_t N = seq_lens_k[r];
        const int64_t nparts = (N + partition_size - 1) / partition_size;
        if (nparts > max_parts) return -3;
        for (int h = 0; h < num_q_heads; ++h) {
            const int g = h / G;
            for (int64_t p = 0; p < nparts; ++p) {
                const int64_t j0 = p * partition_size;
                const int64_t j1 = (j0 + partition_size < N) ? j0 + partition_size : N;
                const int64_t slot = ((int64_t)r * max_parts + p) * num_q_heads + h;
                double *o = part_o + slot * D;
                double m = -INFINITY;
                for (int64_t j = j0; j < j1; ++j) {
                    int64_t ko = kv_offset(&a, r, j, g);
                    if (ko < 0) return -1;
                    double dot = 0.0;
                    for (int d = 0; d < D; ++d)
                        dot += elem(q, (row * num_q_heads + h) * D + d, dtype) *
                               elem(key_cache, ko + d, dtype);
                    double t2 = scale * dot * log2e;
                    if (t2 > m) m = t2;
                }
                double l = 0.0;
                for (int d = 0; d < D; ++d) o[d] = 0.0;
                for (int64_t j = j0; j < j1; ++j) {
                    int64_t ko = kv_offset(&a, r, j, g);
                    double dot = 0.0;
                    for (int d = 0; d < D; ++d)
                        dot += elem(q, (row * num_q_heads + h) * D + d, dtype) *
                               elem(key_cache, ko + d, dtype);
                    double w = exp2(scale * dot * log2e - m);
                    l += w;
                    for (int d = 0; d < D; ++d) o[d] += w * elem(value_cache, ko + d, dtype);
                }
                for (int d = 0; d < D; ++d) o[d] /= l;
                part_m[slot] = m;
                part_l[slot] = l;
            }
        }
    }
    return 0;
}

/*
 * The shared reduce: for each single-query request r and head h with
 * nparts = ceil(N / P) partitions,
 *   M   = max(max_p m_p, sink_h * log2(e))          (sink term only if sinks)
 *   w_p = l_p * 2^(m_p - M)
 *   out = sum_p w_p o_p / (sum_p w_p + 2^(sink_h * log2(e) - M))
 * Requests with no key produce zeros.  Partials are read as float32 (the
 * format the library writes) or float64, per `partials_f32`.
 * out: [S][H_q][D] (one row per single-query request, in request order).
 */
int oracle_split_combine(double *out, const void *part_o, const void *part_m,
                         const void *part_l, int partials_f32, int max_parts,
                         int partition_size, const int32_t *cu_seqlens_q,
                         const int32_t *seq_lens_k, int num_seqs, int num_q_heads, int head_dim,
                         const double *sinks) {
    const double log2e = 1.0 / log(2.0);
    const int D = head_dim;
#define PART(arr, i) (partials_f32 ? (double)((const float *)(arr))[i] : ((const double *)(arr))[i])
    for (int r = 0; r < num_seqs; ++r) {
        for (int h = 0; h < num_q_heads; ++h) {
            double *o = out + ((int64_t)r * num_q_heads + h) * D;
            for (int d = 0; d < D; ++d) o[d] = 0.0;
            if (cu_seqlens_q[r + 1] - cu_seqlens_q[r] != 1) continue;
            const int64_t N = seq_lens_k[r];
            const int64_t nparts = (N + partition_size - 1) / partition_size;
            if (nparts > max_parts) return -3;
            if (nparts == 0) continue;
            double M = sinks ? sinks[h] * log2e : -INFINITY;
            for (int64_t p = 0; p < nparts; ++p) {
                double m = PART(part_m, ((int64_t)r * max_parts + p) * num_q_heads + h);
                if (m > M) M = m;
            }
            double den = sinks ? exp2(sinks[h] * log2e - M) : 0.0;
            for (int64_t p = 0; p < nparts; ++p) {
                const int64_t slot = ((int64_t)r * max_parts + p) * num_q_heads + h;
                double w = PART(part_l, slot) * exp2(PART(part_m, slot) - M);
                den += w;
                for (int d = 0; d < D; ++d) o[d] += w * PART(part_o, slot * D + d);
            }
            for (int d = 0; d < D; ++d) o[d] /= den;
        }
    }
#undef PART
    return 0;
}

/* ------------------------------------------------------------------------- */
/* Quantised KV cache.  The layered-architecture page (lqnn.cn, section 5)   */
/* lists TurboQuant helpers for the KV cache without a format; the reading   */
/* taken here: each token's K (and V) row of one KV head is stored as 8-bit  */
/* floats E4M3 (1 sign, 4 exponent bits with bias 7, 3 mantissa bits, no    */
/* infinity, max 448) with one float32 scale per (token, KV head):          */
/*   amax  = max_d |x_d|                    (x as float32)                   */
/*   inv   = 448 / amax                     (float32 division)              */
/*   code  = E4M3(x_d * inv)                (float32 product, rounded to     */
/*                                           nearest even, saturated at 448) */
/*   scale = amax / 448                     (float32 division)              */
/* and a row of zeros stores codes 0 with scale 0.  The value a code stands  */
/* for is value(code) * scale, taken exactly (float64 here).                 */
/* ------------------------------------------------------------------------- */

/* The number an E4M3 code stands for (NaN for the codes S.1111.111). */
double oracle_e4m3_value(int code) {
    const int sign = (code >> 7) & 1, e = (code >> 3) & 15, m = code & 7;
    double v;
    if (e == 15 && m == 7) return NAN;
    if (e == 0) v = ldexp((double)m / 8.0, -6);                 /* subnormal */
    else v = ldexp(1.0 + (double)m / 8.0, e - 7);
    return sign ? -v : v;
}

/* Nearest E4M3 code to v (a float32), ties to the even code, |v| above the  */
/* largest finite value saturating to it, the sign kept (a negative value    */
/* too small for the smallest subnormal gives negative zero).  The finite    */
/* non-negative codes 0 .. 0x7E stand for increasing values, so the nearest  */
/* is one of the two codes around |v| (found by bisection).                  */
int oracle_e4m3_encode(float v) {
    const double x = fabs((double)v);
    int best;
    if (x >= 448.0) {
        best = 0x7E;
    } else {
        int lo = 0, hi = 0x7E;                /* value(lo) <= x < value(hi) */
        while (hi - lo > 1) {
            const int mid = (lo + hi) / 2;
            if (oracle_e4m3_value(mid) <= x) lo = mid;
            else hi = mid;
        }
        const double elo = x - oracle_e4m3_value(lo), ehi = oracle_e4m3_value(hi) - x;
        best = (elo < ehi || (elo == ehi && (lo & 1) == 0)) ? lo : hi;
    }
    return signbit(v) ? (best | 0x80) : best;
}

/* reshape_and_cache into the quantised cache: for each token t with slot   */
/* s = slot_mapping[t] >= 0, for each KV head h, the row of key (value) is   */
/* quantised into key_codes[(s * H_kv + h) * D + d] and key_scales[s * H_kv   */
/* + h].  Returns 0, or -1 if a slot lies outside the pool.                  */
int oracle_quantize_kv_fp8(const void *key, const void *value, int64_t kv_token_stride,
                           uint8_t *key_codes, uint8_t *value_codes, float *key_scales,
                           float *value_scales, const int64_t *slot_mapping, int64_t num_tokens,
                           int num_kv_heads, int head_dim, int block_size, int64_t num_blocks,
                           int in_dtype) {
    const int D = head_dim;
    for (int64_t t = 0; t < num_tokens; ++t) {
        const int64_t slot = slot_mapping[t];
        if (slot < 0) continue; /* padding token */
        if (slot >= num_blocks * block_size) return -1;
        for (int which = 0; which < 2; ++which) {
            const void *src = which ? value : key;
            uint8_t *codes = which ? value_codes : key_codes;
            float *scales = which ? value_scales : key_scales;
            for (int h = 0; h < num_kv_heads; ++h) {
                const int64_t in0 = t * kv_token_stride + (int64_t)h * D;
                const int64_t out0 = (slot * num_kv_heads + h) * D;
                float amax = 0.0f;
                for (int d = 0; d < D; ++d) {
                    const float x = (float)elem(src, in0 + d, in_dtype);
                    if (fabsf(x) > amax) amax = fabsf(x);
                }
                if (amax == 0.0f) {
                    for (int d = 0; d < D; ++d) codes[out0 + d] = 0;
                    scales[slot * num_kv_heads + h] = 0.0f;
                    continue;
                }
                const float inv = 448.0f / amax;
                for (int d = 0; d < D; ++d) {
                    const float x = (float)elem(src, in0 + d, in_dtype);
                    const float y = x * inv;
                    codes[out0 + d] = (uint8_t)oracle_e4m3_encode(y);
                }
                scales[slot * num_kv_heads + h] = amax / 448.0f;
            }
        }
    }
    return 0;
}
