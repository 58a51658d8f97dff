/*
 * fp64 CPU oracle for absorbed ("data-movement friendly") MLA decode over a
 * paged latent KV cache.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the
 * benchmark's CPU-baseline leg may load this library.  It shares no code,
 * header, table or constant with the CUDA library; it is written from the
 * MLA pages and is deliberately plain: no blocking, no fusion, no online
 * softmax.  Every bf16/e4m3 input is decoded to double exactly and all
 * arithmetic is double precision.
 *
 * What each function follows:
 *  - oracle_decode: the MQA of vllm/v1/attention/backends/mla/common.py,
 *    module docstring, "Data-Movement Friendly Approach": scores of the
 *    absorbed query [ql_nope | q_pe] (Lkv+R = 576 wide) against the shared
 *    latent rows [kv_c | k_pe], softmax, values = kv_c (Lkv = 512 wide), plus
 *    the natural-log LSE that "return_softmax_lse" hands to merge_attn_states
 *    ("Chunked Prefill" section).  The scale is the kernels' explicit
 *    `self.scale` argument (MLACommonImpl / AiterMLAImpl.forward_mqa), not an
 *    SDPA default.  Rows are fetched through the block table:
 *    cache[block_table[b, j / page], j % page, :] with cache shape
 *    (num_blocks, block_size, head_size) (get_kv_cache_shape).  With Sq query
 *    tokens per request, query token t sees keys [0, seq_len - Sq + 1 + t)
 *    (vllm.v1.attention.backends.mla.rocm_aiter_mla, AiterMLAImpl.forward_mqa,
 *    multi-token verify: verify token t sees the context plus the new tokens
 *    up to and including itself).
 *  - oracle_merge: merge_attn_states of two partial results over disjoint key
 *    sets (common.py docstring, "Chunked Prefill"); the formula is not
 *    printed on the pages, it is the softmax over the union of the key sets.
 *  - oracle_cache_write: concat_and_cache_mla (MLACommonImpl.forward;
 *    MLAAttention.forward -> do_kv_cache_update): row `slot` of the flattened
 *    cache receives [kv_c | k_pe]; negative slots are padding and skipped.
 *    For an fp8 cache the stored code is e4m3(x / kv_scale) with the divide
 *    done in float32; dequantisation multiplies by kv_scale
 *    (vllm.model_executor.layers.attention.mla_attention, calc_kv_scales:
 *    k_scale = abs-max / range).
 *  - oracle_gather_cache: gather_and_maybe_dequant_cache of the chunked
 *    prefill context path (common.py, MLACommonImpl._compute_prefill_context;
 *    the chunk metadata of MLACommonMetadataBuilder): request b's rows go to
 *    dst[cu_seq_lens[b] .. cu_seq_lens[b+1]), row j of them is the latent row
 *    at context position seq_starts[b] + j, fetched through the block table;
 *    a bf16 cache is copied, an e4m3 cache is dequantised to the model dtype
 *    as bf16(float32(code) * kv_scale) (float32 product, then round to
 *    nearest even).
 *  - e4m3: OCP FP8 E4M3 ("fn") -- 1 sign, 4 exponent (bias 7), 3 mantissa
 *    bits, no infinities, S.1111.111 is NaN, largest finite 448; encoding
 *    rounds to nearest, ties to even, and saturates finite overflow to +-448.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

#define ORC_LKV 512
#define ORC_DQK 576

enum { ORC_CACHE_BF16 = 0, ORC_CACHE_E4M3 = 1 };

/* ---------------------------------------------------------------- formats */

double oracle_bf16_to_f64(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;   /* bf16 is the top half of an IEEE binary32 */
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

double oracle_e4m3_to_f64(uint8_t c)
{
    int s = c >> 7, e = (c >> 3) & 15, m = c & 7;
    double mag;
    if (e == 15 && m == 7)
        return NAN;
    if (e == 0)
        mag = ldexp((double)m, -9);               /* subnormal: m/8 * 2^-6 */
    else
        mag = ldexp((double)(8 + m), e - 7 - 3);  /* (1 + m/8) * 2^(e-7) */
    return s ? -mag : mag;
}

static double round_half_even(double q)
{
    double f = floor(q), r = q - f;
    if (r > 0.5)
        return f + 1.0;
    if (r < 0.5)
        return f;
    return fmod(f, 2.0) == 0.0 ? f : f + 1.0;
}

uint8_t oracle_f32_to_e4m3(float xf)
{
    uint8_t sign = signbit(xf) ? 0x80 : 0x00;
    double a = fabs((double)xf);
    int e2, E, code;
    double quantum, n;
    if (isnan(xf))
        return sign | 0x7F;
    if (a >= 448.0)
        return sign | 0x7E;                      /* saturate finite overflow (and inf) */
    if (a < ldexp(1.0, -6)) {
        E = -6;                                  /* subnormal range: quantum 2^-9 */
    } else {
        frexp(a, &e2);                           /* a = f * 2^e2, f in [0.5, 1) */
        E = e2 - 1;                              /* floor(log2 a) */
    }
    quantum = ldexp(1.0, E - 3);                 /* 3 mantissa bits */
    n = round_half_even(a / quantum);            /* exact power-of-two scaling */
    if (E == -6 && n < 8.0) {
        code = (int)n;                           /* exponent field 0 */
    } else {
        if (n >= 16.0) {                         /* rounded up into the next binade */
            E += 1;
            n = 8.0;
        }
        code = ((E + 7) << 3) | ((int)n - 8);
    }
    if (code > 0x7E)
        code = 0x7E;
    return sign | (uint8_t)code;
}

void oracle_decode_bf16_array(const uint16_t *in, double *out, int64_t n)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = oracle_bf16_to_f64(in[i]);
}

void oracle_decode_e4m3_array(const uint8_t *in, double *out, int64_t n)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = oracle_e4m3_to_f64(in[i]);
}

void oracle_encode_e4m3_array(const float *in, uint8_t *out, int64_t n)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = oracle_f32_to_e4m3(in[i]);
}

/* ------------------------------------------------------------ cache write */

int oracle_cache_write(const uint16_t *kv_c, const uint16_t *k_pe, const int64_t *slot_mapping,
                       int64_t num_tokens, void *cache, int64_t num_blocks, int page_size,
                       int cache_dtype, float kv_scale)
{
    int64_t nslots = num_blocks * (int64_t)page_size;
    for (int64_t i = 0; i < num_tokens; ++i) {
        int64_t slot = slot_mapping[i];
        if (slot < 0)
            continue;
        if (slot >= nslots)
            return -1;
        for (int d = 0; d < ORC_DQK; ++d) {
            uint16_t x = d < ORC_LKV ? kv_c[i * ORC_LKV + d] : k_pe[i * (ORC_DQK - ORC_LKV) + d - ORC_LKV];
            if (cache_dtype == ORC_CACHE_BF16) {
                ((uint16_t *)cache)[slot * ORC_DQK + d] = x;
            } else {
                float v = (float)oracle_bf16_to_f64(x);
                float scaled = v / kv_scale;      /* float32, correctly rounded */
                ((uint8_t *)cache)[slot * ORC_DQK + d] = oracle_f32_to_e4m3(scaled);
            }
        }
    }
    return 0;
}

/* ---------------------------------------------------------- context gather */

/* float32 -> bf16 bits, round to nearest, ties to even (NaN stays a quiet NaN). */
static uint16_t oracle_f32_to_bf16(float f)
{
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    if ((u & 0x7F800000u) == 0x7F800000u && (u & 0x007FFFFFu))
        return (uint16_t)((u >> 16) | 0x0040u);
    uint32_t keep = u >> 16, rest = u & 0xFFFFu;
    if (rest > 0x8000u || (rest == 0x8000u && (keep & 1u)))
        keep += 1;
    return (uint16_t)keep;
}

int oracle_gather_cache(const void *cache, int64_t num_blocks, int page_size, int cache_dtype, float kv_scale,
                        const int32_t *block_table, int max_pages, const int32_t *cu_seq_lens,
                        const int32_t *seq_starts, int batch, uint16_t *dst, int64_t dst_rows)
{
    for (int b = 0; b < batch; ++b) {
        int64_t n = (int64_t)cu_seq_lens[b + 1] - cu_seq_lens[b];
        for (int64_t j = 0; j < n; ++j) {
            int64_t pos = (int64_t)(seq_starts ? seq_starts[b] : 0) + j;
            int64_t r = cu_seq_lens[b] + j;
            if (r < 0 || r >= dst_rows || pos < 0 || pos >= (int64_t)max_pages * page_size)
                return -1;
            int64_t page = block_table[(int64_t)b * max_pages + pos / page_size];
            if (page < 0 || page >= num_blocks)
                return -1;
            int64_t row = page * page_size + pos % page_size;
            for (int d = 0; d < ORC_DQK; ++d) {
                if (cache_dtype == ORC_CACHE_BF16) {
                    dst[r * ORC_DQK + d] = ((const uint16_t *)cache)[row * ORC_DQK + d];
                } else {
                    float v = (float)oracle_e4m3_to_f64(((const uint8_t *)cache)[row * ORC_DQK + d]);
                    dst[r * ORC_DQK + d] = oracle_f32_to_bf16(v * kv_scale);   /* float32 product */
                }
            }
        }
    }
    return 0;
}

/* ----------------------------------------------------------------- decode */

struct decode_job {
    const double *q;            /* [T, N, 576] */
    const void *cache;
    int64_t num_blocks;
    int page_size, cache_dtype;
    double kv_scale;
    const int32_t *block_table;
    int max_pages;
    const int32_t *seq_lens, *qsl;
    int batch, num_heads;
    double scale;
    const int64_t *rows;        /* flattened t*N + h, or NULL for all rows */
    int64_t nrows;
    int64_t key_begin, key_end; /* key_end < 0: no upper limit */
    double *out, *lse;
    int nthreads;
    int error;
};

struct decode_thread {
    struct decode_job *job;
    int tid;
    int error;
};

static double cache_value(const struct decode_job *J, int64_t page, int off, int d)
{
    int64_t idx = (page * J->page_size + off) * ORC_DQK + d;
    if (J->cache_dtype == ORC_CACHE_BF16)
        return oracle_bf16_to_f64(((const uint16_t *)J->cache)[idx]);
    return oracle_e4m3_to_f64(((const uint8_t *)J->cache)[idx]) * J->kv_scale;
}

static int request_of(const int32_t *qsl, int batch, int64_t t)
{
    int lo = 0, hi = batch - 1;            /* last b with qsl[b] <= t */
    while (lo < hi) {
        int mid = (lo + hi + 1) / 2;
        if (qsl[mid] <= t)
            lo = mid;
        else
            hi = mid - 1;
    }
    return lo;
}

/* One query row: returns 0, or -1 when a referenced page is out of range. */
static int decode_row(const struct decode_job *J, int64_t r, double *o, double *lse, double **sbuf,
                      int64_t *sbuf_len)
{
    int64_t t = r / J->num_heads;
    int b = request_of(J->qsl, J->batch, t);
    int64_t sq = J->qsl[b + 1] - J->qsl[b];
    int64_t L = (int64_t)J->seq_lens[b] - sq + 1 + (t - J->qsl[b]);
    int64_t k0 = J->key_begin > 0 ? J->key_begin : 0;
    int64_t k1 = L > 0 ? L : 0;
    const double *qrow = J->q + r * ORC_DQK;
    double m = -INFINITY, l = 0.0;

    if (J->key_end >= 0 && J->key_end < k1)
        k1 = J->key_end;
    for (int d = 0; d < ORC_LKV; ++d)
        o[d] = 0.0;
    if (k1 <= k0) {                       /* no visible key: empty softmax */
        *lse = -INFINITY;
        return 0;
    }
    if (k1 - k0 > *sbuf_len) {
        free(*sbuf);
        *sbuf_len = k1 - k0;
        *sbuf = (double *)malloc(sizeof(double) * (size_t)*sbuf_len);
    }
    for (int64_t j = k0; j < k1; ++j) {
        int64_t lp = j / J->page_size;
        int64_t page;
        double dot = 0.0;
        if (lp >= J->max_pages)
            return -1;
        page = J->block_table[(int64_t)b * J->max_pages + lp];
        if (page < 0 || page >= J->num_blocks)
            return -1;
        for (int d = 0; d < ORC_DQK; ++d)
            dot += qrow[d] * cache_value(J, page, (int)(j % J->page_size), d);
        (*sbuf)[j - k0] = J->scale * dot;
        if ((*sbuf)[j - k0] > m)
            m = (*sbuf)[j - k0];
    }
    for (int64_t j = k0; j < k1; ++j) {
        int64_t page = J->block_table[(int64_t)b * J->max_pages + j / J->page_size];
        double p = exp((*sbuf)[j - k0] - m);
        l += p;
        for (int d = 0; d < ORC_LKV; ++d)
            o[d] += p * cache_value(J, page, (int)(j % J->page_size), d);
    }
    for (int d = 0; d < ORC_LKV; ++d)
        o[d] /= l;
    *lse = m + log(l);
    return 0;
}

static void *decode_worker(void *arg)
{
    struct decode_thread *T = (struct decode_thread *)arg;
    struct decode_job *J = T->job;
    double *sbuf = NULL;
    int64_t sbuf_len = 0;
    for (int64_t i = T->tid; i < J->nrows; i += J->nthreads) {
        int64_t r = J->rows ? J->rows[i] : i;
        if (decode_row(J, r, J->out + i * ORC_LKV, J->lse + i, &sbuf, &sbuf_len) != 0)
            T->error = -1;
    }
    free(sbuf);
    return NULL;
}

int oracle_num_cores(void)
{
    long n = sysconf(_SC_NPROCESSORS_ONLN);
    return n > 0 ? (int)n : 1;
}

/*
 * out[i, :] / lse[i] = attention of query row rows[i] (flattened t*N + h) over
 * its visible keys restricted to [key_begin, key_end).  Returns the number of
 * threads used, or -1 on a bad argument or an out-of-range page.
 */
int oracle_decode(const double *q, const void *cache, int64_t num_blocks, int page_size,
                  int cache_dtype, double kv_scale, const int32_t *block_table, int max_pages,
                  const int32_t *seq_lens, const int32_t *qsl, int batch, int num_heads,
                  double scale, const int64_t *rows, int64_t nrows, int64_t key_begin,
                  int64_t key_end, double *out, double *lse, int nthreads)
{
    struct decode_job J;
    struct decode_thread *T;
    pthread_t *th;
    int err = 0;

    if (batch <= 0 || num_heads <= 0 || page_size <= 0 || nrows < 0)
        return -1;
    if (cache_dtype != ORC_CACHE_BF16 && cache_dtype != ORC_CACHE_E4M3)
        return -1;
    if (nthreads <= 0)
        nthreads = oracle_num_cores();
    if (nthreads > nrows)
        nthreads = nrows > 0 ? (int)nrows : 1;
    J = (struct decode_job){q, cache, num_blocks, page_size, cache_dtype, kv_scale, block_table,
                            max_pages, seq_lens, qsl, batch, num_heads, scale, rows, nrows,
                            key_begin, key_end, out, lse, nthreads, 0};
    T = (struct decode_thread *)calloc((size_t)nthreads, sizeof *T);
    th = (pthread_t *)calloc((size_t)nthreads, sizeof *th);
    for (int i = 0; i < nthreads; ++i) {
        T[i].job = &J;
        T[i].tid = i;
        if (nthreads == 1)
            decode_worker(&T[i]);
        else
            pthread_create(&th[i], NULL, decode_worker, &T[i]);
    }
    for (int i = 0; i < nthreads; ++i) {
        if (nthreads > 1)
            pthread_join(th[i], NULL);
        if (T[i].error)
            err = -1;
    }
    free(T);
    free(th);
    return err ? -1 : nthreads;
}

/* ------------------------------------------------------------------ merge */

void oracle_merge(const double *o_a, const double *lse_a, const double *o_b, const double *lse_b,
                  int64_t rows, int dim, double *out, double *lse)
{
    for (int64_t r = 0; r < rows; ++r) {
        double la = lse_a[r], lb = lse_b[r];
        if (la == -INFINITY && lb == -INFINITY) {   /* both sides saw no key */
            for (int d = 0; d < dim; ++d)
                out[r * dim + d] = 0.0;
            lse[r] = -INFINITY;
            continue;
        }
        double m = la > lb ? la : lb;
        double wa = exp(la - m), wb = exp(lb - m), s = wa + wb;
        for (int d = 0; d < dim; ++d)
            out[r * dim + d] = (wa * o_a[r * dim + d] + wb * o_b[r * dim + d]) / s;
        lse[r] = m + log(s);
    }
}
