/*
 * oracle.c -- the plain CPU oracle for batched attention over a paged K/V pool.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the slow, obviously-correct statement
 * of what the GPU path computes.  Only tests/, __graft_entry__.smoke() and the
 * cpu_baseline / reference legs of bench.py may load it.  It shares no code,
 * header, table or constant with the CUDA library in paged_kv_continuous_pa_gb300/,
 * and the library never calls it.
 *
 * Sources (the pages' titles and sections):
 *   - "GPU inference engine engineering", section "Batching without running out
 *     of cache": the K/V memory is a paged pool addressed through a per-sequence
 *     block table of 32-token pages; every step is a set of rows, each with its
 *     own token, sequence and position.
 *   - "Building an LLM runtime from scratch on NVIDIA H100", section "Bug #1":
 *     paged decode attention loads K and V pages and runs an FP32 online softmax.
 *     The oracle computes the same quantity exactly (up to FP64 rounding), by the
 *     textbook definition softmax(q.K^T * scale) . V, with no blocking.
 *   - "GPU inference engine engineering", section "The same bits in any batch":
 *     BF16 key/value storage with round-to-nearest-even.
 *   - "Engines for the card you have", section "One checkpoint, many engines":
 *     an FP8 key/value cache with calibration.  The pages leave the calibration's
 *     granularity open; the oracle takes a per-tensor scale, or one scale per
 *     KV head.
 *
 * Readings where the pages are silent:
 *   - a row at position p attends keys 0..p inclusive (causal, own token included);
 *   - q head g reads kv head g / (Hq / Hkv);
 *   - fp8 is OCP E4M3 (bias 7, max finite 448, no infinities, S.1111.111 is NaN),
 *     encoded as satfinite-RNE(x / scale) with x / scale one IEEE binary32 division;
 *   - decoding an fp8 code gives value(code) * scale.
 *
 * Everything is in FP64 except the two encoders, whose inputs are binary32 by
 * definition.  Compile without contraction (-ffp-contract=off) so that the one
 * binary32 division in the fp8 encoder is exactly the IEEE operation.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

enum { OR_F32 = 0, OR_BF16 = 1, OR_E4M3 = 2 };

/* ------------------------------------------------------------------ bf16 -- */

/* fp32 -> bf16 with round-to-nearest, ties to even, on the bit pattern:
 * keep the top 16 bits, add half an ulp of bf16 plus the parity of the kept
 * part so that exact ties go to the even neighbour.  NaN stays a quiet NaN. */
uint16_t oracle_bf16_from_f32(float x)
{
    uint32_t u;
    memcpy(&u, &x, 4);
    if ((u & 0x7f800000u) == 0x7f800000u && (u & 0x007fffffu) != 0u)
        return (uint16_t)((u >> 16) | 0x0040u);
    uint32_t keep_lsb = (u >> 16) & 1u;
    u += 0x7fffu + keep_lsb;
    return (uint16_t)(u >> 16);
}

double oracle_bf16_to_f64(uint16_t h)
{
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, 4);
    return (double)f;
}

/* ------------------------------------------------------------- fp8 e4m3 -- */

/* Value of an E4M3 code from its fields (OCP 8-bit floating point, E4M3):
 * sign s, 4-bit exponent e with bias 7, 3-bit mantissa m.
 *   e == 0          : subnormal, (m / 8) * 2^(1 - 7)
 *   e == 15, m == 7 : NaN (the only non-finite encoding)
 *   otherwise       : (1 + m / 8) * 2^(e - 7)                                 */
double oracle_e4m3_to_f64(uint8_t code)
{
    int s = code >> 7;
    int e = (code >> 3) & 0xf;
    int m = code & 0x7;
    double v;
    if (e == 15 && m == 7)
        return NAN;
    if (e == 0)
        v = ldexp((double)m / 8.0, 1 - 7);
    else
        v = ldexp(1.0 + (double)m / 8.0, e - 7);
    return s ? -v : v;
}

/* Nearest E4M3 code to a binary32 value, ties to the even code, saturating to
 * +-448 (the largest finite code 0x7E) instead of overflowing.  The positive
 * finite codes 0x00..0x7E are strictly increasing in value, so the two
 * neighbours of |x| are found by bisection over the codes, and the decision
 * compares |x| with their midpoint, which has at most five significant bits
 * and is therefore exact in double, as is |x| itself.                         */
uint8_t oracle_e4m3_from_f32(float x)
{
    if (isnan(x))
        return 0x7f;
    uint8_t sign = signbit(x) ? 0x80 : 0x00;
    double a = fabs((double)x);
    if (a >= 448.0)
        return sign | 0x7e;
    int lo = 0, hi = 0x7e; /* invariant: value(lo) <= a < value(hi) */
    while (hi - lo > 1) {
        int mid = (lo + hi) / 2;
        if (oracle_e4m3_to_f64((uint8_t)mid) <= a)
            lo = mid;
        else
            hi = mid;
    }
    double vlo = oracle_e4m3_to_f64((uint8_t)lo);
    double vhi = oracle_e4m3_to_f64((uint8_t)hi);
    double midpoint = 0.5 * (vlo + vhi);
    int code;
    if (a < midpoint)
        code = lo;
    else if (a > midpoint)
        code = hi;
    else
        code = (lo & 1) ? hi : lo;
    return sign | (uint8_t)code;
}

void oracle_e4m3_from_f32_array(const float *x, uint8_t *out, int64_t n)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = oracle_e4m3_from_f32(x[i]);
}

/* --------------------------------------------------------- element codec -- */

static size_t elt_size(int dtype)
{
    return dtype == OR_F32 ? 4 : dtype == OR_BF16 ? 2 : 1;
}

/* Input element i of an array of dtype (f32 or bf16) as binary32, exactly. */
static float load_as_f32(const void *base, int dtype, int64_t i)
{
    if (dtype == OR_F32)
        return ((const float *)base)[i];
    uint32_t u = (uint32_t)((const uint16_t *)base)[i] << 16;
    float f;
    memcpy(&f, &u, 4);
    return f;
}

/* Stored pool element i, decoded to double.  fp8 is multiplied by its scale. */
static double load_pool(const void *pool, int dtype, int64_t i, float scale)
{
    if (dtype == OR_F32)
        return (double)((const float *)pool)[i];
    if (dtype == OR_BF16)
        return oracle_bf16_to_f64(((const uint16_t *)pool)[i]);
    return oracle_e4m3_to_f64(((const uint8_t *)pool)[i]) * (double)scale;
}

/* Encode one input element into pool slot i.
 * Returns 0 on success, -1 for an unsupported (input, storage) pair. */
static int store_pool(void *pool, int kv_dtype, int64_t i, const void *src, int in_dtype,
                      int64_t j, float scale)
{
    if (kv_dtype == OR_F32) {
        ((float *)pool)[i] = load_as_f32(src, in_dtype, j); /* f32 copy or exact bf16 widening */
        return 0;
    }
    if (kv_dtype == OR_BF16) {
        if (in_dtype == OR_BF16)
            ((uint16_t *)pool)[i] = ((const uint16_t *)src)[j];
        else
            ((uint16_t *)pool)[i] = oracle_bf16_from_f32(((const float *)src)[j]);
        return 0;
    }
    if (kv_dtype == OR_E4M3) {
        volatile float q = load_as_f32(src, in_dtype, j) / scale; /* one IEEE binary32 division */
        ((uint8_t *)pool)[i] = oracle_e4m3_from_f32(q);
        return 0;
    }
    return -1;
}

/* ----------------------------------------------------------------- append -- */

/* Scatter every row's new key and value into its page slot.
 *
 * Layouts:  k_new, v_new  [n_rows][Hkv][D]            in_dtype (f32 or bf16)
 *           block_tables  [num_seqs][max_blocks]       int32, -1 = unused
 *           k_pool, v_pool [num_pages][Hkv][P][D]      kv_dtype
 * Row r with sequence s and position p writes page block_tables[s][p / P],
 * slot p % P, for every kv head and every element, in row order.
 * Returns 0, or -1 if a row's sequence, position or page is out of range (the
 * rows before it are written), or -2 for an unsupported dtype pair.           */
int oracle_append_h(int32_t n_rows, const void *k_new, const void *v_new, int32_t in_dtype,
                    const int32_t *seq_ids, const int32_t *positions, const int32_t *block_tables,
                    int32_t num_seqs, int32_t max_blocks, int32_t num_pages, int32_t page_size,
                    int32_t num_kv_heads, int32_t head_dim, int32_t kv_dtype, const float *k_scales,
                    const float *v_scales, void *k_pool, void *v_pool)
{
    const int P = page_size, H = num_kv_heads, D = head_dim;
    for (int32_t r = 0; r < n_rows; ++r) {
        int32_t s = seq_ids[r], p = positions[r];
        if (s < 0 || s >= num_seqs || p < 0 || p / P >= max_blocks)
            return -1;
        int32_t page = block_tables[(int64_t)s * max_blocks + p / P];
        if (page < 0 || page >= num_pages)
            return -1;
        int32_t slot = p % P;
        for (int h = 0; h < H; ++h)
            for (int d = 0; d < D; ++d) {
                int64_t dst = (((int64_t)page * H + h) * P + slot) * D + d;
                int64_t src = ((int64_t)r * H + h) * D + d;
                if (store_pool(k_pool, kv_dtype, dst, k_new, in_dtype, src, k_scales[h]) ||
                    store_pool(v_pool, kv_dtype, dst, v_new, in_dtype, src, v_scales[h]))
                    return -2;
            }
    }
    return 0;
}

/* The same with one scale for every kv head (a per-tensor scale). */
int oracle_append(int32_t n_rows, const void *k_new, const void *v_new, int32_t in_dtype,
                  const int32_t *seq_ids, const int32_t *positions, const int32_t *block_tables,
                  int32_t num_seqs, int32_t max_blocks, int32_t num_pages, int32_t page_size,
                  int32_t num_kv_heads, int32_t head_dim, int32_t kv_dtype, float k_scale,
                  float v_scale, void *k_pool, void *v_pool)
{
    if (num_kv_heads <= 0)
        return -2;
    float *ks = (float *)malloc(sizeof(float) * (size_t)num_kv_heads);
    float *vs = (float *)malloc(sizeof(float) * (size_t)num_kv_heads);
    int st = -3;
    if (ks && vs) {
        for (int h = 0; h < num_kv_heads; ++h) {
            ks[h] = k_scale;
            vs[h] = v_scale;
        }
        st = oracle_append_h(n_rows, k_new, v_new, in_dtype, seq_ids, positions, block_tables, num_seqs,
                             max_blocks, num_pages, page_size, num_kv_heads, head_dim, kv_dtype, ks, vs,
                             k_pool, v_pool);
    }
    free(ks);
    free(vs);
    return st;
}

/* -------------------------------------------------------------- attention -- */

typedef struct {
    int32_t n_rows;
    const void *q;
    int32_t q_dtype, num_q_heads;
    const int32_t *seq_ids, *positions, *block_tables;
    int32_t num_seqs, max_blocks, num_pages, page_size, num_kv_heads, head_dim, kv_dtype;
    const float *k_scales, *v_scales;  /* per kv head */
    const void *k_pool, *v_pool;
    double softmax_scale;
    double *out;
    int32_t row_begin, row_end;
    int status;
} attn_args;

/* Attention for rows [row_begin, row_end) by the definition.  For row r with
 * sequence s and position p, and query head g (kv head h = g / G):
 *   keys t = 0..p, fetched page by page: page = block_tables[s][t / P], slot t % P
 *   score_t = scale * sum_d q[r][g][d] * K[t][d]
 *   w_t     = exp(score_t - max_t score_t)
 *   out[r][g][:] = sum_t w_t * V[t][:] / sum_t w_t
 * All in double; out is [n_rows][Hq][D] double.                               */
static void attention_rows(attn_args *a)
{
    const int P = a->page_size, H = a->num_kv_heads, D = a->head_dim, Hq = a->num_q_heads;
    const int G = Hq / H;
    int64_t cap = (int64_t)a->max_blocks * P;
    double *score = (double *)malloc(sizeof(double) * (size_t)(cap > 0 ? cap : 1));
    double *acc = (double *)malloc(sizeof(double) * (size_t)D);
    int32_t *page_of = (int32_t *)malloc(sizeof(int32_t) * (size_t)(a->max_blocks > 0 ? a->max_blocks : 1));
    if (!score || !acc || !page_of) {
        a->status = -3;
        goto done;
    }
    for (int32_t r = a->row_begin; r < a->row_end; ++r) {
        int32_t s = a->seq_ids[r], p = a->positions[r];
        if (s < 0 || s >= a->num_seqs || p < 0 || (int64_t)p >= cap) {
            a->status = -1;
            goto done;
        }
        int64_t L = (int64_t)p + 1;
        /* gather this row's pages through its block table */
        for (int64_t j = 0; j * P < L; ++j) {
            page_of[j] = a->block_tables[(int64_t)s * a->max_blocks + j];
            if (page_of[j] < 0 || page_of[j] >= a->num_pages) {
                a->status = -1;
                goto done;
            }
        }
        for (int g = 0; g < Hq; ++g) {
            int h = g / G;
            int64_t qoff = ((int64_t)r * Hq + g) * D;
            double m = -INFINITY;
            for (int64_t t = 0; t < L; ++t) {
                int64_t base = (((int64_t)page_of[t / P] * H + h) * P + t % P) * D;
                double dot = 0.0;
                for (int d = 0; d < D; ++d)
                    dot += (double)load_as_f32(a->q, a->q_dtype, qoff + d) *
                           load_pool(a->k_pool, a->kv_dtype, base + d, a->k_scales[h]);
                score[t] = a->softmax_scale * dot;
                if (score[t] > m)
                    m = score[t];
            }
            double z = 0.0;
            for (int d = 0; d < D; ++d)
                acc[d] = 0.0;
            for (int64_t t = 0; t < L; ++t) {
                double w = exp(score[t] - m);
                int64_t base = (((int64_t)page_of[t / P] * H + h) * P + t % P) * D;
                z += w;
                for (int d = 0; d < D; ++d)
                    acc[d] += w * load_pool(a->v_pool, a->kv_dtype, base + d, a->v_scales[h]);
            }
            for (int d = 0; d < D; ++d)
                a->out[qoff + d] = acc[d] / z;
        }
    }
done:
    free(score);
    free(acc);
    free(page_of);
}

static void *attention_thread(void *p)
{
    attention_rows((attn_args *)p);
    return NULL;
}

/* Returns 0, -1 for an out-of-range row or page, -2 for bad arguments, -3 if
 * host memory ran out.  softmax_scale <= 0 means 1/sqrt(head_dim).
 * n_threads > 1 splits the rows into contiguous ranges, one per thread; each
 * row's arithmetic is the same whichever thread runs it.                     */
int oracle_attention_h(int32_t n_rows, const void *q, int32_t q_dtype, int32_t num_q_heads,
                       const int32_t *seq_ids, const int32_t *positions, const int32_t *block_tables,
                       int32_t num_seqs, int32_t max_blocks, int32_t num_pages, int32_t page_size,
                       int32_t num_kv_heads, int32_t head_dim, int32_t kv_dtype, const float *k_scales,
                       const float *v_scales, const void *k_pool, const void *v_pool, double softmax_scale,
                       double *out, int32_t n_threads)
{
    if (n_rows < 0 || num_kv_heads <= 0 || num_q_heads % num_kv_heads != 0 || page_size <= 0 ||
        head_dim <= 0 || (q_dtype != OR_F32 && q_dtype != OR_BF16) ||
        (kv_dtype != OR_F32 && kv_dtype != OR_BF16 && kv_dtype != OR_E4M3))
        return -2;
    if (softmax_scale <= 0.0)
        softmax_scale = 1.0 / sqrt((double)head_dim);
    if (n_threads < 1)
        n_threads = 1;
    if (n_threads > n_rows)
        n_threads = n_rows > 0 ? n_rows : 1;
    attn_args *args = (attn_args *)calloc((size_t)n_threads, sizeof(attn_args));
    pthread_t *tid = (pthread_t *)calloc((size_t)n_threads, sizeof(pthread_t));
    if (!args || !tid) {
        free(args);
        free(tid);
        return -3;
    }
    for (int i = 0; i < n_threads; ++i) {
        attn_args *a = &args[i];
        a->n_rows = n_rows;
        a->q = q;
        a->q_dtype = q_dtype;
        a->num_q_heads = num_q_heads;
        a->seq_ids = seq_ids;
        a->positions = positions;
        a->block_tables = block_tables;
        a->num_seqs = num_seqs;
        a->max_blocks = max_blocks;
        a->num_pages = num_pages;
        a->page_size = page_size;
        a->num_kv_heads = num_kv_heads;
        a->head_dim = head_dim;
        a->kv_dtype = kv_dtype;
        a->k_scales = k_scales;
        a->v_scales = v_scales;
        a->k_pool = k_pool;
        a->v_pool = v_pool;
        a->softmax_scale = softmax_scale;
        a->out = out;
        a->row_begin = (int32_t)((int64_t)n_rows * i / n_threads);
        a->row_end = (int32_t)((int64_t)n_rows * (i + 1) / n_threads);
        a->status = 0;
    }
    int started = 0;
    for (int i = 1; i < n_threads; ++i) {
        if (pthread_create(&tid[i], NULL, attention_thread, &args[i]) != 0)
            break;
        started = i;
    }
    attention_rows(&args[0]);
    /* rows of threads that could not be started run here, in order */
    for (int i = started + 1; i < n_threads; ++i)
        attention_rows(&args[i]);
    for (int i = 1; i <= started; ++i)
        pthread_join(tid[i], NULL);
    int status = 0;
    for (int i = 0; i < n_threads; ++i)
        if (args[i].status != 0 && status == 0)
            status = args[i].status;
    free(args);
    free(tid);
    return status;
}

size_t oracle_elt_size(int32_t dtype)
{
    return elt_size(dtype);
}

/* The same with one scale for every kv head (a per-tensor scale). */
int oracle_attention(int32_t n_rows, const void *q, int32_t q_dtype, int32_t num_q_heads,
                     const int32_t *seq_ids, const int32_t *positions, const int32_t *block_tables,
                     int32_t num_seqs, int32_t max_blocks, int32_t num_pages, int32_t page_size,
                     int32_t num_kv_heads, int32_t head_dim, int32_t kv_dtype, float k_scale,
                     float v_scale, const void *k_pool, const void *v_pool, double softmax_scale,
                     double *out, int32_t n_threads)
{
    if (num_kv_heads <= 0)
        return -2;
    float *ks = (float *)malloc(sizeof(float) * (size_t)num_kv_heads);
    float *vs = (float *)malloc(sizeof(float) * (size_t)num_kv_heads);
    int st = -3;
    if (ks && vs) {
        for (int h = 0; h < num_kv_heads; ++h) {
            ks[h] = k_scale;
            vs[h] = v_scale;
        }
        st = oracle_attention_h(n_rows, q, q_dtype, num_q_heads, seq_ids, positions, block_tables, num_seqs,
                                max_blocks, num_pages, page_size, num_kv_heads, head_dim, kv_dtype, ks, vs,
                                k_pool, v_pool, softmax_scale, out, n_threads);
    }
    free(ks);
    free(vs);
    return st;
}
