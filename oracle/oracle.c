/*
 * oracle.c -- plain fp64 CPU oracle for split-K paged decode attention.
 *
 * TEST INFRASTRUCTURE ONLY. It is built on its own into liboracle.so and is
 * loaded by the tests, the smoke check and the CPU-baseline leg of the
 * benchmark, never by the library. It shares no code with the CUDA path.
 *
 * What is computed, for every sequence b, query token t and query head h:
 *
 *   kv head      k     = h / (num_q_heads / num_kv_heads)
 *                        (GQA head fusion: a tile covers `group` heads that
 *                         read one K/V stream; FA4Config page, field `group`
 *                         and method BM_eff)
 *   visible keys n_vis = L_b - num_q + t + 1
 *                        (the num_q new tokens are the last num_q positions
 *                         of the cache; key j is visible to token t when
 *                         j <= L_b - num_q + t)
 *   key row      K_j   = k_pages[page_table[b][j / PS]][k][j % PS][:]
 *                        (block-indirected paged cache: FA4Config page,
 *                         method v_row_major, "gmem_row = block_idx * stride")
 *   value row    V_j   = v_pages[same][:ov]  or  K_j[:ov] for the MLA latent
 *                        (FA4Config page, methods shared_kv_cols and
 *                         rope_depth: K_nope and V share one row)
 *   s_j = scale * sum_d q[b,t,h,d] * K_j[d]
 *   out = sum_j exp(s_j - m) V_j / sum_j exp(s_j - m),  m = max_j s_j
 *   lse = m + ln sum_j exp(s_j - m)
 *
 * A row with no visible key gets out = 0 and lse = -inf.
 *
 * oracle_partitioned reaches the same numbers the way the split-K kernel
 * does: each partition keeps a max in raw q.k units and a sum of
 * exp2((s_raw - max) * c) with c = scale * log2(e) (the `scale_log2e`
 * argument), normalises its own output by its own sum, and the partitions
 * are merged with the log-sum-exp weights of the fa4_splitk_combine_write
 * page (description, first paragraph):
 *   Gmax = max_p max_p,  Gsum = sum_p sum_p * exp2((max_p - Gmax) * c),
 *   w_p = sum_p * exp2((max_p - Gmax) * c) / Gsum,  O = sum_p w_p * O_p.
 * Everything is fp64; bf16 inputs are widened exactly.
 */
#include "oracle.h"

#include <math.h>
#include <pthread.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

static double widen_bf16(uint16_t bits)
{
    uint32_t u = (uint32_t)bits << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

static int shape_ok(const oracle_shape* s)
{
    if (!s) return 0;
    if (s->batch < 0 || s->num_q < 1 || s->num_q_heads < 1 || s->num_kv_heads < 1) return 0;
    if (s->num_q_heads % s->num_kv_heads) return 0;
    if (s->qk_depth < 1 || s->ov_depth < 1 || s->page_size < 1) return 0;
    if (s->max_pages_per_seq < 0 || s->num_pages < 0) return 0;
    if (s->v_in_k && s->ov_depth > s->qk_depth) return 0;
    return 1;
}

/* Address of key row j of sequence b, kv head k; NULL if the page id is bad. */
static const uint16_t* key_row(const oracle_shape* s, const uint16_t* k_pages,
                               const int32_t* page_table, int b, int k, int64_t j)
{
    int64_t slot = j / s->page_size;
    if (slot >= s->max_pages_per_seq) return NULL;
    int32_t phys = page_table[(int64_t)b * s->max_pages_per_seq + slot];
    if (phys < 0 || phys >= s->num_pages) return NULL;
    int64_t row = ((int64_t)phys * s->num_kv_heads + k) * s->page_size + j % s->page_size;
    return k_pages + row * s->qk_depth;
}

static const uint16_t* value_row(const oracle_shape* s, const uint16_t* k_pages,
                                 const uint16_t* v_pages, const int32_t* page_table,
                                 int b, int k, int64_t j)
{
    if (s->v_in_k) return key_row(s, k_pages, page_table, b, k, j);
    int64_t slot = j / s->page_size;
    if (slot >= s->max_pages_per_seq) return NULL;
    int32_t phys = page_table[(int64_t)b * s->max_pages_per_seq + slot];
    if (phys < 0 || phys >= s->num_pages) return NULL;
    int64_t row = ((int64_t)phys * s->num_kv_heads + k) * s->page_size + j % s->page_size;
    return v_pages + row * s->ov_depth;
}

typedef struct row_job {
    const oracle_shape* s;
    double scale;
    const uint16_t *q, *k, *v;
    const int32_t *pt, *lens, *rows, *bounds;
    int64_t n_rows;
    int num_parts;
    double *out, *lse, *pmax, *psum;
    int tid, nthreads;
    int failed;
    /* fp8 cache (oracle_decode_fp8 only) */
    const uint8_t *k8, *v8;
    const uint16_t* krope;
    const float* kscale;
    int rope_depth;
} row_job;

/* q.k for one (row, key), unscaled, exact products of widened bf16. */
static double dot_row(const uint16_t* qrow, const uint16_t* krow, int depth)
{
    double acc = 0.0;
    for (int d = 0; d < depth; ++d) acc += widen_bf16(qrow[d]) * widen_bf16(krow[d]);
    return acc;
}

/* The plain definition for one query row (b, t, h). */
static int plain_row(row_job* J, int b, int t, int h, double* o, double* lse_out, double* sbuf)
{
    const oracle_shape* s = J->s;
    int group = s->num_q_heads / s->num_kv_heads;
    int k = h / group;
    int64_t L = J->lens[b];
    int64_t n_vis = L - s->num_q + t + 1;
    for (int d = 0; d < s->ov_depth; ++d) o[d] = 0.0;
    if (n_vis <= 0) {
        if (lse_out) *lse_out = -INFINITY;
        return 0;
    }
    const uint16_t* qrow = J->q + (((int64_t)b * s->num_q + t) * s->num_q_heads + h) * s->qk_depth;
    double m = -INFINITY;
    for (int64_t j = 0; j < n_vis; ++j) {
        const uint16_t* kr = key_row(s, J->k, J->pt, b, k, j);
        if (!kr) return -1;
        sbuf[j] = J->scale * dot_row(qrow, kr, s->qk_depth);
        if (sbuf[j] > m) m = sbuf[j];
    }
    double l = 0.0;
    for (int64_t j = 0; j < n_vis; ++j) {
        double e = exp(sbuf[j] - m);
        l += e;
        const uint16_t* vr = value_row(s, J->k, J->v, J->pt, b, k, j);
        if (!vr) return -1;
        for (int d = 0; d < s->ov_depth; ++d) o[d] += e * widen_bf16(vr[d]);
    }
    for (int d = 0; d < s->ov_depth; ++d) o[d] /= l;
    if (lse_out) *lse_out = m + log(l);
    return 0;
}

/* The split path for one query row: per-partition state, then the combine. */
static int split_row(row_job* J, int b, int t, int h, double* o, double* lse_out,
                     double* pmax, double* psum, double* obuf)
{
    const oracle_shape* s = J->s;
    const int P = J->num_parts;
    const double c = J->scale * (1.0 / log(2.0)); /* scale * log2(e) */
    int group = s->num_q_heads / s->num_kv_heads;
    int k = h / group;
    int64_t L = J->lens[b];
    int64_t n_vis = L - s->num_q + t + 1;
    const int32_t* bnd = J->bounds + (int64_t)b * (P + 1);
    const uint16_t* qrow = J->q + (((int64_t)b * s->num_q + t) * s->num_q_heads + h) * s->qk_depth;

    /* Pass 1: every partition on its own. obuf is [P][ov_depth]. */
    for (int p = 0; p < P; ++p) {
        double* op = obuf + (int64_t)p * s->ov_depth;
        for (int d = 0; d < s->ov_depth; ++d) op[d] = 0.0;
        int64_t lo = bnd[p], hi = bnd[p + 1];
        if (hi > n_vis) hi = n_vis;
        if (lo < 0) lo = 0;
        double mx = -INFINITY;
        for (int64_t j = lo; j < hi; ++j) {
            const uint16_t* kr = key_row(s, J->k, J->pt, b, k, j);
            if (!kr) return -1;
            double raw = dot_row(qrow, kr, s->qk_depth);
            if (raw > mx) mx = raw;
        }
        double sum = 0.0;
        for (int64_t j = lo; j < hi; ++j) {
            const uint16_t* kr = key_row(s, J->k, J->pt, b, k, j);
            const uint16_t* vr = value_row(s, J->k, J->v, J->pt, b, k, j);
            if (!vr) return -1;
            double e = exp2((dot_row(qrow, kr, s->qk_depth) - mx) * c);
            sum += e;
            for (int d = 0; d < s->ov_depth; ++d) op[d] += e * widen_bf16(vr[d]);
        }
        if (sum > 0.0)
            for (int d = 0; d < s->ov_depth; ++d) op[d] /= sum;
        pmax[p] = mx;
        psum[p] = sum;
    }

    /* Pass 2: the log-sum-exp combine. Empty partitions (sum 0) carry no
     * weight and are skipped so that -inf - -inf never appears. */
    double gmax = -INFINITY;
    for (int p = 0; p < P; ++p)
        if (psum[p] > 0.0 && pmax[p] > gmax) gmax = pmax[p];
    for (int d = 0; d < s->ov_depth; ++d) o[d] = 0.0;
    if (gmax == -INFINITY) {
        if (lse_out) *lse_out = -INFINITY;
        return 0;
    }
    double gsum = 0.0;
    for (int p = 0; p < P; ++p)
        if (psum[p] > 0.0) gsum += psum[p] * exp2((pmax[p] - gmax) * c);
    for (int p = 0; p < P; ++p) {
        if (psum[p] <= 0.0) continue;
        double w = psum[p] * exp2((pmax[p] - gmax) * c) / gsum;
        const double* op = obuf + (int64_t)p * s->ov_depth;
        for (int d = 0; d < s->ov_depth; ++d) o[d] += w * op[d];
    }
    /* natural-log LSE of the scaled scores: sum_j exp(scale*(s_j - Gmax)) = Gsum */
    if (lse_out) *lse_out = J->scale * gmax + log(gsum);
    return 0;
}

static void* plain_worker(void* arg)
{
    row_job* J = (row_job*)arg;
    const oracle_shape* s = J->s;
    int64_t max_len = 0;
    for (int b = 0; b < s->batch; ++b)
        if (J->lens[b] > max_len) max_len = J->lens[b];
    double* sbuf = (double*)malloc(sizeof(double) * (size_t)(max_len > 0 ? max_len : 1));
    if (!sbuf) { J->failed = 1; return NULL; }
    if (J->rows) {
        for (int64_t i = J->tid; i < J->n_rows; i += J->nthreads) {
            int b = J->rows[3 * i], t = J->rows[3 * i + 1], h = J->rows[3 * i + 2];
            if (b < 0 || b >= s->batch || t < 0 || t >= s->num_q || h < 0 || h >= s->num_q_heads) {
                J->failed = 1;
                break;
            }
            if (plain_row(J, b, t, h, J->out + i * s->ov_depth, J->lse ? J->lse + i : NULL, sbuf)) {
                J->failed = 1;
                break;
            }
        }
    } else {
        int64_t total = (int64_t)s->batch * s->num_q * s->num_q_heads;
        for (int64_t i = J->tid; i < total; i += J->nthreads) {
            int h = (int)(i % s->num_q_heads);
            int t = (int)((i / s->num_q_heads) % s->num_q);
            int b = (int)(i / ((int64_t)s->num_q_heads * s->num_q));
            if (plain_row(J, b, t, h, J->out + i * s->ov_depth, J->lse ? J->lse + i : NULL, sbuf)) {
                J->failed = 1;
                break;
            }
        }
    }
    free(sbuf);
    return NULL;
}

static void* split_worker(void* arg)
{
    row_job* J = (row_job*)arg;
    const oracle_shape* s = J->s;
    const int P = J->num_parts;
    double* obuf = (double*)malloc(sizeof(double) * (size_t)P * s->ov_depth);
    double* pm = (double*)malloc(sizeof(double) * (size_t)P);
    double* ps = (double*)malloc(sizeof(double) * (size_t)P);
    if (!obuf || !pm || !ps) { J->failed = 1; free(obuf); free(pm); free(ps); return NULL; }
    int64_t total = (int64_t)s->batch * s->num_q * s->num_q_heads;
    for (int64_t i = J->tid; i < total; i += J->nthreads) {
        int h = (int)(i % s->num_q_heads);
        int t = (int)((i / s->num_q_heads) % s->num_q);
        int b = (int)(i / ((int64_t)s->num_q_heads * s->num_q));
        if (split_row(J, b, t, h, J->out + i * s->ov_depth, J->lse ? J->lse + i : NULL, pm, ps, obuf)) {
            J->failed = 1;
            break;
        }
        if (J->pmax) for (int p = 0; p < P; ++p) J->pmax[i * P + p] = pm[p];
        if (J->psum) for (int p = 0; p < P; ++p) J->psum[i * P + p] = ps[p];
    }
    free(obuf);
    free(pm);
    free(ps);
    return NULL;
}

static int run_jobs(row_job* proto, void* (*fn)(void*), int num_threads)
{
    if (num_threads <= 0) num_threads = 1;
    if (num_threads > 1024) num_threads = 1024;
    row_job* jobs = (row_job*)calloc((size_t)num_threads, sizeof(row_job));
    pthread_t* th = (pthread_t*)calloc((size_t)num_threads, sizeof(pthread_t));
    char* spawned = (char*)calloc((size_t)num_threads, 1);
    if (!jobs || !th || !spawned) { free(jobs); free(th); free(spawned); return -1; }
    for (int i = 0; i < num_threads; ++i) {
        jobs[i] = *proto;
        jobs[i].tid = i;
        jobs[i].nthreads = num_threads;
        if (i > 0) spawned[i] = pthread_create(&th[i], NULL, fn, &jobs[i]) == 0;
    }
    fn(&jobs[0]);
    int failed = jobs[0].failed;
    for (int i = 1; i < num_threads; ++i) {
        if (spawned[i]) pthread_join(th[i], NULL);
        else fn(&jobs[i]); /* thread creation failed: do its share here */
        failed |= jobs[i].failed;
    }
    free(jobs);
    free(th);
    free(spawned);
    return failed ? -1 : 0;
}

static int lens_ok(const oracle_shape* s, const int32_t* lens)
{
    for (int b = 0; b < s->batch; ++b)
        if (lens[b] < 0 || (int64_t)lens[b] > (int64_t)s->max_pages_per_seq * s->page_size) return 0;
    return 1;
}

int oracle_decode(const oracle_shape* s, double scale, const uint16_t* q,
                  const uint16_t* k_pages, const uint16_t* v_pages,
                  const int32_t* page_table, const int32_t* seq_lens,
                  const int32_t* rows, int64_t n_rows,
                  double* out, double* lse, int num_threads)
{
    if (!shape_ok(s) || !q || !k_pages || (!v_pages && !s->v_in_k) || !page_table || !seq_lens || !out)
        return -1;
    if (rows && n_rows < 0) return -1;
    if (!lens_ok(s, seq_lens)) return -1;
    row_job proto;
    memset(&proto, 0, sizeof proto);
    proto.s = s;
    proto.scale = scale;
    proto.q = q;
    proto.k = k_pages;
    proto.v = v_pages;
    proto.pt = page_table;
    proto.lens = seq_lens;
    proto.rows = rows;
    proto.n_rows = n_rows;
    proto.out = out;
    proto.lse = lse;
    return run_jobs(&proto, plain_worker, num_threads);
}

int oracle_partitioned(const oracle_shape* s, double scale, const uint16_t* q,
                       const uint16_t* k_pages, const uint16_t* v_pages,
                       const int32_t* page_table, const int32_t* seq_lens,
                       const int32_t* bounds, int num_parts,
                       double* out, double* lse,
                       double* part_max, double* part_sum, int num_threads)
{
    if (!shape_ok(s) || !q || !k_pages || (!v_pages && !s->v_in_k) || !page_table || !seq_lens || !out)
        return -1;
    if (!bounds || num_parts < 1) return -1;
    if (!lens_ok(s, seq_lens)) return -1;
    for (int b = 0; b < s->batch; ++b)
        for (int p = 0; p < num_parts; ++p)
            if (bounds[(int64_t)b * (num_parts + 1) + p] > bounds[(int64_t)b * (num_parts + 1) + p + 1])
                return -1;
    row_job proto;
    memset(&proto, 0, sizeof proto);
    proto.s = s;
    proto.scale = scale;
    proto.q = q;
    proto.k = k_pages;
    proto.v = v_pages;
    proto.pt = page_table;
    proto.lens = seq_lens;
    proto.bounds = bounds;
    proto.num_parts = num_parts;
    proto.out = out;
    proto.lse = lse;
    proto.pmax = part_max;
    proto.psum = part_sum;
    return run_jobs(&proto, split_worker, num_threads);
}

/* ------------------------------------------------------------------------
 * fp8 KV cache: the cache dtype, the separate rope dtype and the per-token K
 * scale of the FA4Config page (struct parameters qkv_dtype, rope_dtype_ and
 * scale_dtype_; methods num_k_scale_bufs, q_rope_bytes and rope_depth).
 *
 * The cache holds OCP FP8 E4M3 codes (1 sign bit, 4 exponent bits with bias
 * 7, 3 mantissa bits; exponent field 0 is subnormal, m/8 * 2^-6; the code
 * S.1111.111 is NaN; there is no infinity; the largest finite value is 448).
 * Key row j of kv head k, at cache row r = (page * Hkv + k) * PS + j % PS:
 *   K_j[0 : qk - R)  = k_scale[r] * e4m3(k8[r][0 : qk - R])   (k_scale 1 if absent)
 *   K_j[qk - R : qk] = bf16(k_rope[r][0 : R])                  (R = rope_depth, unscaled)
 * Value row: V_j = e4m3(v8[r][0 : ov]) (no scale: the pages scale K only),
 * or, in the latent layout, the first ov values of the dequantized fp8 part
 * of the key row, k_scale[r] * e4m3(k8[r][0 : ov]) -- the stored row is one
 * latent vector, so its K and V readings dequantize alike.
 * Everything else is the plain definition of plain_row, in fp64.
 * ------------------------------------------------------------------------ */
static double decode_e4m3(uint8_t x)
{
    int sign = x >> 7;
    int e = (x >> 3) & 15;
    int m = x & 7;
    if (e == 15 && m == 7) return NAN;
    double v = e == 0 ? ldexp((double)m / 8.0, -6) : ldexp(1.0 + (double)m / 8.0, e - 7);
    return sign ? -v : v;
}

/* Cache row of key j of sequence b, kv head k, or -1 on a bad page id. */
static int64_t cache_row(const oracle_shape* s, const int32_t* page_table, int b, int k, int64_t j)
{
    int64_t slot = j / s->page_size;
    if (slot >= s->max_pages_per_seq) return -1;
    int32_t phys = page_table[(int64_t)b * s->max_pages_per_seq + slot];
    if (phys < 0 || phys >= s->num_pages) return -1;
    return ((int64_t)phys * s->num_kv_heads + k) * s->page_size + j % s->page_size;
}

/* decode_e4m3 of every code, filled once. */
static double e4m3_table[256];
static pthread_once_t e4m3_once = PTHREAD_ONCE_INIT;
static void fill_e4m3_table(void)
{
    for (int c = 0; c < 256; ++c) e4m3_table[c] = decode_e4m3((uint8_t)c);
}

static int fp8_key(const row_job* J, int64_t r, double* dst)
{
    const oracle_shape* s = J->s;
    const int d8 = s->qk_depth - J->rope_depth;
    const double ks = J->kscale ? (double)J->kscale[r] : 1.0;
    const uint8_t* src = J->k8 + r * d8;
    for (int d = 0; d < d8; ++d) dst[d] = ks * e4m3_table[src[d]];
    for (int d = 0; d < J->rope_depth; ++d) dst[d8 + d] = widen_bf16(J->krope[r * J->rope_depth + d]);
    return 0;
}

static int fp8_value(const row_job* J, int64_t r, double* dst)
{
    const oracle_shape* s = J->s;
    if (s->v_in_k) {
        const int d8 = s->qk_depth - J->rope_depth;
        const double ks = J->kscale ? (double)J->kscale[r] : 1.0;
        for (int d = 0; d < s->ov_depth; ++d) dst[d] = ks * e4m3_table[J->k8[r * d8 + d]];
    } else {
        for (int d = 0; d < s->ov_depth; ++d) dst[d] = e4m3_table[J->v8[r * s->ov_depth + d]];
    }
    return 0;
}

/* plain_row over the fp8 cache; kbuf holds qk_depth doubles, vbuf ov_depth. */
static int plain_row_fp8(row_job* J, int b, int t, int h, double* o, double* lse_out, double* sbuf,
                         double* kbuf, double* vbuf)
{
    const oracle_shape* s = J->s;
    int group = s->num_q_heads / s->num_kv_heads;
    int k = h / group;
    int64_t L = J->lens[b];
    int64_t n_vis = L - s->num_q + t + 1;
    for (int d = 0; d < s->ov_depth; ++d) o[d] = 0.0;
    if (n_vis <= 0) {
        if (lse_out) *lse_out = -INFINITY;
        return 0;
    }
    const uint16_t* qrow = J->q + (((int64_t)b * s->num_q + t) * s->num_q_heads + h) * s->qk_depth;
    double m = -INFINITY;
    for (int64_t j = 0; j < n_vis; ++j) {
        int64_t r = cache_row(s, J->pt, b, k, j);
        if (r < 0) return -1;
        fp8_key(J, r, kbuf);
        double acc = 0.0;
        for (int d = 0; d < s->qk_depth; ++d) acc += widen_bf16(qrow[d]) * kbuf[d];
        sbuf[j] = J->scale * acc;
        if (sbuf[j] > m) m = sbuf[j];
    }
    double l = 0.0;
    for (int64_t j = 0; j < n_vis; ++j) {
        double e = exp(sbuf[j] - m);
        l += e;
        int64_t r = cache_row(s, J->pt, b, k, j);
        fp8_value(J, r, vbuf);
        for (int d = 0; d < s->ov_depth; ++d) o[d] += e * vbuf[d];
    }
    for (int d = 0; d < s->ov_depth; ++d) o[d] /= l;
    if (lse_out) *lse_out = m + log(l);
    return 0;
}

static void* fp8_worker(void* arg)
{
    row_job* J = (row_job*)arg;
    const oracle_shape* s = J->s;
    int64_t max_len = 0;
    for (int b = 0; b < s->batch; ++b)
        if (J->lens[b] > max_len) max_len = J->lens[b];
    double* sbuf = (double*)malloc(sizeof(double) * (size_t)(max_len > 0 ? max_len : 1));
    double* kbuf = (double*)malloc(sizeof(double) * (size_t)s->qk_depth);
    double* vbuf = (double*)malloc(sizeof(double) * (size_t)s->ov_depth);
    if (!sbuf || !kbuf || !vbuf) { J->failed = 1; free(sbuf); free(kbuf); free(vbuf); return NULL; }
    int64_t total = J->rows ? J->n_rows : (int64_t)s->batch * s->num_q * s->num_q_heads;
    for (int64_t i = J->tid; i < total; i += J->nthreads) {
        int b, t, h;
        if (J->rows) {
            b = J->rows[3 * i];
            t = J->rows[3 * i + 1];
            h = J->rows[3 * i + 2];
            if (b < 0 || b >= s->batch || t < 0 || t >= s->num_q || h < 0 || h >= s->num_q_heads) {
                J->failed = 1;
                break;
            }
        } else {
            h = (int)(i % s->num_q_heads);
            t = (int)((i / s->num_q_heads) % s->num_q);
            b = (int)(i / ((int64_t)s->num_q_heads * s->num_q));
        }
        if (plain_row_fp8(J, b, t, h, J->out + i * s->ov_depth, J->lse ? J->lse + i : NULL, sbuf, kbuf, vbuf)) {
            J->failed = 1;
            break;
        }
    }
    free(sbuf);
    free(kbuf);
    free(vbuf);
    return NULL;
}

int oracle_decode_fp8(const oracle_shape* s, int rope_depth, double scale, const uint16_t* q,
                      const uint8_t* k8, const uint8_t* v8, const uint16_t* k_rope, const float* k_scale,
                      const int32_t* page_table, const int32_t* seq_lens,
                      const int32_t* rows, int64_t n_rows,
                      double* out, double* lse, int num_threads)
{
    if (!shape_ok(s) || !q || !k8 || (!v8 && !s->v_in_k) || !page_table || !seq_lens || !out) return -1;
    if (rope_depth < 0 || rope_depth >= s->qk_depth || (rope_depth > 0 && !k_rope)) return -1;
    if (s->v_in_k && s->ov_depth > s->qk_depth - rope_depth) return -1;
    if (rows && n_rows < 0) return -1;
    if (!lens_ok(s, seq_lens)) return -1;
    pthread_once(&e4m3_once, fill_e4m3_table);
    row_job proto;
    memset(&proto, 0, sizeof proto);
    proto.s = s;
    proto.scale = scale;
    proto.q = q;
    proto.k8 = k8;
    proto.v8 = v8;
    proto.krope = k_rope;
    proto.kscale = k_scale;
    proto.rope_depth = rope_depth;
    proto.pt = page_table;
    proto.lens = seq_lens;
    proto.rows = rows;
    proto.n_rows = n_rows;
    proto.out = out;
    proto.lse = lse;
    return run_jobs(&proto, fp8_worker, num_threads);
}

/* One E4M3 code widened (for the pins). */
double oracle_e4m3_value(int code) { return decode_e4m3((uint8_t)code); }

int oracle_hardware_threads(void)
{
    long n = sysconf(_SC_NPROCESSORS_ONLN);
    return n > 0 ? (int)n : 1;
}
