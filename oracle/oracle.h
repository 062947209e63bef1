/*
 * oracle.h -- interface of the fp64 CPU oracle for paged decode attention.
 *
 * TEST INFRASTRUCTURE ONLY: this header and oracle.c are used by the tests,
 * by the smoke check and by the CPU-baseline leg of the benchmark. The
 * library under split_paged_decode_gb300/ neither includes nor links them,
 * and they include nothing from it.
 */
#ifndef SPD_ORACLE_H
#define SPD_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Shape of one decode call. All tensors are dense, row-major, bf16 bit
 * patterns carried as uint16:
 *   q          [batch][num_q][num_q_heads][qk_depth]
 *   k_pages    [num_pages][num_kv_heads][page_size][qk_depth]
 *   v_pages    [num_pages][num_kv_heads][page_size][ov_depth]
 *              (ignored when v_in_k: V is then the first ov_depth columns
 *               of the K row, the MLA latent layout)
 *   page_table [batch][max_pages_per_seq] int32 physical page ids
 *   seq_lens   [batch] int32, the KV length L_b including the num_q new tokens
 */
typedef struct oracle_shape {
    int batch;
    int num_q;
    int num_q_heads;
    int num_kv_heads;
    int qk_depth;
    int ov_depth;
    int page_size;
    int max_pages_per_seq;
    int num_pages;
    int v_in_k;
} oracle_shape;

/* Plain softmax attention, one pass per query row, fp64 throughout.
 * rows == NULL: every (b, t, h); out is [batch][num_q][num_q_heads][ov_depth],
 * lse is [batch][num_q][num_q_heads].
 * rows != NULL: n_rows triples (b, t, h); out is [n_rows][ov_depth], lse
 * [n_rows]. lse may be NULL. Returns 0, or -1 on a bad argument (page id out
 * of range, non-divisible heads, ...). num_threads <= 0 means 1. */
int oracle_decode(const oracle_shape* s, double scale, const uint16_t* q,
                  const uint16_t* k_pages, const uint16_t* v_pages,
                  const int32_t* page_table, const int32_t* seq_lens,
                  const int32_t* rows, int64_t n_rows,
                  double* out, double* lse, int num_threads);

/* The same result reached through an explicit split of the key axis and the
 * log-sum-exp combine. bounds is [batch][num_parts + 1], non-decreasing key
 * positions; partition p of sequence b covers keys [bounds[p], bounds[p+1]).
 * Every (b, t, h) is computed; out / lse as for oracle_decode with rows ==
 * NULL. part_max / part_sum, when not NULL, receive each partition's running
 * max (raw q.k units) and exp2-sum, [batch][num_q][num_q_heads][num_parts]. */
int oracle_partitioned(const oracle_shape* s, double scale, const uint16_t* q,
                       const uint16_t* k_pages, const uint16_t* v_pages,
                       const int32_t* page_table, const int32_t* seq_lens,
                       const int32_t* bounds, int num_parts,
                       double* out, double* lse,
                       double* part_max, double* part_sum, int num_threads);

/* Plain attention over an fp8 (OCP E4M3) cache, fp64 throughout. The shape's
 * qk_depth is the full key width: an E4M3 part of qk_depth - rope_depth
 * columns, dequantized with the per-token K scale, then rope_depth bf16
 * columns (unscaled). Layouts, with r = (page * Hkv + kv head) * PS + j % PS:
 *   k8       uint8 [num_pages][Hkv][PS][qk_depth - rope_depth]
 *   v8       uint8 [num_pages][Hkv][PS][ov_depth], NULL for the latent layout
 *            (V = the first ov_depth dequantized values of the E4M3 part)
 *   k_rope   bf16 bits [num_pages][Hkv][PS][rope_depth], NULL if rope_depth 0
 *   k_scale  float [num_pages][Hkv][PS], NULL for all ones
 * rows / out / lse as for oracle_decode. Returns 0 or -1 on a bad argument. */
int oracle_decode_fp8(const oracle_shape* s, int rope_depth, double scale, const uint16_t* q,
                      const uint8_t* k8, const uint8_t* v8, const uint16_t* k_rope, const float* k_scale,
                      const int32_t* page_table, const int32_t* seq_lens,
                      const int32_t* rows, int64_t n_rows,
                      double* out, double* lse, int num_threads);

/* The value of one E4M3 code (0..255) as the fp8 oracle reads it. */
double oracle_e4m3_value(int code);

/* Threads the host offers (sysconf), for reporting the baseline's core count. */
int oracle_hardware_threads(void);

#ifdef __cplusplus
}
#endif

#endif
