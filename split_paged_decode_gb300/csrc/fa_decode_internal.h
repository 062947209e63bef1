// fa_decode_internal.h -- types shared by the host planner and the kernels of
// libfa_decode.so (not installed; the public interface is include/fa_decode.h).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "fa_decode.h"

namespace fad {

constexpr uint64_t kDefaultWaitLimitNs = 1000000000ull;  // one second
constexpr int kMaxSplit = 16;

// Per-sequence split rule for splitk == 0: short sequences keep one CTA per
// (sequence, kv head), longer ones spread over 2 or 4.
__host__ __device__ inline int auto_split_for_len(int len)
{
    return len <= 1024 ? 1 : (len <= 4096 ? 2 : 4);
}

// Stream-K partition of `total` tiles over `clusters` ranges: the first tile
// of cluster c's range, and the cluster whose range holds tile x (the largest
// c with sk_begin(c) <= x).
__host__ __device__ inline int64_t sk_begin(int64_t total, int clusters, int64_t c)
{
    return c * total / clusters;
}
__host__ __device__ inline int sk_cluster_of(int64_t total, int clusters, int64_t x)
{
    return (int)(((x + 1) * clusters + total - 1) / total - 1);
}

// Everything a decode kernel needs, passed by value as a __grid_constant__
// parameter block (the tensor maps must live in parameter, constant or global
// memory for TMA to read them).
struct DecodeParams {
    CUtensorMap tm_k;    // K rows: [num_pages*Hkv*PS][Dk] bf16, box {64, box_rows}, 128B swizzle
    CUtensorMap tm_v;    // V rows: [num_pages*Hkv*PS][Dv] (unused for the latent layout)
    CUtensorMap tm_out;  // out: 3-D {Dv, Hq, B*T} bf16, box {out_chunk_cols, heads_per_cta, tokens_per_cta}
    CUtensorMap tm_rope; // E4M3 latent cache: the bf16 rope rows [num_pages*Hkv*PS][rope], box {64, box_rows}
    const uint16_t* q;   // bf16 bits [B][T][Hq][Dk]
    const int32_t* page_table;
    const int32_t* seq_lens;
    float* lse;
    unsigned int* status;
    int batch, num_q, num_q_heads, num_kv_heads, group;
    int qk_depth, ov_depth, page_size, max_pages, num_pages;
    int rows;            // real query rows per CTA (T*g, or heads_per_cta when row-blocked)
    int row_blocks;      // CTAs along grid y per kv head
    int heads_per_cta;   // heads covered by one CTA (g, or the row-block size)
    int tokens_per_cta;  // tokens covered by one CTA (T, or 1 when row-blocked)
    int splitk;          // cluster size P of this launch
    int auto_split;      // 1: a cluster works on sequence b only if auto_split_for_len(L_b) == P
    int dyn_split;       // 1: per-sequence split in one launch of 4-CTA clusters (tcgen05 shallow ring)
    int box_rows;        // key rows per K/V TMA box: min(page_size, keys per tile)
    int band_cols;       // output columns owned by one cluster rank: Dv / P
    int out_chunk_cols;  // columns per output TMA store box: min(band_cols, 256); Dv / 4 under dyn_split
    int32_t oob_row;     // a row coordinate past the end of the cache views (zero fill)
    float scale, scale_log2e;
    uint32_t debug_flags;
    uint64_t wait_limit_ns;
    unsigned long long* trace;  // per-CTA timeline (FA_TRACE_WORDS_PER_CTA words each) or NULL
    int64_t trace_ctas;         // CTAs the trace buffer holds
    // Stream-K partition (sk_tiles > 0; the deep-ring kernel only, when the
    // units alone would leave resident clusters idle): each unit's key range
    // counts as sk_tiles tiles of 128 keys (a full page-table row), the units'
    // ranges are laid end to end (sk_total = units * sk_tiles) and cluster c
    // of sk_clusters takes tiles [c * sk_total / G, (c + 1) * sk_total / G):
    // the end of one unit and the start of the next at most. A unit whose
    // range several clusters share is merged over DSMEM per cluster as usual;
    // each cluster's normalised band and (max, sum) go to chunk_o / chunk_ms
    // (slot 2c or 2c + 1: the cluster's first or second unit) and the last
    // cluster to count in (chunk_count, which it resets) merges the chunks.
    int sk_tiles;
    int sk_clusters;
    int64_t sk_total;
    float* chunk_o;             // [slot][P][band_cols][rows_capacity]
    float2* chunk_ms;           // [slot][P][rows_capacity]: (max, sum) in raw score units
    unsigned int* chunk_count;  // [slot][P]: per shared unit, at its first cluster's slot; zero between launches
    // fp8 cache: per-token K scales, float [num_pages * Hkv * PS] (the cache
    // row index), or NULL for unit scales.
    const float* k_scale;
};

// Geometry of one compiled kernel variant, for planning and validation.
struct KernelGeometry {
    const void* func;    // the __global__ function
    int threads;
    int keys_per_tile;   // BN
    int stages;
    int rows_capacity;   // RB: query rows one CTA holds
    int smem_bytes;
    const char* name;
};

// Kernel variants of the SIMT (warp-level FMA) path. Returns false when no
// variant exists for (qk, ov, latent, rows_capacity).
bool simt_geometry(int qk_depth, int ov_depth, bool latent, int rows_capacity, KernelGeometry* g);
// The SIMT kernel over an E4M3 latent cache (V = the first ov dequantized
// codes of the key row) whose last rope_depth key columns come from a bf16
// cache of their own. Returns false when no variant exists.
bool simt_fp8_latent_geometry(int qk_depth, int ov_depth, int rope_depth, int rows_capacity, KernelGeometry* g);

// Kernel variants of the tcgen05 path (head dim 128, <= 16 rows per CTA) with
// a ring of `nslot` 32 KB K/V tile slots; stream_k selects the variant of the
// deep ring that takes the stream-K partition.
bool tc_geometry(int qk_depth, int ov_depth, int rows, int nslot, bool stream_k, KernelGeometry* g);
// The same kernel over an fp8 (OCP E4M3) cache: nslot counts 32 KB of ring
// (twice as many 16 KB E4M3 tile slots).
bool tc_fp8_geometry(int qk_depth, int ov_depth, int rows, int nslot, bool stream_k, KernelGeometry* g);
// The tcgen05 kernel of the MLA latent layout (qk 576 = nope 512 + rope 64,
// ov 512, V = the latent rows' first 512 columns) for num_q == 1 and a
// multiple of 64 heads per kv head: 64 heads per CTA.
bool mla_tc_geometry(int qk_depth, int ov_depth, int nope_depth, int heads_per_kv, int num_q, KernelGeometry* g);
// The same kernel over the E4M3 latent cache: 512 codes per row with a
// per-token K scale, the 64 rope columns from a bf16 cache of their own.
bool mla_tc_fp8_geometry(int qk_depth, int ov_depth, int nope_depth, int rope_depth, int heads_per_kv, int num_q,
                         KernelGeometry* g);
// The stream-K partition is used only while every cluster rank keeps at
// least this many 128-key tiles of its range.
constexpr int kChunkMinTilesPerRank = 4;
constexpr int kTcSlotsShared = 3;  // two CTAs per SM (grids of more than one wave)
constexpr int kTcSlotsAlone = 6;   // one CTA per SM, 192 KB of loads in flight

}  // namespace fad
