// splitk_combine.cuh -- the cluster split-K epilogue of the SIMT kernels and
// the GQA tcgen05 kernel: publish this CTA's partial result, merge all
// partitions' results for this CTA's band of output columns over distributed
// shared memory, cast to bf16 and TMA-store the band.
//
// Follows the fa4_splitk_combine_write page (Modular MAX docs): pass 2 is a
// reduce-scatter in which cluster rank p owns the output column band
// [p * Dv / P, (p + 1) * Dv / P); it reads every rank's (max, sum) and every
// rank's normalised partial O for its band, forms
//   Gmax = max_q max_q,  Gsum = sum_q sum_q * exp2((max_q - Gmax) * c),
//   w_q  = sum_q * exp2((max_q - Gmax) * c) / Gsum,  O = sum_q w_q * O_q,
// (c = scale * log2 e; the sum_q factor cancels each partial's own
// normalisation) and stores its band. One publish barrier (an mbarrier that
// every rank arrives on remotely, released at cluster scope) makes the staged
// partials visible before the remote reads; no second cluster barrier is
// needed because the bf16 band is packed into a buffer no peer reads, and the
// kernel's terminal cluster barrier keeps every rank's staged bands alive
// until all ranks have finished reading them.
#pragma once

#include "device_common.cuh"

namespace fad {

// Layout contract with the kernels:
//   stage_s  float [P][RB][BW]: rank-local normalised partial O, band-major
//            (element (r, col) at ((col / BW) * RB + r) * BW + col % BW)
//   maxsum_s float2 [RB]: (max in raw q.k units, sum of exp2((s - max) * c));
//            an empty partition holds (-inf, 0)
//   out_s    bf16 [BW / OC][RB][OC]: this rank's packed band in store boxes of
//            OC = min(BW, 256) columns, rows r = t * heads + hh
// Rows >= p.rows are padding: they are merged (harmlessly) but never stored.
//
// Called by `nthreads` threads with ids `tid` in [0, nthreads), after a
// barrier of the group that follows the staging writes, and (P > 1) after a
// cluster barrier wait that guarantees every rank has initialised its
// publish barrier. Thread tid 0 of the calling group publishes. `bar_id`
// names a hardware barrier private to the group.
//
// A kernel that merges several units in turn with the same buffers passes
// the parity of this unit's publish phase and a `stage_free_bar` (count P):
// once this rank has read every peer's stage (its own included), it arrives
// on that barrier in every rank, and a rank rewrites its stage for the next
// unit only after its own barrier has completed the phase. A peer's publish for unit n + 1 then
// cannot reach a rank before that rank's unit-n phase has completed (it would
// need that rank's reads of the peer's unit-n stage), so one publish barrier
// alternates parity safely. stage_free_bar == 0: a single unit, no arrivals.
//
// The P partitions are the cluster ranks rbase .. rbase + P - 1 (rbase > 0
// when a cluster serves several units of a smaller split; `rank` is this
// CTA's index among them), each owning bw = Dv / P output columns (bw 0: the
// launch's band width).
template <int RB>
__device__ __forceinline__ void splitk_merge_and_store(const DecodeParams& p, int P, int rank, int b,
                                                       int kvh, int row_block, const float* stage_s,
                                                       const float2* maxsum_s, uint16_t* out_s,
                                                       uint32_t publish_bar, uint32_t publish_parity,
                                                       uint32_t stage_free_bar, volatile int* abort_flag,
                                                       int tid, int nthreads, uint32_t bar_id, int rbase = 0,
                                                       int bw = 0)
{
    const int BW = bw > 0 ? bw : p.band_cols;
    const float c = p.scale_log2e;
    const uint32_t stage_base = smem_addr(stage_s);
    const uint32_t maxsum_base = smem_addr(maxsum_s);

    if (P > 1) {
        if (tid == 0) {
            // Round 1: every rank tells every rank (itself included) that its
            // stage is complete. The preceding CTA barrier orders the other
            // threads' staging writes before this release.
            for (int q = 0; q < P; ++q) mbar_arrive_cluster(map_shared_rank(publish_bar, rbase + q));
        }
        mbar_wait<true>(publish_bar, publish_parity, abort_flag, p.status, p.wait_limit_ns);
    }

    const int chunks = BW / 4;
    if (P <= 4) {
        // Up to four partitions (the per-sequence split): every partition's
        // (max, sum) and band values of an item are loaded before any is used,
        // so the remote reads are in flight together; the sums keep partition
        // order and skip empty partitions as the general loop below does.
        for (int it = tid; it < RB * chunks; it += nthreads) {
            const int r = it / chunks;
            const int j = (it % chunks) * 4;
            const uint32_t off = 4u * ((uint32_t)(rank * RB + r) * BW + j);
            float2 ms[4];
            float4 v[4];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const int qq = rbase + min(q, P - 1);
                ms[q] = (P > 1) ? ld_dsmem_f2(map_shared_rank(maxsum_base + 8u * r, qq)) : maxsum_s[r];
                v[q] = (P > 1) ? ld_dsmem_f4(map_shared_rank(stage_base + off, qq))
                               : *reinterpret_cast<const float4*>(stage_s + (rank * RB + r) * BW + j);
            }
            float gmax = -INFINITY;
#pragma unroll
            for (int q = 0; q < 4; ++q)
                if (q < P && ms[q].y > 0.f) gmax = fmaxf(gmax, ms[q].x);
            float wq[4];
            float gsum = 0.f;
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                wq[q] = (q < P && ms[q].y > 0.f) ? ms[q].y * ex2_approx((ms[q].x - gmax) * c) : 0.f;
                gsum += wq[q];
            }
            const float inv = gsum > 0.f ? 1.f / gsum : 0.f;
            float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                if (wq[q] > 0.f) {
                    const float w = wq[q] * inv;
                    o.x = fmaf(w, v[q].x, o.x);
                    o.y = fmaf(w, v[q].y, o.y);
                    o.z = fmaf(w, v[q].z, o.z);
                    o.w = fmaf(w, v[q].w, o.w);
                }
            }
            uint2 packed = make_uint2(float2_to_bf16x2(o.x, o.y), float2_to_bf16x2(o.z, o.w));
            const int OC = p.out_chunk_cols;
            *reinterpret_cast<uint2*>(out_s + ((j / OC) * RB + r) * OC + j % OC) = packed;
            if (rank == 0 && j == 0 && r < p.rows && p.lse != nullptr) {
                const int t = r / p.heads_per_cta;
                const int h = kvh * p.group + row_block * p.heads_per_cta + r % p.heads_per_cta;
                const float lse = gsum > 0.f ? p.scale * gmax + lg2_approx(gsum) * 0.6931471805599453f
                                             : -INFINITY;
                p.lse[((int64_t)b * p.num_q + t) * p.num_q_heads + h] = lse;
            }
        }
    } else
    for (int it = tid; it < RB * chunks; it += nthreads) {
        const int r = it / chunks;
        const int j = (it % chunks) * 4;
        float mq[kMaxSplit], wq[kMaxSplit];
        float gmax = -INFINITY;
        for (int q = 0; q < P; ++q) {
            float2 ms = (P > 1) ? ld_dsmem_f2(map_shared_rank(maxsum_base + 8u * r, rbase + q)) : maxsum_s[r];
            mq[q] = ms.x;
            wq[q] = ms.y;
            if (ms.y > 0.f) gmax = fmaxf(gmax, ms.x);
        }
        float gsum = 0.f;
        for (int q = 0; q < P; ++q) {
            float w = 0.f;
            if (wq[q] > 0.f) w = wq[q] * ex2_approx((mq[q] - gmax) * c);
            wq[q] = w;
            gsum += w;
        }
        const float inv = gsum > 0.f ? 1.f / gsum : 0.f;
        float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
        const uint32_t off = 4u * ((uint32_t)(rank * RB + r) * BW + j);
        for (int q = 0; q < P; ++q) {
            if (wq[q] <= 0.f) continue;
            float4 v = (P > 1) ? ld_dsmem_f4(map_shared_rank(stage_base + off, rbase + q))
                               : *reinterpret_cast<const float4*>(stage_s + (rank * RB + r) * BW + j);
            const float w = wq[q] * inv;
            o.x = fmaf(w, v.x, o.x);
            o.y = fmaf(w, v.y, o.y);
            o.z = fmaf(w, v.z, o.z);
            o.w = fmaf(w, v.w, o.w);
        }
        uint2 packed = make_uint2(float2_to_bf16x2(o.x, o.y), float2_to_bf16x2(o.z, o.w));
        const int OC = p.out_chunk_cols;
        *reinterpret_cast<uint2*>(out_s + ((j / OC) * RB + r) * OC + j % OC) = packed;

        if (rank == 0 && j == 0 && r < p.rows && p.lse != nullptr) {
            const int t = r / p.heads_per_cta;
            const int h = kvh * p.group + row_block * p.heads_per_cta + r % p.heads_per_cta;
            // natural-log LSE of the scaled scores: scale * Gmax + ln(Gsum)
            const float lse = gsum > 0.f ? p.scale * gmax + lg2_approx(gsum) * 0.6931471805599453f
                                         : -INFINITY;
            p.lse[((int64_t)b * p.num_q + t) * p.num_q_heads + h] = lse;
        }
    }

    // bf16 band complete in shared memory -> one TMA store of the band.
    fence_proxy_async_smem();
    named_barrier_sync(bar_id, nthreads);
    if (tid == 0) {
        // Every thread's remote reads are complete (their values are in the
        // band); release the peers' stages for their next unit.
        if (stage_free_bar != 0) {
            if (P > 1)
                for (int q = 0; q < P; ++q) mbar_arrive_cluster(map_shared_rank(stage_free_bar, rbase + q));
            else
                mbar_arrive(stage_free_bar);
        }
        const int OC = p.out_chunk_cols;
        for (int c0 = 0; c0 < BW; c0 += OC)
            tma_store_3d(&p.tm_out, smem_addr(out_s + (c0 / OC) * RB * OC), rank * BW + c0,
                         kvh * p.group + row_block * p.heads_per_cta, b * p.num_q);
        tma_store_commit();
        tma_store_wait_read();  // the band's shared memory may be released once read
    }
}

// ---------------------------------------------------------------------------
// Push variant (the multi-unit tcgen05 kernel). Pulling peers' partials with
// remote loads needs a release at cluster scope on the publishing side, and
// on a CTA whose loads are streaming such a release waits microseconds for
// the copies in flight. Here every rank instead pushes, from registers, the
// columns of its normalised partial O that each band owner needs, plus its
// per-row (max, sum), into the owner's receive buffer with st.async; the
// bytes complete on the owner's recv_full barrier, so the owner merges from
// its own shared memory once that barrier's phase completes.
//
// Receive buffer of rank q, one per buffer index:
//   recv_o  float  [P][BW][RB]: rank p's partial, column c of q's band, row r
//           at ((p * BW + c) * RB + r)
//   recv_ms float2 [P][RB]:     rank p's (max, sum) of row r
// Bytes expected per unit: P * BW * RB * 4 + P * RB * 8.
// ---------------------------------------------------------------------------
__host__ __device__ constexpr int pushed_bytes(int P, int BW, int RB) { return P * BW * RB * 4 + P * RB * 8; }

// Row weights over the `nq` pushed partials (recv_ms [nq][RB]: raw max,
// sum; nq <= 2 kMaxSplit) by the whole warp: lane (row r = lane % RB, group
// g = lane / RB) takes partials g, g + G, ... (G = 32 / RB lanes per row),
// all its loads in flight together, and xor shuffles over the row's G lanes
// reduce Gmax (over the partials that saw keys) and Gsum. Writes
// w_q = sum_q * exp2((max_q - Gmax) * c) / Gsum (0 for an empty partial)
// into wtab [nq][RB]; every lane of row r returns (Gmax, Gsum).
template <int RB>
__device__ __forceinline__ float2 partial_weights(const float2* recv_ms, float* wtab, int nq, int lane, float c)
{
    static_assert(32 % RB == 0, "a row's lanes tile the warp");
    constexpr int G = 32 / RB;
    constexpr int K = (2 * kMaxSplit + G - 1) / G;  // partials per lane at most
    const int r = lane % RB, g = lane / RB;
    float2 m[K];
#pragma unroll
    for (int k = 0; k < K; ++k) {
        const int q = g + G * k;
        m[k] = q < nq ? recv_ms[q * RB + r] : make_float2(-INFINITY, 0.f);
    }
    float gmax = -INFINITY;
#pragma unroll
    for (int k = 0; k < K; ++k)
        if (m[k].y > 0.f) gmax = fmaxf(gmax, m[k].x);
#pragma unroll
    for (int sh = RB; sh < 32; sh <<= 1) gmax = fmaxf(gmax, __shfl_xor_sync(0xffffffffu, gmax, sh));
    float gsum = 0.f;
#pragma unroll
    for (int k = 0; k < K; ++k) {
        m[k].y = m[k].y > 0.f ? m[k].y * ex2_approx((m[k].x - gmax) * c) : 0.f;
        gsum += m[k].y;
    }
#pragma unroll
    for (int sh = RB; sh < 32; sh <<= 1) gsum += __shfl_xor_sync(0xffffffffu, gsum, sh);
    const float inv = gsum > 0.f ? 1.f / gsum : 0.f;
#pragma unroll
    for (int k = 0; k < K; ++k) {
        const int q = g + G * k;
        if (q < nq) wtab[q * RB + r] = m[k].y * inv;
    }
    return make_float2(gmax, gsum);
}

// Lanes of a band of BW columns (a power of two): PG = 32 / BW lanes per
// column when BW < 32 (each takes every PG-th partial), else one; lane's
// first column, column step and partial group.
struct BandLanes {
    int col0, step, pg, PG;
};
__device__ __forceinline__ BandLanes band_lanes(int BW, int lane)
{
    const int PG = BW < 32 ? 32 / BW : 1, per = 32 / PG;
    return BandLanes{lane % per, per, lane / per, PG};
}

// o[RB] = sum over the nq partials of w_q * (partial q's column `col`)
// (recv_o [nq][BW][RB]; weights wtab [nq][RB]), the partials pg, pg + PG,
// ... on this lane, four per round with their loads in flight together; with
// PG > 1 xor shuffles add the column's PG lanes, so each of them ends with
// the total. Every lane of the warp calls it the same number of times.
template <int RB>
__device__ __forceinline__ void partial_band(const float* recv_o, const float* wtab, int nq, int BW, int col,
                                             const BandLanes& bl, float (&o)[RB])
{
#pragma unroll
    for (int r = 0; r < RB; ++r) o[r] = 0.f;
    for (int q0 = bl.pg; q0 < nq; q0 += 4 * bl.PG) {
        float4 v[4][RB / 4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const float4* src =
                reinterpret_cast<const float4*>(recv_o + (min(q0 + j * bl.PG, nq - 1) * BW + col) * RB);
#pragma unroll
            for (int r4 = 0; r4 < RB / 4; ++r4) v[j][r4] = src[r4];
        }
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            if (q0 + j * bl.PG < nq) {
                const float4* wq = reinterpret_cast<const float4*>(wtab + (q0 + j * bl.PG) * RB);
#pragma unroll
                for (int r4 = 0; r4 < RB / 4; ++r4) {
                    const float4 w = wq[r4];
                    o[4 * r4 + 0] = fmaf(w.x, v[j][r4].x, o[4 * r4 + 0]);
                    o[4 * r4 + 1] = fmaf(w.y, v[j][r4].y, o[4 * r4 + 1]);
                    o[4 * r4 + 2] = fmaf(w.z, v[j][r4].z, o[4 * r4 + 2]);
                    o[4 * r4 + 3] = fmaf(w.w, v[j][r4].w, o[4 * r4 + 3]);
                }
            }
        }
    }
    for (int sh = 32 / bl.PG; sh < 32; sh <<= 1) {
#pragma unroll
        for (int r = 0; r < RB; ++r) o[r] += __shfl_xor_sync(0xffffffffu, o[r], sh);
    }
}

// Merge by one warp (`lane` 0..31) of the `nq` partials in this rank's
// receive buffer (one per rank, or one per (rank, softmax warpgroup)), cast,
// TMA store of the band and lse (rank 0). The caller has waited for the
// buffer's recv_full phase; it releases the buffer afterwards. `wtab` is
// float [nq][RB] of scratch for the combine weights.
template <int RB>
__device__ __forceinline__ void splitk_merge_pushed(const DecodeParams& p, int P, int rank, int b, int kvh,
                                                    const float* recv_o, const float2* recv_ms, float* wtab,
                                                    uint16_t* out_s, int lane, int nq)
{
    const int BW = p.band_cols;
    const float c = p.scale_log2e;
    // The previous unit's store of out_s must have read it.
    if (lane == 0) tma_store_wait_read();
    __syncwarp();
    // Per row: Gmax over the partitions that saw keys, Gsum, and the weights
    // w_q = sum_q * exp2((max_q - Gmax) * c) / Gsum (0 for an empty partition).
    {
        const float2 gm = partial_weights<RB>(recv_ms, wtab, nq, lane, c);
        const float gmax = gm.x, gsum = gm.y;
        const int r = lane;  // lanes 0 .. RB - 1 hold rows 0 .. RB - 1
        if (lane < RB && rank == 0 && r < p.rows && p.lse != nullptr) {
            const int t = r / p.heads_per_cta;
            const int h = kvh * p.group + r % p.heads_per_cta;
            // natural-log LSE of the scaled scores: scale * Gmax + ln(Gsum)
            p.lse[((int64_t)b * p.num_q + t) * p.num_q_heads + h] =
                gsum > 0.f ? p.scale * gmax + lg2_approx(gsum) * 0.6931471805599453f : -INFINITY;
        }
    }
    __syncwarp();
    const int OC = p.out_chunk_cols;
    const BandLanes bl = band_lanes(BW, lane);
    for (int col = bl.col0; col < BW; col += bl.step) {
        float o[RB];
        partial_band<RB>(recv_o, wtab, nq, BW, col, bl, o);
        if (bl.pg == 0) {
            __nv_bfloat16* dst = reinterpret_cast<__nv_bfloat16*>(out_s) + (col / OC) * RB * OC + col % OC;
#pragma unroll
            for (int r = 0; r < RB; ++r) dst[r * OC] = __float2bfloat16_rn(o[r]);
        }
    }
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) {
        for (int c0 = 0; c0 < BW; c0 += OC)
            tma_store_3d(&p.tm_out, smem_addr(out_s + (c0 / OC) * RB * OC), rank * BW + c0, kvh * p.group,
                         b * p.num_q);
        tma_store_commit();
    }
}

// The same merge for unit `u` under the stream-K partition, in the cluster
// `cluster`: when several clusters' ranges share the unit, the cluster's
// merged band is one chunk of it. The chunk (fp32, normalised, with the
// per-row Gmax and Gsum) goes to the scratch slot of (cluster, unit), and the
// last of the unit's clusters to count in for this band merges the chunks by
// the same rule one level up (in cluster order, so the result does not depend
// on which cluster comes last), stores the band and lse (rank 0) and resets
// the count. `wtab` is float [max(nq, 16)][RB]; a unit has at most 16 chunks.
template <int RB>
__device__ __noinline__ void splitk_merge_pushed_sk(const DecodeParams& p, int P, int rank, int b, int kvh, int u,
                                                    int cluster, const float* recv_o, const float2* recv_ms,
                                                    float* wtab, uint16_t* out_s, int lane, int nq)
{
    const int64_t Nv = p.sk_tiles, TOT = p.sk_total;
    const int G = p.sk_clusters;
    const int c_first = sk_cluster_of(TOT, G, (int64_t)u * Nv);
    const int S = sk_cluster_of(TOT, G, (int64_t)(u + 1) * Nv - 1) - c_first + 1;
    if (S == 1) {  // the unit lies in this cluster's range alone
        splitk_merge_pushed<RB>(p, P, rank, b, kvh, recv_o, recv_ms, wtab, out_s, lane, nq);
        return;
    }
    // Scratch slot of (cluster c, unit u): 2c, or 2c + 1 for the second unit
    // of c's range. Only the unit's first cluster can have started in an
    // earlier unit (every later one starts inside this unit).
    const int first_second = sk_begin(TOT, G, c_first) < (int64_t)u * Nv ? 1 : 0;
    auto slot = [&](int c) -> int64_t { return 2 * (int64_t)c + (c == c_first ? first_second : 0); };
    const int BW = p.band_cols;
    const float c = p.scale_log2e;
    const int64_t mine = slot(cluster);
    float* const my_o = p.chunk_o + (mine * P + rank) * BW * RB;
    // This chunk: weights over the cluster's pushed partials, then the band.
    {
        const float2 gm = partial_weights<RB>(recv_ms, wtab, nq, lane, c);
        if (lane < RB) p.chunk_ms[(mine * P + rank) * RB + lane] = gm;
    }
    __syncwarp();
    const BandLanes bl = band_lanes(BW, lane);
    for (int col = bl.col0; col < BW; col += bl.step) {
        float o[RB];
        partial_band<RB>(recv_o, wtab, nq, BW, col, bl, o);
        if (bl.pg == 0) {
            float4* dst = reinterpret_cast<float4*>(my_o + col * RB);
#pragma unroll
            for (int r4 = 0; r4 < RB / 4; ++r4)
                dst[r4] = make_float4(o[4 * r4], o[4 * r4 + 1], o[4 * r4 + 2], o[4 * r4 + 3]);
        }
    }
    // Publish this chunk's band (every lane's writes, then one count); the
    // cluster that completes the count reads every chunk's band.
    __threadfence();
    __syncwarp();
    // One count per shared unit, at its first cluster's slot for it (slots are
    // distinct across the shared units of a launch).
    unsigned int* count = p.chunk_count + slot(c_first) * P + rank;
    unsigned int last = 0;
    if (lane == 0) last = atomicAdd(count, 1u) == (unsigned int)(S - 1) ? 1u : 0u;
    if (!__shfl_sync(0xffffffffu, last, 0)) return;
    __threadfence();
    // The band below: lane takes (column, 4-row group) items. Its first
    // item's first four chunks are loaded now, in flight together with the
    // (max, sum) reads of the weights.
    const int items = BW * (RB / 4);
    auto chunk_item = [&](int k, int idx) -> float4 {
        const int col = idx / (RB / 4), r4 = idx % (RB / 4);
        return __ldcg(reinterpret_cast<const float4*>(
                          p.chunk_o + ((slot(c_first + min(k, S - 1)) * P + rank) * BW + col) * RB) +
                      r4);
    };
    float4 first[4];
    if (lane < items) {
#pragma unroll
        for (int j = 0; j < 4; ++j) first[j] = chunk_item(j, lane);
    }
    // Chunk weights per row (lane r < RB <= 16), every chunk's (max, sum) in
    // flight at once: these reads queue behind the streaming loads.
    if (lane < RB) {
        const int r = lane;
        // Loads without a guard (chunks past S read chunk S - 1 and are
        // dropped below), so that all of them are in flight at once.
        float2 ms[kMaxSplit];
#pragma unroll
        for (int k = 0; k < kMaxSplit; ++k)
            ms[k] = __ldcg(p.chunk_ms + (slot(c_first + min(k, S - 1)) * P + rank) * RB + r);
#pragma unroll
        for (int k = 0; k < kMaxSplit; ++k)
            if (k >= S) ms[k] = make_float2(-INFINITY, 0.f);
        float gmax = -INFINITY;
#pragma unroll
        for (int k = 0; k < kMaxSplit; ++k)
            if (ms[k].y > 0.f) gmax = fmaxf(gmax, ms[k].x);
        float wk[kMaxSplit];
        float gsum = 0.f;
#pragma unroll
        for (int k = 0; k < kMaxSplit; ++k) {
            wk[k] = ms[k].y > 0.f ? ms[k].y * ex2_approx((ms[k].x - gmax) * c) : 0.f;
            gsum += wk[k];
        }
        const float inv = gsum > 0.f ? 1.f / gsum : 0.f;
#pragma unroll
        for (int k = 0; k < kMaxSplit; ++k)
            if (k < S) wtab[k * RB + r] = wk[k] * inv;
        if (rank == 0 && r < p.rows && p.lse != nullptr) {
            const int t = r / p.heads_per_cta;
            const int h = kvh * p.group + r % p.heads_per_cta;
            p.lse[((int64_t)b * p.num_q + t) * p.num_q_heads + h] =
                gsum > 0.f ? p.scale * gmax + lg2_approx(gsum) * 0.6931471805599453f : -INFINITY;
        }
    }
    __syncwarp();
    if (lane == 0) {
        *count = 0u;            // every chunk of this launch has counted
        tma_store_wait_read();  // the previous unit's store has read out_s
    }
    __syncwarp();
    // The band: lane takes (column, 4-row group) pairs, every chunk's values
    // of a pair in flight at once.
    const int OC = p.out_chunk_cols;
    for (int idx = lane; idx < items; idx += 32) {
        const int col = idx / (RB / 4), r4 = idx % (RB / 4);
        // Four chunks per round, loaded without a guard (clamped to chunk
        // S - 1), so a round's loads are in flight at once.
        float o[4] = {0.f, 0.f, 0.f, 0.f};
        for (int k0 = 0; k0 < S; k0 += 4) {
            float4 v[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) v[j] = (idx == lane && k0 == 0) ? first[j] : chunk_item(k0 + j, idx);
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                if (k0 + j < S) {
                    const float4 w = *reinterpret_cast<const float4*>(wtab + (k0 + j) * RB + 4 * r4);
                    o[0] = fmaf(w.x, v[j].x, o[0]);
                    o[1] = fmaf(w.y, v[j].y, o[1]);
                    o[2] = fmaf(w.z, v[j].z, o[2]);
                    o[3] = fmaf(w.w, v[j].w, o[3]);
                }
            }
        }
        __nv_bfloat16* dst = reinterpret_cast<__nv_bfloat16*>(out_s) + (col / OC) * RB * OC + col % OC;
#pragma unroll
        for (int i = 0; i < 4; ++i) dst[(4 * r4 + i) * OC] = __float2bfloat16_rn(o[i]);
    }
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) {
        for (int c0 = 0; c0 < BW; c0 += OC)
            tma_store_3d(&p.tm_out, smem_addr(out_s + (c0 / OC) * RB * OC), rank * BW + c0, kvh * p.group,
                         b * p.num_q);
        tma_store_commit();
    }
}

}  // namespace fad
