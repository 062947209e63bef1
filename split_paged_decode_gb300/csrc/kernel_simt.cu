// kernel_simt.cu -- the warp-level FMA decode kernel (sm_103a).
//
// One CTA = one cluster rank p of one (sequence, kv head[, row block]).
// Warp roles:
//   warps 0..3  compute: S = Q K^T over a tile of BN keys, online softmax in
//               exp2 form with the running (max, sum) in raw score units,
//               correction of O when the max moves, O += P V;
//   warp 4      load: walks the page table and issues TMA tile loads of K and
//               V (128-byte swizzled, one box per 64 columns and per page
//               segment) into a STAGES-deep shared-memory ring guarded by
//               full / empty mbarriers.
// After the key loop the CTA stages its normalised partial O and (max, sum),
// and the cluster merges them (splitk_combine.cuh).
//
// Geometry follows the FA4Config page (Modular MAX docs): GQA rows of one kv
// head fused into one tile (field group, method BM_eff), paged K/V addressed
// as block_idx * stride rows (method v_row_major), the split-K cluster
// (field splitk_partitions, methods cluster_size and with_splitk), and for
// the latent layout K_nope and V sharing one shared-memory stage (field
// use_shared_kv, method shared_kv_cols).
#include "fa_decode_internal.h"
#include "fp8.cuh"
#include "splitk_combine.cuh"

namespace fad {

// FP8: the E4M3 cache in the latent layout (FA4Config page: qkv_dtype E4M3,
// scale_dtype_ for the per-token K scale, rope_dtype_ for a bf16 rope part):
// a key row is D8 = DK - ROPE E4M3 codes (scaled by the key's K scale)
// followed by ROPE bf16 rope values (unscaled) from a cache of their own, and
// V is the first DV dequantized codes of the same row.
template <int DK, int DV, int BN, int STAGES, int RB, bool LATENT, bool FP8 = false, int ROPE = 0>
struct SimtCfg {
    static constexpr int NCW = 4;                   // compute warps
    static constexpr int NCT = NCW * 32;            // compute threads
    static constexpr int THREADS = NCT + 32;        // + one load warp
    static constexpr int D8 = FP8 ? DK - ROPE : 0;  // E4M3 columns of a key row
    static constexpr int K8BOX = D8 / 128;          // their 128-column (128-byte) TMA boxes
    static constexpr int RBOX = ROPE / 64;          // 64-column bf16 boxes of the rope part
    static constexpr int KBOX = FP8 ? K8BOX + RBOX : DK / 64;  // TMA boxes per K row
    static constexpr int VBOX = DV / 64;
    static constexpr int K_BYTES = KBOX * BN * 128;
    static constexpr int V_BYTES = LATENT ? 0 : VBOX * BN * 128;
    static constexpr int TILE_BYTES = K_BYTES + V_BYTES;  // bytes a stage's TMA boxes bring
    static constexpr int SC_BYTES = FP8 ? BN * 4 : 0;     // FP8: the tile's per-key K scales, after the boxes
    static constexpr int STAGE_BYTES = (TILE_BYTES + SC_BYTES + 1023) / 1024 * 1024;
    // Region offsets. Every region starts on 128 bytes; those a TMA copy
    // touches (the K/V ring and the bf16 output band) start on 1024 bytes.
    static constexpr int align_up(int x, int a) { return (x + a - 1) / a * a; }
    static constexpr int OFF_Q = STAGES * STAGE_BYTES;                         // float [RB][DK]
    static constexpr int OFF_S = align_up(OFF_Q + RB * DK * 4, 128);          // float [RB][BN]
    static constexpr int OFF_ALPHA = align_up(OFF_S + RB * BN * 4, 128);      // float [RB]
    static constexpr int OFF_MAXSUM = align_up(OFF_ALPHA + RB * 4, 128);      // float2 [RB]
    static constexpr int OFF_STAGE = align_up(OFF_MAXSUM + RB * 8, 128);      // float [RB][DV]
    static constexpr int OFF_OUT = align_up(OFF_STAGE + RB * DV * 4, 1024);   // bf16 [RB][DV]
    static constexpr int OFF_BAR = align_up(OFF_OUT + RB * DV * 2, 128);      // full[S], empty[S], publish
    static constexpr int OFF_FLAG = OFF_BAR + (2 * STAGES + 1) * 8;           // abort flag, consumed count
    static constexpr int SMEM_BYTES = OFF_FLAG + 16 + 1024;                    // + base alignment slack
    static_assert(STAGE_BYTES % 1024 == 0 && OFF_OUT % 1024 == 0, "TMA regions on 1024 bytes");

    // QK^T mapping: thread -> (key kk = t % BN, row group rg = t / BN)
    static constexpr int QK_GROUPS = NCT / BN;
    static constexpr int QK_ROWS = (RB + QK_GROUPS - 1) / QK_GROUPS;
    // PV mapping: thread -> (4-column chunks, row lane)
    static constexpr int NCH = DV / 4;
    static constexpr int PV_ROW_LANES = NCH >= NCT ? 1 : NCT / NCH;
    static constexpr int PV_CHUNKS = NCH >= NCT ? NCH / NCT : 1;
    static constexpr int PV_ROWS = (RB + PV_ROW_LANES - 1) / PV_ROW_LANES;
    // softmax mapping: warp w owns rows w, w + NCW, ...
    static constexpr int SM_ROWS = (RB + NCW - 1) / NCW;

    static_assert(DK % 64 == 0 && DV % 64 == 0, "depths are whole 64-column boxes");
    static_assert(NCT % BN == 0 && BN % 32 == 0, "tile of keys must divide the compute threads");
    static_assert(NCH % NCT == 0 || NCT % NCH == 0, "column chunks must tile the threads");
    static_assert(!LATENT || DV <= DK, "latent V is a prefix of the K row");
    static_assert(!FP8 || (LATENT && D8 % 128 == 0 && ROPE % 64 == 0 && DV <= D8 && DV % 128 == 0),
                  "E4M3: the latent layout, whole 128-column code boxes, V inside the codes");
    static_assert(SMEM_BYTES <= 232448, "shared memory budget of one CTA");
};

// Byte offset of element (row, col) inside a K or V tile held as 64-column,
// 128-byte-swizzled TMA boxes: box-major, then key row, 16-byte unit XOR row.
__device__ __forceinline__ uint32_t swz_offset(int row, int col, int bn)
{
    const int box = col >> 6;
    const int unit = (col & 63) >> 3;
    return (uint32_t)((box * bn + row) * 128 + ((unit ^ (row & 7)) << 4) + (col & 7) * 2);
}

// The same for one-byte (E4M3) elements: 128-column boxes.
__device__ __forceinline__ uint32_t swz8_offset(int row, int col, int bn)
{
    const int box = col >> 7;
    const int unit = (col & 127) >> 4;
    return (uint32_t)((box * bn + row) * 128 + ((unit ^ (row & 7)) << 4) + (col & 15));
}

// Four E4M3 codes, in memory order, as four floats (exact: every E4M3 value
// is a half value).
__device__ __forceinline__ float4 e4m3x4_to_float4(uint32_t w)
{
    const float2 a = __half22float2(__half2(__nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)(w & 0xffffu), __NV_E4M3)));
    const float2 b = __half22float2(__half2(__nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)(w >> 16), __NV_E4M3)));
    return make_float4(a.x, a.y, b.x, b.y);
}

template <int DK, int DV, int BN, int STAGES, int RB, bool LATENT, bool FP8 = false, int ROPE = 0>
__global__ void __launch_bounds__(SimtCfg<DK, DV, BN, STAGES, RB, LATENT, FP8, ROPE>::THREADS, 1)
    simt_decode_kernel(const __grid_constant__ DecodeParams p)
{
    using C = SimtCfg<DK, DV, BN, STAGES, RB, LATENT, FP8, ROPE>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
    const uint32_t sbase = smem_addr(smem);

    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;
    const int P = p.splitk;
    const int rank = (int)blockIdx.x;  // cluster dims are (P, 1, 1) and gridDim.x == P
    const int kvh = (int)blockIdx.y / p.row_blocks;
    const int row_block = (int)blockIdx.y % p.row_blocks;
    const int b = (int)blockIdx.z;
    grid_dependency_wait();  // inputs may come from the previous kernel in the stream
    grid_dependency_launch();

    int L = p.seq_lens[b];
    if (L < 0) {
        if (tid == 0 && rank == 0) atomicOr(p.status, FA_STATUS_BAD_PAGE);
        L = 0;
    }
    // Ragged batches launch once per cluster size; a cluster keeps only the
    // sequences whose length asks for its size (uniform across the cluster).
    if (p.auto_split && auto_split_for_len(L) != P) return;

    float* q_s = reinterpret_cast<float*>(smem + C::OFF_Q);
    float* s_s = reinterpret_cast<float*>(smem + C::OFF_S);
    float* alpha_s = reinterpret_cast<float*>(smem + C::OFF_ALPHA);
    float2* maxsum_s = reinterpret_cast<float2*>(smem + C::OFF_MAXSUM);
    float* stage_s = reinterpret_cast<float*>(smem + C::OFF_STAGE);
    uint16_t* out_s = reinterpret_cast<uint16_t*>(smem + C::OFF_OUT);
    const uint32_t full_bar = sbase + C::OFF_BAR;
    const uint32_t empty_bar = full_bar + 8 * STAGES;
    const uint32_t publish_bar = full_bar + 16 * STAGES;
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_FLAG);
    volatile int* consumed_s = abort_flag + 1;  // tiles the compute warps finished waiting for

    if (tid == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(full_bar + 8 * s, 1);
            mbar_init(empty_bar + 8 * s, C::NCW);
        }
        mbar_init(publish_bar, P);
        *abort_flag = 0;
        *consumed_s = 0;
        fence_mbarrier_init_cluster();
    }
    if (warp == C::NCW && lane == 0) {
        tma_prefetch_map(&p.tm_k);
        if (!LATENT) tma_prefetch_map(&p.tm_v);
    }

    // Q rows of this CTA -> fp32 in shared memory (rows >= p.rows are zero).
    // Row r is token r / heads_per_cta, head kvh*g + row_block*heads_per_cta + r % heads_per_cta.
    if (warp < C::NCW) {
        const uint32_t* q32 = reinterpret_cast<const uint32_t*>(p.q);
        for (int idx = tid; idx < RB * DK / 2; idx += C::NCT) {
            const int r = idx / (DK / 2);
            const int d2 = idx % (DK / 2);
            float2 v = make_float2(0.f, 0.f);
            if (r < p.rows) {
                const int t = r / p.heads_per_cta;
                const int h = kvh * p.group + row_block * p.heads_per_cta + r % p.heads_per_cta;
                v = bf16x2_to_float2(q32[(((int64_t)b * p.num_q + t) * p.num_q_heads + h) * (DK / 2) + d2]);
            }
            q_s[r * DK + 2 * d2] = v.x;
            q_s[r * DK + 2 * d2 + 1] = v.y;
        }
    }
    __syncthreads();
    if (P > 1) cluster_arrive_relaxed();  // waited before the merge publishes to peers

    // This rank's share of the key tiles: whole BN-key tiles split evenly,
    // the remainder going to the low ranks (an empty share is allowed).
    const int n_tiles = (L + BN - 1) / BN;
    const int base = n_tiles / P, rem = n_tiles % P;
    const int tile_begin = rank * base + min(rank, rem);
    const int tile_count = base + (rank < rem ? 1 : 0);

    // Running softmax state (owned by the softmax lanes) and the O accumulator.
    float m_run[C::SM_ROWS], l_run[C::SM_ROWS];
#pragma unroll
    for (int k = 0; k < C::SM_ROWS; ++k) {
        m_run[k] = -INFINITY;
        l_run[k] = 0.f;
    }
    float acc[C::PV_ROWS][C::PV_CHUNKS][4];
#pragma unroll
    for (int k = 0; k < C::PV_ROWS; ++k)
#pragma unroll
        for (int ch = 0; ch < C::PV_CHUNKS; ++ch)
#pragma unroll
            for (int e = 0; e < 4; ++e) acc[k][ch][e] = 0.f;

    int issued = 0;  // tiles whose loads the load lane has issued
    if (warp == C::NCW) {
        // ------------------------------------------------------------ load warp
        if (lane == 0 && !(p.debug_flags & FA_DEBUG_SKIP_LOADS)) {
            const uint64_t policy = l2_policy_evict_first();
            const int segs = BN / p.box_rows;
            for (int i = 0; i < tile_count; ++i) {
                const int s = i % STAGES;
                if (i >= STAGES &&
                    !mbar_wait(empty_bar + 8 * s, ((i / STAGES) & 1) ^ 1, abort_flag, p.status, p.wait_limit_ns))
                    break;
                const int key0 = (tile_begin + i) * BN;
                const uint32_t dst = sbase + s * C::STAGE_BYTES;
                // Cache row of page segment seg of this tile (the zero-fill row
                // past the sequence or on a bad page, which is flagged).
                auto seg_row = [&](int seg) -> int32_t {
                    const int key = key0 + seg * p.box_rows;
                    int32_t row = p.oob_row;
                    if (key < L) {
                        const int slot = key / p.page_size;
                        const int phys = slot < p.max_pages ? p.page_table[(int64_t)b * p.max_pages + slot] : -1;
                        if (phys >= 0 && phys < p.num_pages)
                            row = (phys * p.num_kv_heads + kvh) * p.page_size + key % p.page_size;
                        else
                            atomicOr(p.status, FA_STATUS_BAD_PAGE);
                    }
                    return row;
                };
                if constexpr (FP8) {
                    // The E4M3 boxes, the bf16 rope boxes and, with K scales, one
                    // bulk copy of each segment's scales (zeros, written before the
                    // arrive that publishes them, for a zero-fill segment).
                    int32_t rows[BN / 8];  // segs <= BN / 8: page_size is a multiple of 8
                    uint32_t sc_bytes = 0;
                    float* sc_s = reinterpret_cast<float*>(smem + s * C::STAGE_BYTES + C::TILE_BYTES);
                    for (int seg = 0; seg < segs; ++seg) {
                        rows[seg] = seg_row(seg);
                        if (p.k_scale != nullptr) {
                            if (rows[seg] != p.oob_row)
                                sc_bytes += (uint32_t)(p.box_rows * 4);
                            else
                                for (int r = 0; r < p.box_rows; ++r) sc_s[seg * p.box_rows + r] = 0.f;
                        }
                    }
                    // Zeros written here may later be overwritten by a bulk copy into this stage.
                    if (p.k_scale != nullptr) fence_proxy_async_smem();
                    mbar_arrive_expect_tx(full_bar + 8 * s, (uint32_t)C::TILE_BYTES + sc_bytes);
                    issued = i + 1;
                    for (int seg = 0; seg < segs; ++seg) {
                        const int32_t row = rows[seg];
                        const uint32_t seg_off = seg * p.box_rows * 128;
#pragma unroll
                        for (int c = 0; c < C::K8BOX; ++c)
                            tma_load_2d(dst + c * BN * 128 + seg_off, &p.tm_k, c * 128, row, full_bar + 8 * s,
                                        policy);
#pragma unroll
                        for (int c = 0; c < C::RBOX; ++c)
                            tma_load_2d(dst + (C::K8BOX + c) * BN * 128 + seg_off, &p.tm_rope, c * 64, row,
                                        full_bar + 8 * s, policy);
                        if (p.k_scale != nullptr && row != p.oob_row)
                            bulk_load(dst + C::TILE_BYTES + seg * p.box_rows * 4, p.k_scale + row,
                                      (uint32_t)(p.box_rows * 4), full_bar + 8 * s);
                    }
                } else {
                    mbar_arrive_expect_tx(full_bar + 8 * s, C::TILE_BYTES);
                    issued = i + 1;
                    for (int seg = 0; seg < segs; ++seg) {
                        const int32_t row = seg_row(seg);
                        const uint32_t seg_off = seg * p.box_rows * 128;
#pragma unroll
                        for (int c = 0; c < C::KBOX; ++c)
                            tma_load_2d(dst + c * BN * 128 + seg_off, &p.tm_k, c * 64, row, full_bar + 8 * s, policy);
                        if (!LATENT) {
#pragma unroll
                            for (int c = 0; c < C::VBOX; ++c)
                                tma_load_2d(dst + C::K_BYTES + c * BN * 128 + seg_off, &p.tm_v, c * 64, row,
                                            full_bar + 8 * s, policy);
                        }
                    }
                }
            }
        }
    } else {
        // --------------------------------------------------------- compute warps
        const int kk = tid % BN;           // QK^T: this thread's key within the tile
        const int rg = tid / BN;           // ... and its row group
        const int pv_lane = tid % (C::NCH >= C::NCT ? C::NCT : C::NCH);
        const int pv_row0 = tid / (C::NCH >= C::NCT ? C::NCT : C::NCH);
        const float c2 = p.scale_log2e;

        for (int i = 0; i < tile_count; ++i) {
            const int s = i % STAGES;
            mbar_wait(full_bar + 8 * s, (i / STAGES) & 1, abort_flag, p.status, p.wait_limit_ns);
            // Also orders the previous tile's P V reads before this tile's S writes.
            // The abort decision is reduced over the compute threads, so it is uniform.
            if (named_barrier_or(1, C::NCT, *abort_flag != 0)) break;
            if (tid == 0) *consumed_s = i + 1;
            const uint8_t* kt = smem + s * C::STAGE_BYTES;
            const uint8_t* vt = LATENT ? kt : kt + C::K_BYTES;
            const float* sc_s = reinterpret_cast<const float*>(kt + C::TILE_BYTES);  // FP8: per-key K scales
            const bool scaled = FP8 && p.k_scale != nullptr;
            const int key0 = (tile_begin + i) * BN;

            // ---- S = Q K^T for key kk, rows rg + QK_GROUPS * k (raw units, masked)
            {
                float sacc[C::QK_ROWS];
#pragma unroll
                for (int k = 0; k < C::QK_ROWS; ++k) sacc[k] = 0.f;
                if constexpr (FP8) {
                    // E4M3 part (16 codes per 16-byte unit), times the key's scale
#pragma unroll 2
                    for (int cc = 0; cc < C::D8 / 16; ++cc) {
                        const uint4 kw = *reinterpret_cast<const uint4*>(kt + swz8_offset(kk, cc * 16, BN));
                        const float4 k0 = e4m3x4_to_float4(kw.x), k1 = e4m3x4_to_float4(kw.y);
                        const float4 k2 = e4m3x4_to_float4(kw.z), k3 = e4m3x4_to_float4(kw.w);
#pragma unroll
                        for (int k = 0; k < C::QK_ROWS; ++k) {
                            const int r = rg + C::QK_GROUPS * k;
                            if (C::QK_ROWS * C::QK_GROUPS > RB && r >= RB) continue;
                            const float4* qv = reinterpret_cast<const float4*>(q_s + r * DK + cc * 16);
                            const float4 qa = qv[0], qb = qv[1], qc = qv[2], qd = qv[3];
                            float a = sacc[k];
                            a = fmaf(qa.x, k0.x, a);
                            a = fmaf(qa.y, k0.y, a);
                            a = fmaf(qa.z, k0.z, a);
                            a = fmaf(qa.w, k0.w, a);
                            a = fmaf(qb.x, k1.x, a);
                            a = fmaf(qb.y, k1.y, a);
                            a = fmaf(qb.z, k1.z, a);
                            a = fmaf(qb.w, k1.w, a);
                            a = fmaf(qc.x, k2.x, a);
                            a = fmaf(qc.y, k2.y, a);
                            a = fmaf(qc.z, k2.z, a);
                            a = fmaf(qc.w, k2.w, a);
                            a = fmaf(qd.x, k3.x, a);
                            a = fmaf(qd.y, k3.y, a);
                            a = fmaf(qd.z, k3.z, a);
                            a = fmaf(qd.w, k3.w, a);
                            sacc[k] = a;
                        }
                    }
                    if (scaled) {
                        const float ks = sc_s[kk];
#pragma unroll
                        for (int k = 0; k < C::QK_ROWS; ++k) sacc[k] *= ks;
                    }
                }
                // bf16 columns: the whole row, or (FP8) the rope part after the codes
                constexpr int BF_COLS = FP8 ? ROPE : DK;
                constexpr int BF_Q0 = FP8 ? C::D8 : 0;        // its first column in Q
                constexpr int BF_OFF = FP8 ? C::K8BOX * BN * 128 : 0;  // its first box in the stage
#pragma unroll 2
                for (int cc = 0; cc < BF_COLS / 8; ++cc) {
                    const uint4 kw = *reinterpret_cast<const uint4*>(kt + BF_OFF + swz_offset(kk, cc * 8, BN));
                    const float2 k01 = bf16x2_to_float2(kw.x), k23 = bf16x2_to_float2(kw.y);
                    const float2 k45 = bf16x2_to_float2(kw.z), k67 = bf16x2_to_float2(kw.w);
#pragma unroll
                    for (int k = 0; k < C::QK_ROWS; ++k) {
                        const int r = rg + C::QK_GROUPS * k;
                        if (C::QK_ROWS * C::QK_GROUPS > RB && r >= RB) continue;
                        const float4 qa = *reinterpret_cast<const float4*>(q_s + r * DK + BF_Q0 + cc * 8);
                        const float4 qb = *reinterpret_cast<const float4*>(q_s + r * DK + BF_Q0 + cc * 8 + 4);
                        float a = sacc[k];
                        a = fmaf(qa.x, k01.x, a);
                        a = fmaf(qa.y, k01.y, a);
                        a = fmaf(qa.z, k23.x, a);
                        a = fmaf(qa.w, k23.y, a);
                        a = fmaf(qb.x, k45.x, a);
                        a = fmaf(qb.y, k45.y, a);
                        a = fmaf(qb.z, k67.x, a);
                        a = fmaf(qb.w, k67.y, a);
                        sacc[k] = a;
                    }
                }
                const int key = key0 + kk;
#pragma unroll
                for (int k = 0; k < C::QK_ROWS; ++k) {
                    const int r = rg + C::QK_GROUPS * k;
                    if (r >= RB) continue;
                    const int t = r / p.heads_per_cta;
                    const int n_vis = L - p.num_q + t + 1;  // causal at the cache tail
                    s_s[r * BN + kk] = (r < p.rows && key < n_vis) ? sacc[k] : -INFINITY;
                }
            }
            named_barrier_sync(1, C::NCT);

            // ---- online softmax per row (warp-owned rows), exp2 form
#pragma unroll
            for (int k = 0; k < C::SM_ROWS; ++k) {
                const int r = warp + C::NCW * k;
                if (r >= RB) continue;
                float v[BN / 32];
                float tmax = -INFINITY;
#pragma unroll
                for (int j = 0; j < BN / 32; ++j) {
                    v[j] = s_s[r * BN + lane + 32 * j];
                    tmax = fmaxf(tmax, v[j]);
                }
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, o));
                const float m_new = fmaxf(m_run[k], tmax);
                float alpha = 1.f, psum = 0.f;
                if (m_new != -INFINITY) {
                    alpha = (m_run[k] == -INFINITY) ? 0.f : ex2_approx((m_run[k] - m_new) * c2);
#pragma unroll
                    for (int j = 0; j < BN / 32; ++j) {
                        const float pj = (v[j] == -INFINITY) ? 0.f : ex2_approx((v[j] - m_new) * c2);
                        psum += pj;
                        s_s[r * BN + lane + 32 * j] = pj;
                    }
                } else {
#pragma unroll
                    for (int j = 0; j < BN / 32; ++j) s_s[r * BN + lane + 32 * j] = 0.f;
                }
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) psum += __shfl_xor_sync(0xffffffffu, psum, o);
                l_run[k] = l_run[k] * alpha + psum;
                m_run[k] = m_new;
                if (lane == 0) alpha_s[r] = alpha;
            }
            named_barrier_sync(1, C::NCT);

            // ---- correction and O += P V for rows pv_row0 + PV_ROW_LANES * k
#pragma unroll
            for (int k = 0; k < C::PV_ROWS; ++k) {
                const int r = pv_row0 + C::PV_ROW_LANES * k;
                if (r >= RB) continue;
                const float a = alpha_s[r];
#pragma unroll
                for (int ch = 0; ch < C::PV_CHUNKS; ++ch)
#pragma unroll
                    for (int e = 0; e < 4; ++e) acc[k][ch][e] *= a;
            }
            const int j_end = min(BN, L - key0);  // rows past L_b never enter P V
#pragma unroll 2
            for (int j = 0; j < j_end; ++j) {
                float pr[C::PV_ROWS];
                const float vs = scaled ? sc_s[j] : 1.f;  // FP8 latent V: the key's scale, on P
#pragma unroll
                for (int k = 0; k < C::PV_ROWS; ++k) {
                    const int r = pv_row0 + C::PV_ROW_LANES * k;
                    pr[k] = (r < RB) ? s_s[r * BN + j] * vs : 0.f;
                }
#pragma unroll
                for (int ch = 0; ch < C::PV_CHUNKS; ++ch) {
                    const int col = (pv_lane + ch * C::NCT) * 4;
                    float2 v01, v23;
                    if constexpr (FP8) {
                        const float4 v = e4m3x4_to_float4(*reinterpret_cast<const uint32_t*>(vt + swz8_offset(j, col, BN)));
                        v01 = make_float2(v.x, v.y);
                        v23 = make_float2(v.z, v.w);
                    } else {
                        const uint2 vw = *reinterpret_cast<const uint2*>(vt + swz_offset(j, col, BN));
                        v01 = bf16x2_to_float2(vw.x);
                        v23 = bf16x2_to_float2(vw.y);
                    }
#pragma unroll
                    for (int k = 0; k < C::PV_ROWS; ++k) {
                        acc[k][ch][0] = fmaf(pr[k], v01.x, acc[k][ch][0]);
                        acc[k][ch][1] = fmaf(pr[k], v01.y, acc[k][ch][1]);
                        acc[k][ch][2] = fmaf(pr[k], v23.x, acc[k][ch][2]);
                        acc[k][ch][3] = fmaf(pr[k], v23.y, acc[k][ch][3]);
                    }
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(empty_bar + 8 * s);  // this warp is done with the stage
        }

        // ---- stage the normalised partial O and (max, sum)
        if (lane == 0) {
#pragma unroll
            for (int k = 0; k < C::SM_ROWS; ++k) {
                const int r = warp + C::NCW * k;
                if (r < RB) maxsum_s[r] = make_float2(m_run[k], l_run[k]);
            }
        }
        named_barrier_sync(1, C::NCT);
        const int BW = p.band_cols;
#pragma unroll
        for (int k = 0; k < C::PV_ROWS; ++k) {
            const int r = pv_row0 + C::PV_ROW_LANES * k;
            if (r >= RB) continue;
            const float l = maxsum_s[r].y;
            float inv = 0.f;
            if (l > 0.f) inv = __frcp_rn(l);
#pragma unroll
            for (int ch = 0; ch < C::PV_CHUNKS; ++ch) {
                const int col = (pv_lane + ch * C::NCT) * 4;
                const int q = col / BW, j = col % BW;
                *reinterpret_cast<float4*>(stage_s + (q * RB + r) * BW + j) =
                    make_float4(acc[k][ch][0] * inv, acc[k][ch][1] * inv, acc[k][ch][2] * inv,
                                acc[k][ch][3] * inv);
            }
        }
    }

    __syncthreads();  // staging complete (all warps; the load warp is idle here)
    if (P > 1) cluster_wait();  // every rank's publish barrier is initialised
    if (warp < C::NCW) {
        splitk_merge_and_store<RB>(p, P, rank, b, kvh, row_block, stage_s, maxsum_s, out_s, publish_bar, 0,
                                   0, abort_flag, tid, C::NCT, 1);
    } else if (lane == 0 && *abort_flag) {
        // Gave up early: let copies already issued, but never consumed, land
        // before the CTA exits (each wait again bounded).
        volatile int keep_waiting = 0;
        for (int i = *consumed_s; i < issued; ++i)
            mbar_wait(full_bar + 8 * (i % STAGES), (i / STAGES) & 1, &keep_waiting, p.status, p.wait_limit_ns);
    }
    __syncwarp();
    if (P > 1) cluster_sync_all();  // peers may still read this CTA's staged bands until here
}

// ---------------------------------------------------------------------------
// Variants and their geometry
// ---------------------------------------------------------------------------
template <int DK, int DV, int BN, int STAGES, int RB, bool LATENT, bool FP8 = false, int ROPE = 0>
static bool fill_geometry(KernelGeometry* g, const char* name)
{
    using C = SimtCfg<DK, DV, BN, STAGES, RB, LATENT, FP8, ROPE>;
    g->func = reinterpret_cast<const void*>(&simt_decode_kernel<DK, DV, BN, STAGES, RB, LATENT, FP8, ROPE>);
    g->threads = C::THREADS;
    g->keys_per_tile = BN;
    g->stages = STAGES;
    g->rows_capacity = RB;
    g->smem_bytes = C::SMEM_BYTES;
    g->name = name;
    return true;
}

bool simt_geometry(int qk, int ov, bool latent, int rb, KernelGeometry* g)
{
#define FAD_SIMT(DK, DV, BN, ST, RB, LAT, SUFFIX)                                              \
    if (qk == DK && ov == DV && latent == LAT && rb == RB)                                      \
        return fill_geometry<DK, DV, BN, ST, RB, LAT>(                                          \
            g, "simt_d" #DK "_v" #DV "_bn" #BN "_s" #ST "_r" #RB SUFFIX);
    FAD_SIMT(64, 64, 64, 4, 4, false, "")
    FAD_SIMT(64, 64, 64, 4, 8, false, "")
    FAD_SIMT(64, 64, 64, 4, 16, false, "")
    FAD_SIMT(128, 128, 64, 4, 4, false, "")
    FAD_SIMT(128, 128, 64, 4, 8, false, "")
    FAD_SIMT(128, 128, 64, 4, 16, false, "")
    FAD_SIMT(576, 512, 32, 3, 16, true, "_latent")
    FAD_SIMT(576, 512, 32, 2, 16, false, "")
#undef FAD_SIMT
    return false;
}

bool simt_fp8_latent_geometry(int qk, int ov, int rope, int rb, KernelGeometry* g)
{
    // MLA: 512 E4M3 latent columns (V = all of them) and a 64-column bf16 rope.
    if (qk == 576 && ov == 512 && rope == 64 && rb == 16)
        return fill_geometry<576, 512, 32, 4, 16, true, true, 64>(g, "simt_e4m3_d576_r64_v512_bn32_s4_r16_latent");
    return false;
}

}  // namespace fad
