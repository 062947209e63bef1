// kernel_mla_tc.cu -- the tcgen05 decode kernel for the MLA latent layout
// (sm_103a): qk = 576 (nope 512 + rope 64), ov = 512, V = the first 512
// columns of the same latent rows, many query heads per kv head.
//
// With 64 or more heads the fused tile is a dense contraction, so both
// products run on the tensor core with 64 heads per CTA on N and keys / value
// columns on M = 128:
//   S^T [128 keys x 64 heads]  = K_tile [128 x 576] . Q^T         (A, B K-major)
//   O^T [512 dv  x 64 heads]  += V_tile^T [512 x 128] . P^T        (A MN-major)
// O^T (256 TMEM columns: four 128-dv blocks x 64 heads) accumulates in tensor
// memory over the whole key range and is corrected in place only when the
// lazy-rescale vote moves a head's running max; S^T is double-buffered (two
// buffers of two accumulators). The 576-wide K tile streams through the ring
// as four 128-column items plus the 64-column rope item, and V as four
// 128-column items that re-read the same rows (they are still in L2).
//
// Warp roles (one CTA = one cluster rank of one (sequence, 64-head block)):
//   warp 0      load: page-table walk (warp-wide blocks of entries, a block
//               ahead) and TMA loads of the items into a ring of 4 x 32 KB
//               slots, tile by tile in the order K(0) K(1) V(0) K(2) V(1) ...
//   warp 1      MMA S: allocates the 512 TMEM columns, issues every S^T;
//   warp 2      MMA O: issues every O^T += V^T P^T; each MMA warp frees a
//               ring slot with a commit once the products that read it are done;
//   warps 3-10  softmax: two warpgroups, each owning 32 of the 64 heads
//               (thread = TMEM lane = key for S^T, = value column for O^T);
//               online softmax in exp2 form, P^T to shared memory as bf16,
//               in-place correction of O^T; then the split-K epilogue
//               over all 256 softmax threads: each rank pushes the other
//               bands' columns of its partial O from TMEM into their owners'
//               drained rings (st.async, distributed shared memory) and
//               combines its own band from TMEM with what it receives.
//
// Geometry follows the FA4Config page (Modular MAX docs): MLA depth split
// into nope and rope (q_nope / q_rope), one O accumulator for the wide V
// (single_o), V as the nope prefix of the shared latent row (use_shared_kv),
// split-K clusters (splitk_partitions).
//
// FP8: the E4M3 latent cache (FA4Config page: qkv_dtype E4M3, scale_dtype_
// for the per-token K scale, rope_dtype_ for the bf16 rope part). A key row
// is 512 codes, scaled by the key's K scale, followed by 64 bf16 rope values
// from a cache of their own; V is the 512 scaled codes. The code part of S^T
// is a kind::f8f6f4 product against Q^T carried as two E4M3 operands (16 h
// and l, fp8.cuh; each head scaled by a power of two sigma_h first) into one
// accumulator, the rope part a kind::f16 product into the other:
//   S = acc_codes / (16 sigma_h) * k_scale_j + acc_rope.
// O^T += V^T P'^T takes the codes as they are and P' = P k_scale_j / Sigma as
// two E4M3 operands (16 P' = h + l), where Sigma is a power of two above
// every K scale of the current tile (raised when a tile brings a larger
// scale, lowered when a tile's scales all lie 16x below it, with O corrected
// like a moved max; the scales are non-negative), so P' <= P and the O partial
// is acc Sigma / 16. The ring items carry twice the columns of a bf16 item: K as
// two 256-code items plus the rope item, V as two items; the per-token
// scales come in a ring of their own.
#include "fa_decode_internal.h"
#include "device_common.cuh"
#include "fp8.cuh"
#include "tcgen05.cuh"

namespace fad {

template <bool FP8>
struct MlaCfgT {
    static constexpr int ROWS = 64;                 // heads per CTA (N of both MMAs)
    static constexpr int BN = 128;                  // keys per tile (M of S^T)
    static constexpr int DK = 576, DV = 512;
    // Four 32 KB slots (in-flight bytes bound this kernel) leave room for one P buffer.
    static constexpr int NSLOT = 4;
    static constexpr int P_BUFS = 1;
    static constexpr int ATOM_BYTES = BN * 128;     // 16 KB: 64 columns of a tile
    static constexpr int SLOT_BYTES = 2 * ATOM_BYTES;
    // K: 4 x 128 columns + the 64-column rope (FP8: 2 x 256 codes + the rope);
    // V: 4 x 128 columns (FP8: 2 x 256 codes). An item is two 128-byte boxes
    // (one for the rope item).
    static constexpr int KITEMS = FP8 ? 3 : 5;
    static constexpr int VITEMS = FP8 ? 2 : 4;
    static constexpr int ITEM_COLS = FP8 ? 256 : 128;  // cache columns of a two-box item
    static constexpr float RESCALE = FP8 ? 4.0f : 8.0f;  // lazy rescale: P <= 2^RESCALE (FP8: 16 P' <= 448)
    static constexpr int KS = FP8 ? 4 : 0;          // FP8: per-token K scale ring entries (one tile each)
    static constexpr int Q_ATOM = ROWS * 128;       // 8 KB: 64 depth columns of the 64 heads (FP8: 128 codes)
    static constexpr int Q_BYTES = 9 * Q_ATOM;      // 72 KB
    static constexpr int P_ATOM = ROWS * 128;       // 8 KB: 64 keys of P^T
    static constexpr int P_BYTES = 2 * P_ATOM;      // 16 KB
    // TMEM: S^T [2 buffers][2 accumulators][64 columns] at 0, O^T [4 dv blocks][64 columns] at 256.
    static constexpr int S_ACC = 64, S_BUF = 2 * S_ACC, TMEM_S0 = 0, TMEM_O0 = 2 * S_BUF;
    static constexpr int TMEM_COLS = 512;
    static constexpr int WG0 = 3;                   // softmax warps 3-6 (heads 0-31), 7-10 (heads 32-63)
    static constexpr int THREADS = 32 * (WG0 + 8);  // 352

    static constexpr int OFF_RING = 0;                               // NSLOT x 32 KB
    static constexpr int OFF_Q = NSLOT * SLOT_BYTES;                 // 9 atoms [64 heads][128 B]
    static constexpr int OFF_P = OFF_Q + Q_BYTES;                    // [P_BUFS][2 atoms][64 heads][128 B]
    static constexpr int OFF_RED = OFF_P + P_BUFS * P_BYTES;         // float [2 warpgroups][4 quadrants][32]
    // barriers: slot_full[NSLOT], slot_empty[NSLOT], s_full[2], s_empty[2], p_full[2],
    // o_full[2], q_full, recv_ms, mma_done, tmem_ready, v_zeroed[4], recv_o, ready[kMaxSplit],
    // (FP8) ks_full[KS], ks_empty[KS]
    static constexpr int OFF_BAR = OFF_RED + 2 * 4 * 32 * 4;
    static constexpr int NBAR = 2 * NSLOT + 17 + kMaxSplit + 2 * KS;
    static constexpr int OFF_ROWS = OFF_BAR + NBAR * 8;              // int [4 tiles][16 segments]
    static constexpr int OFF_MISC = OFF_ROWS + 4 * 16 * 4;           // tmem base, abort, S next item, O next item
    // FP8: K scales float [KS][BN], 1 / (16 sigma_h) float [64], tile scale maxima float [2][4]
    static constexpr int OFF_KS = (OFF_MISC + 16 + 127) / 128 * 128;  // bulk copy destinations: 16-byte aligned
    static constexpr int OFF_QINV = OFF_KS + KS * BN * 4;
    static constexpr int OFF_SIG = OFF_QINV + (FP8 ? ROWS * 4 : 0);
    static constexpr int SMEM_BYTES = OFF_SIG + (FP8 ? 32 : 0) + 1024;
    // Split-K epilogue, once every product of the CTA has completed, over the
    // drained ring, Q and P: the partials the other ranks push for this
    // rank's band, f32 [P - 1][BW][64] (at most 15/16 of 128 KB), their rows' (max, sum) float2 [P - 1][64], the bf16 band
    // [BW / OC][64][OC] (at most 64 KB) and the combine weights float [P][64].
    static constexpr int OFF_RECV = 0;
    static constexpr int OFF_RECV_MS = ROWS * DV * 4;
    static constexpr int OFF_OUT = OFF_RECV_MS + 8192;
    static constexpr int OFF_WTAB = OFF_OUT + ROWS * DV * 2;
    static_assert((kMaxSplit - 1) * ROWS * 8 <= OFF_OUT - OFF_RECV_MS, "pushed row statistics fit");
    static_assert(OFF_WTAB + kMaxSplit * ROWS * 4 <= OFF_RED, "epilogue buffers fit below the softmax scratch");
    static_assert(OFF_Q % 1024 == 0 && OFF_P % 1024 == 0, "swizzle atoms on 1024 bytes");
    static_assert(OFF_KS % 16 == 0 && OFF_QINV % 16 == 0, "K scale copies and float4 reads");
    static_assert(SMEM_BYTES <= 232448, "dynamic shared memory per CTA");
};

// Item positions: a tile's K items form one group and its V items another;
// the groups come in the order K(0) K(1) V(0) K(2) V(1) ... K(n-1) V(n-2)
// V(n-1). Group position of tile i's K and tile t's V, and the index of the
// first item of the group at position g.
__device__ __forceinline__ int mla_k_group(int i) { return i == 0 ? 0 : 2 * i - 1; }
__device__ __forceinline__ int mla_v_group(int t, int n) { return t == n - 1 ? 2 * n - 1 : 2 * t + 2; }
template <bool FP8>
__device__ __forceinline__ int mla_group_item(int g, int n)
{
    const int nk = g == 0 ? 0 : min(n, (g + 2) / 2);  // K groups before position g
    return MlaCfgT<FP8>::KITEMS * nk + MlaCfgT<FP8>::VITEMS * (g - nk);
}

template <bool FP8>
__global__ void __launch_bounds__(MlaCfgT<FP8>::THREADS, 1) mla_tc_decode_kernel(const __grid_constant__ DecodeParams p)
{
    using C = MlaCfgT<FP8>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
    const uint32_t sbase = smem_addr(smem);

    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;
    const int P = p.splitk;
    const int rank = (int)blockIdx.x;
    const int kvh = (int)blockIdx.y / p.row_blocks;
    const int row_block = (int)blockIdx.y % p.row_blocks;
    const int b = (int)blockIdx.z;

    // Optional timeline trace (a profiling aid): one thread writes each event.
    const int64_t cta_lin = (int64_t)blockIdx.x + (int64_t)gridDim.x * (blockIdx.y + (int64_t)gridDim.y * blockIdx.z);
    unsigned long long* const trace =
        (p.trace != nullptr && cta_lin < p.trace_ctas) ? p.trace + cta_lin * FA_TRACE_WORDS_PER_CTA : nullptr;
    auto stamp = [&](int slot) {
        if (trace) trace[slot] = global_timer_ns();
    };
    if (tid == 0) stamp(0);
    grid_dependency_wait();  // inputs may come from the previous kernel in the stream
    grid_dependency_launch();

    int L = p.seq_lens[b];
    // The load warp's first block of page-table entries, read while the
    // length is in flight, guessing that the sequence fills its row (checked
    // once the length is known): the two reads overlap instead of following
    // one another. spec_raw -2: this lane read nothing.
    int spec_begin = -1, spec_count = 0, spec_raw = -2;
    if (warp == 0 && p.max_pages <= INT32_MAX / C::BN / p.page_size) {
        const int ntg = (p.max_pages * p.page_size + C::BN - 1) / C::BN;
        spec_begin = rank * (ntg / P) + min(rank, ntg % P);
        spec_count = ntg / P + (rank < ntg % P ? 1 : 0);
        const int segs = C::BN / p.box_rows;
        const int t = lane / segs;
        const int pslot = ((spec_begin + t) * C::BN + (lane % segs) * p.box_rows) / p.page_size;
        if (t < spec_count && pslot < p.max_pages) spec_raw = p.page_table[(int64_t)b * p.max_pages + pslot];
    }
    if (L < 0) {
        if (tid == 0 && rank == 0) atomicOr(p.status, FA_STATUS_BAD_PAGE);
        L = 0;
    }
    if (p.auto_split && auto_split_for_len(L) != P) return;  // uniform across the cluster

    const uint32_t bar0 = sbase + C::OFF_BAR;
    const uint32_t slot_full = bar0, slot_empty = bar0 + 8 * C::NSLOT;
    const uint32_t s_full = bar0 + 16 * C::NSLOT, s_empty = s_full + 16, p_full = s_full + 32, o_full = s_full + 48;
    const uint32_t q_full = s_full + 64, recv_ms_bar = s_full + 72, mma_done = s_full + 80, tmem_ready = s_full + 88;
    const uint32_t v_zeroed = s_full + 96;  // [4]: the last tile's V items with their rows past L zeroed
    // Split-K epilogue: the pushed partials' bytes land on recv_o_bar (and
    // their row statistics on recv_ms_bar); rank q arrives on ready[q] once
    // its drained ring may take this rank's pushes.
    const uint32_t recv_o_bar = s_full + 128, ready_bar = s_full + 136;
    // FP8 K scale ring: tile t's scales in entry t % KS (full: the copies landed;
    // empty: every softmax warp has read them).
    const uint32_t ks_full = s_full + 8 * (17 + kMaxSplit), ks_empty = ks_full + 8 * C::KS;
    const bool scaled = FP8 && p.k_scale != nullptr;
    volatile uint32_t* tmem_slot = reinterpret_cast<volatile uint32_t*>(smem + C::OFF_MISC);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 4);
    const uint32_t s_next = sbase + C::OFF_MISC + 8, o_next = sbase + C::OFF_MISC + 12;
    float* red_s = reinterpret_cast<float*>(smem + C::OFF_RED);

    if (tid == 0) {
        for (int s = 0; s < C::NSLOT; ++s) {
            mbar_init(slot_full + 8 * s, 1);
            mbar_init(slot_empty + 8 * s, 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(s_full + 8 * i, 1);
            mbar_init(s_empty + 8 * i, 8);  // one arrival per softmax warp
            mbar_init(p_full + 8 * i, 8);
            mbar_init(o_full + 8 * i, 1);
        }
        mbar_init(q_full, 8);
        mbar_init(recv_ms_bar, 1);
        mbar_init(recv_o_bar, 1);
        for (int q = 0; q < kMaxSplit; ++q) mbar_init(ready_bar + 8 * q, 1);
        mbar_init(mma_done, 2);
        mbar_init(tmem_ready, 1);
        for (int e = 0; e < C::VITEMS; ++e) mbar_init(v_zeroed + 8 * e, 8);
        for (int e = 0; e < C::KS; ++e) {
            mbar_init(ks_full + 8 * e, 1);
            mbar_init(ks_empty + 8 * e, 8);
        }
        *abort_flag = 0;
        // Next item of each kind to be consumed: K starts at item 0, V at the
        // first item of V(0) (no earlier item is a V item, and with 5-item K
        // groups on a 3-slot ring the S warp must not wait for one).
        const int nt = (L + C::BN - 1) / C::BN;
        const int tc0 = nt / P + (rank < nt % P ? 1 : 0);
        *reinterpret_cast<volatile uint32_t*>(smem + C::OFF_MISC + 8) = 0;
        *reinterpret_cast<volatile uint32_t*>(smem + C::OFF_MISC + 12) =
            tc0 > 0 ? (uint32_t)mla_group_item<FP8>(mla_v_group(0, tc0), tc0) : 0xffffffffu;
        fence_mbarrier_init_cluster();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_map(&p.tm_k);
        if (FP8) tma_prefetch_map(&p.tm_rope);
    }
    __syncthreads();
    if (P > 1) cluster_arrive_relaxed();
    uint32_t tmem = 0;
    if (warp == 1) {
        tmem_alloc(sbase + C::OFF_MISC, C::TMEM_COLS);
        tmem_relinquish();
        tc_fence_before_sync();
        __syncwarp();
        tc_fence_after_sync();
        tmem = *tmem_slot;
        if (lane == 0) mbar_arrive(tmem_ready);
    }

    const int n_tiles = (L + C::BN - 1) / C::BN;
    const int base_t = n_tiles / P, rem = n_tiles % P;
    const int tile_begin = rank * base_t + min(rank, rem);
    const int tile_count = base_t + (rank < rem ? 1 : 0);
    // The rank holding the sequence's last, partial tile zeroes its V rows past L.
    const bool v_tail = tile_count > 0 && (tile_begin + tile_count) * C::BN > L;

    int issued = 0;
    int ks_issued = 0;  // FP8: tiles whose K scale copies were issued
    // Softmax state of this thread's 32 heads.
    float m_run[32], l_part[32];

    if (warp == 0) {
        // ------------------------------------------------------------------ load warp
        if (!(p.debug_flags & FA_DEBUG_SKIP_LOADS)) {
            const uint64_t policy = l2_policy_evict_normal();  // V re-reads these rows from L2
            const int segs = C::BN / p.box_rows;               // page segments per tile: 1, 2, ..., 16
            const int tpb = 32 / segs;                         // tiles per block of page entries
            int32_t* rows_s = reinterpret_cast<int32_t*>(smem + C::OFF_ROWS);
            constexpr int kNoSegment = INT32_MIN, kPastSequence = INT32_MIN + 1;
            // raw >= -1: this lane's entry, already read
            auto block_entry = [&](int tb, int raw = -2) -> int {
                const int t = tb + lane / segs;
                if (t >= tile_count) return kNoSegment;
                const int key = (tile_begin + t) * C::BN + (lane % segs) * p.box_rows;
                if (key >= L) return kPastSequence;
                const int pslot = key / p.page_size;
                if (pslot >= p.max_pages) return -1;
                return raw >= -1 ? raw : p.page_table[(int64_t)b * p.max_pages + pslot];
            };
            // The guess holds when this rank's tiles start where it assumed (every
            // entry the first block needs was then read, at the same page slot).
            const bool guessed = tile_begin == spec_begin && tile_count <= spec_count;
            int blk_cur = block_entry(0, guessed ? spec_raw : -2), blk_next = block_entry(tpb);
            int jj = 0;
            bool ok = true;
            for (int g = 0; ok && g < 2 * tile_count; ++g) {
                // group g: K of tile t or V of tile t
                const bool is_v = (g == 2 * tile_count - 1) || (g > 0 && (g & 1) == 0);
                const int t = is_v ? (g == 2 * tile_count - 1 ? tile_count - 1 : (g - 2) >> 1) : (g + 1) >> 1;
                int32_t row;
                if (!is_v) {
                    if (t > 0 && (t & (tpb - 1)) == 0) {
                        blk_cur = blk_next;
                        blk_next = block_entry(t + tpb);
                    }
                    const int e = __shfl_sync(0xffffffffu, blk_cur, (t & (tpb - 1)) * segs + (lane & (segs - 1)));
                    row = p.oob_row;  // zero fill past the sequence or on a bad page
                    if (lane < segs) {
                        if (e >= 0 && e < p.num_pages) {
                            const int key = (tile_begin + t) * C::BN + lane * p.box_rows;
                            row = (e * p.num_kv_heads + kvh) * p.page_size + key % p.page_size;
                        } else if (e != kNoSegment && e != kPastSequence) {
                            atomicOr(p.status, FA_STATUS_BAD_PAGE);
                        }
                    }
                    if (lane < 16) rows_s[(t & 3) * 16 + lane] = row;
                    if (scaled) {
                        // Tile t's K scales, one bulk copy per page segment in the cache
                        // (none for a zero-filled segment: the softmax masks those keys).
                        const int kse = t % C::KS;
                        if (t >= C::KS) {
                            const bool got = mbar_wait(ks_empty + 8 * kse, ((t / C::KS) & 1) ^ 1, abort_flag,
                                                       p.status, p.wait_limit_ns);
                            if (!__all_sync(0xffffffffu, got)) {
                                ok = false;
                                break;
                            }
                        }
                        const bool copy = lane < segs && row != p.oob_row;
                        // Zeros for a zero-filled segment's keys (a bad page), written
                        // before the arrive that publishes the entry; a later copy into
                        // the entry follows the proxy fence.
                        float* ks_w = reinterpret_cast<float*>(smem + C::OFF_KS) + kse * C::BN;
                        for (int sg = 0; sg < segs; ++sg) {
                            const int32_t r_sg = __shfl_sync(0xffffffffu, row, sg);
                            if (lane == 0 && r_sg == p.oob_row)
                                for (int k = 0; k < p.box_rows; ++k) ks_w[sg * p.box_rows + k] = 0.f;
                        }
                        if (lane == 0) fence_proxy_async_smem();
                        const uint32_t n = __popc(__ballot_sync(0xffffffffu, copy));
                        if (lane == 0) mbar_arrive_expect_tx(ks_full + 8 * kse, n * (uint32_t)p.box_rows * 4u);
                        __syncwarp();
                        if (copy)
                            bulk_load(sbase + C::OFF_KS + (uint32_t)((kse * C::BN + lane * p.box_rows) * 4),
                                      p.k_scale + row, (uint32_t)p.box_rows * 4u, ks_full + 8 * kse);
                        ks_issued = t + 1;
                    }
                } else {
                    row = lane < 16 ? rows_s[(t & 3) * 16 + lane] : p.oob_row;
                }
                const int n_in = is_v ? C::VITEMS : C::KITEMS;
                for (int e = 0; e < n_in; ++e, ++jj) {
                    const int slot = jj % C::NSLOT;
                    if (jj >= C::NSLOT) {
                        const bool got = mbar_wait(slot_empty + 8 * slot, ((jj / C::NSLOT) & 1) ^ 1, abort_flag,
                                                   p.status, p.wait_limit_ns);
                        if (!__all_sync(0xffffffffu, got)) {
                            ok = false;
                            break;
                        }
                    }
                    const bool rope = !is_v && e == C::KITEMS - 1;
                    if (lane == 0) mbar_arrive_expect_tx(slot_full + 8 * slot, rope ? C::ATOM_BYTES : C::SLOT_BYTES);
                    __syncwarp();
                    issued = jj + 1;
                    if (jj == 0 && lane == 0) stamp(1);
                    if (lane < segs) {
                        const uint32_t dst = sbase + C::OFF_RING + slot * C::SLOT_BYTES + lane * p.box_rows * 128;
                        if (rope && FP8) {
                            tma_load_2d(dst, &p.tm_rope, 0, row, slot_full + 8 * slot, policy);
                        } else if (rope) {
                            tma_load_2d(dst, &p.tm_k, C::DV, row, slot_full + 8 * slot, policy);
                        } else {
                            // two 128-byte boxes: 64 bf16 columns or 128 codes each
                            const int col = C::ITEM_COLS * e;
                            tma_load_2d(dst, &p.tm_k, col, row, slot_full + 8 * slot, policy);
                            tma_load_2d(dst + C::ATOM_BYTES, &p.tm_k, col + C::ITEM_COLS / 2, row,
                                        slot_full + 8 * slot, policy);
                        }
                    }
                }
            }
        }
    } else if (warp == 1 || warp == 2) {
        // ------------------------------------------------------------ MMA warps
        // Ring-order rule as in the GQA kernel: a slot's full barrier is
        // waited on for item j only once every item before j - NSLOT + 1 of
        // the other kind has been consumed (published next-item indices).
        if (lane == 0) {
            const bool is_s = (warp == 1);
            const uint32_t other_next = is_s ? o_next : s_next;
            auto ring_turn = [&](int j) -> bool {
                return j < C::NSLOT ||
                       counter_wait(other_next, (uint32_t)(j - C::NSLOT), abort_flag, p.status, p.wait_limit_ns);
            };
            bool ok = true;
            if (is_s) {
                const uint32_t id_s = umma_idesc_bf16_f32(128, C::ROWS, false, false);
                const uint32_t id_s8 = umma_idesc_e4m3_f32(128, C::ROWS, false, false);
                const uint64_t q_desc0 = umma_smem_desc(sbase + C::OFF_Q, 16, 1024, kLayoutSwizzle128);
                const uint64_t k_desc0 = umma_smem_desc(sbase + C::OFF_RING, 16, 1024, kLayoutSwizzle128);
                ok = mbar_wait(q_full, 0, abort_flag, p.status, p.wait_limit_ns);
                for (int i = 0; ok && i < tile_count; ++i) {
                    const int j0 = mla_group_item<FP8>(mla_k_group(i), tile_count);
                    const uint32_t d0 = tmem + C::TMEM_S0 + C::S_BUF * (i & 1);
                    for (int e = 0; ok && e < C::KITEMS; ++e) {
                        const int j = j0 + e, slot = j % C::NSLOT;
                        ok = ring_turn(j) &&
                             mbar_wait(slot_full + 8 * slot, (j / C::NSLOT) & 1, abort_flag, p.status,
                                       p.wait_limit_ns) &&
                             (e > 0 || i < 2 ||
                              mbar_wait(s_empty + 8 * (i & 1), ((i >> 1) - 1) & 1, abort_flag, p.status,
                                        p.wait_limit_ns));
                        if (!ok) break;
                        tc_fence_after_sync();
                        const uint64_t a0 = k_desc0 + (uint64_t)((slot * C::SLOT_BYTES) >> 4);
                        if constexpr (!FP8) {
                            const int steps = e == C::KITEMS - 1 ? 4 : 8;
                            for (int ks = 0; ks < steps; ++ks) {
                                const int gk = 8 * e + ks;  // K-step over the 576 depth columns
                                umma_f16_ss(d0 + C::S_ACC * (gk & 1),
                                            a0 + (uint64_t)(((ks >> 2) * C::ATOM_BYTES + (ks & 3) * 32) >> 4),
                                            q_desc0 + (uint64_t)(((gk >> 2) * C::Q_ATOM + (gk & 3) * 32) >> 4),
                                            id_s, gk >= 2);
                            }
                        } else if (e < C::KITEMS - 1) {
                            // codes: eight K-steps of 32 against Q_hi (16 h) and Q_lo (l), accumulator 0
                            for (int ks = 0; ks < 8; ++ks) {
                                const int gk = 8 * e + ks;  // K-step over the 512 codes
                                const uint64_t a = a0 + (uint64_t)(((ks >> 2) * C::ATOM_BYTES + (ks & 3) * 32) >> 4);
                                const uint64_t qh = q_desc0 + (uint64_t)(((gk >> 2) * C::Q_ATOM + (gk & 3) * 32) >> 4);
                                umma_f8_ss(d0, a, qh, id_s8, gk > 0);
                                umma_f8_ss(d0, a, qh + (uint64_t)((4 * C::Q_ATOM) >> 4), id_s8, 1);
                            }
                        } else {
                            // rope: four bf16 K-steps of 16, accumulator 1
                            for (int ks = 0; ks < 4; ++ks)
                                umma_f16_ss(d0 + C::S_ACC, a0 + (uint64_t)((ks * 32) >> 4),
                                            q_desc0 + (uint64_t)((8 * C::Q_ATOM + ks * 32) >> 4), id_s, ks > 0);
                        }
                        umma_commit(slot_empty + 8 * slot);  // the item's slot is free once these complete
                        st_release_u32(s_next, (uint32_t)(e + 1 < C::KITEMS
                                                              ? j + 1
                                                              : (i + 1 < tile_count
                                                                     ? mla_group_item<FP8>(mla_k_group(i + 1), tile_count)
                                                                     : 0xffffffffu)));
                    }
                    if (ok) umma_commit(s_full + 8 * (i & 1));
                }
            } else {
                const uint32_t id_pv = FP8 ? umma_idesc_e4m3_f32(128, C::ROWS, true, false)
                                           : umma_idesc_bf16_f32(128, C::ROWS, true, false);
                // A = V^T, MN-major: two 64-column atoms one atom apart (LBO), 8-key groups 1024 B apart (SBO)
                const uint64_t v_desc0 = umma_smem_desc(sbase + C::OFF_RING, C::ATOM_BYTES, 1024, kLayoutSwizzle128);
                // B = P^T, K-major: 64-key atoms of 64 heads x 128 B
                const uint64_t p_desc0 = umma_smem_desc(sbase + C::OFF_P, 16, 1024, kLayoutSwizzle128);
                mbar_wait(tmem_ready, 0, abort_flag, p.status, p.wait_limit_ns);
                tc_fence_after_sync();
                tmem = *tmem_slot;
                for (int t = 0; ok && t < tile_count; ++t) {
                    const int j0 = mla_group_item<FP8>(mla_v_group(t, tile_count), tile_count);
                    ok = mbar_wait(p_full + 8 * (t & 1), (t >> 1) & 1, abort_flag, p.status, p.wait_limit_ns);
                    for (int e = 0; ok && e < C::VITEMS; ++e) {
                        const int j = j0 + e, slot = j % C::NSLOT;
                        ok = ring_turn(j) &&
                             mbar_wait(slot_full + 8 * slot, (j / C::NSLOT) & 1, abort_flag, p.status,
                                       p.wait_limit_ns) &&
                             (!v_tail || t + 1 < tile_count ||
                              mbar_wait(v_zeroed + 8 * e, 0, abort_flag, p.status, p.wait_limit_ns));
                        if (!ok) break;
                        tc_fence_after_sync();
                        const uint64_t a0 = v_desc0 + (uint64_t)((slot * C::SLOT_BYTES) >> 4);
                        const uint64_t b0 = p_desc0 + (uint64_t)(((t % C::P_BUFS) * C::P_BYTES) >> 4);
                        if constexpr (!FP8) {
                            const uint32_t d = tmem + C::TMEM_O0 + 64 * e;  // dv block e
#pragma unroll
                            for (int ks = 0; ks < C::BN / 16; ++ks)
                                umma_f16_ss(d, a0 + (uint64_t)((ks * 2048) >> 4),
                                            b0 + (uint64_t)(((ks >> 2) * C::P_ATOM + (ks & 3) * 32) >> 4), id_pv,
                                            t > 0 || ks > 0);
                        } else {
                            // dv blocks 2e, 2e + 1 (one box each); four K-steps of 32 keys
                            // (four 8-key groups of V^T) against P'_hi and P'_lo
#pragma unroll
                            for (int bb = 0; bb < 2; ++bb) {
                                const uint32_t d = tmem + C::TMEM_O0 + 64 * (2 * e + bb);
#pragma unroll
                                for (int ks = 0; ks < 4; ++ks) {
                                    const uint64_t a = a0 + (uint64_t)((bb * C::ATOM_BYTES + ks * 4096) >> 4);
                                    const uint64_t ph = b0 + (uint64_t)((ks * 32) >> 4);
                                    umma_f8_ss(d, a, ph, id_pv, t > 0 || ks > 0);
                                    umma_f8_ss(d, a, ph + (uint64_t)(C::P_ATOM >> 4), id_pv, 1);
                                }
                            }
                        }
                        umma_commit(slot_empty + 8 * slot);
                        st_release_u32(o_next,
                                       (uint32_t)(e + 1 < C::VITEMS
                                                      ? j + 1
                                                      : (t + 1 < tile_count
                                                             ? mla_group_item<FP8>(mla_v_group(t + 1, tile_count), tile_count)
                                                             : 0xffffffffu)));
                    }
                    if (ok) umma_commit(o_full + 8 * (t & 1));
                }
            }
            st_release_u32(is_s ? s_next : o_next, 0xffffffffu);
            umma_commit(mma_done);
            volatile int keep_waiting = 0;
            mbar_wait(mma_done, 0, &keep_waiting, p.status, p.wait_limit_ns);
        }
        __syncwarp();
    } else {
        // ------------------------------------------------- softmax warpgroups
        const int wg = (warp - C::WG0) >> 2;          // heads 32 wg .. 32 wg + 31
        const int wt = tid - 32 * C::WG0 - 128 * wg;  // 0..127
        const uint32_t wg_bar = 1 + wg;
        const int quad = warp & 3;
        const int my_lane = 32 * quad + lane;         // key (S^T) or value column within a dv block (O^T)
        const uint32_t lane_addr = (uint32_t)(32 * quad) << 16;
        const float c2 = p.scale_log2e;
        const int h0 = kvh * p.group + row_block * C::ROWS;  // first head of this CTA

        // Q rows -> nine K-major 128-byte-swizzled atoms. Every load is issued
        // before the first store, so the 18 chunks of a thread arrive together.
        if constexpr (FP8) {
            // Four threads per head: codes [128 part, 128 part + 128) of the nope
            // part (one 128-byte row of atom `part`) and rope chunks 2 part, 2 part
            // + 1. The head is scaled by sigma_h, a power of two with max |q_nope|
            // sigma_h <= 28, and split into 16 e4m3(x) (atoms 0-3) and
            // e4m3(16 (x - e4m3(x))) (atoms 4-7); the rope stays bf16 (atom 8).
            const int T = wt + 128 * wg, hh = T >> 2, part = T & 3;
            const uint4* qg = reinterpret_cast<const uint4*>(p.q + ((int64_t)b * p.num_q_heads + h0 + hh) * C::DK);
            uint4 qv[16], qr[2];
#pragma unroll
            for (int k = 0; k < 16; ++k) qv[k] = __ldg(qg + 16 * part + k);
#pragma unroll
            for (int k = 0; k < 2; ++k) qr[k] = __ldg(qg + 64 + 2 * part + k);
            float amax = 0.f;
#pragma unroll
            for (int k = 0; k < 16; ++k) {
                const uint32_t w4[4] = {qv[k].x, qv[k].y, qv[k].z, qv[k].w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float2 f = bf16x2_to_float2(w4[e]);
                    amax = fmaxf(amax, fmaxf(fabsf(f.x), fabsf(f.y)));
                }
            }
            amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
            amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
            const float sig = e4m3_split_scale(amax, 28.f);
            uint8_t* qa = smem + C::OFF_Q + part * C::Q_ATOM + hh * 128;
#pragma unroll
            for (int u = 0; u < 8; ++u) {  // 16 codes of chunks 2u, 2u + 1
                uint32_t hw[4], lw[4];
#pragma unroll
                for (int c = 0; c < 2; ++c) {
                    const uint32_t w4[4] = {qv[2 * u + c].x, qv[2 * u + c].y, qv[2 * u + c].z, qv[2 * u + c].w};
                    uint32_t hp[4], lp[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const float2 f = bf16x2_to_float2(w4[e]);
                        float h0, l0, h1, l1;
                        e4m3_split(f.x * sig, h0, l0);
                        e4m3_split(f.y * sig, h1, l1);
                        hp[e] = e4m3x2(h0, h1);
                        lp[e] = e4m3x2(l0, l1);
                    }
                    hw[2 * c] = hp[0] | (hp[1] << 16);
                    hw[2 * c + 1] = hp[2] | (hp[3] << 16);
                    lw[2 * c] = lp[0] | (lp[1] << 16);
                    lw[2 * c + 1] = lp[2] | (lp[3] << 16);
                }
                const int off = (u ^ (hh & 7)) << 4;
                *reinterpret_cast<uint4*>(qa + off) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
                *reinterpret_cast<uint4*>(qa + 4 * C::Q_ATOM + off) = make_uint4(lw[0], lw[1], lw[2], lw[3]);
            }
#pragma unroll
            for (int k = 0; k < 2; ++k) {
                const int c = 2 * part + k;
                *reinterpret_cast<uint4*>(smem + C::OFF_Q + 8 * C::Q_ATOM + hh * 128 + ((c ^ (hh & 7)) << 4)) = qr[k];
            }
            if (part == 0) reinterpret_cast<float*>(smem + C::OFF_QINV)[hh] = 0.0625f / sig;
        } else {
            constexpr int kChunks = C::ROWS * (C::DK / 8) / 256;  // 16-byte chunks per thread
            static_assert(kChunks * 256 == C::ROWS * (C::DK / 8), "Q chunks split evenly");
            uint4 qv[kChunks];
            const uint4* qg = reinterpret_cast<const uint4*>(p.q + ((int64_t)b * p.num_q_heads + h0) * C::DK);
#pragma unroll
            for (int k = 0; k < kChunks; ++k) qv[k] = __ldg(qg + (wt + 128 * wg + 256 * k));
#pragma unroll
            for (int k = 0; k < kChunks; ++k) {
                const int idx = wt + 128 * wg + 256 * k;
                const int r = idx / 72, u = idx % 72;  // 16-byte chunk u of head r (heads are contiguous)
                *reinterpret_cast<uint4*>(smem + C::OFF_Q + (u >> 3) * C::Q_ATOM + r * 128 +
                                          (((u & 7) ^ (r & 7)) << 4)) = qv[k];
            }
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(q_full);
        if (FP8) named_barrier_sync(3, 256);  // every head's 1 / (16 sigma_h) is written
        mbar_wait(tmem_ready, 0, abort_flag, p.status, p.wait_limit_ns);
        tc_fence_after_sync();
        tmem = *tmem_slot;

#pragma unroll
        for (int r = 0; r < 32; ++r) {
            m_run[r] = -INFINITY;
            l_part[r] = 0.f;
        }
        const uint32_t col_wg = 32 * wg;  // this warpgroup's columns in every S^T / O^T accumulator
        float* red_w = red_s + wg * 4 * 32;
        bool seen_abort = false;
        // FP8: Sigma, the power of two that bounds every K scale this warpgroup
        // has folded into P (0 before the first); O^T holds 16 / Sigma times the
        // scaled partial.
        float sig_run = 0.f;
        float* sig_w = reinterpret_cast<float*>(smem + C::OFF_SIG) + 4 * wg;
        for (int i = 0; i < tile_count; ++i) {
            mbar_wait(s_full + 8 * (i & 1), (i >> 1) & 1, abort_flag, p.status, p.wait_limit_ns);
            if (i == 0 && wt == 0 && wg == 0) {
                stamp(2);
                stamp(5);  // unit 0: first S observed
            }
            tc_fence_after_sync();
            float s[32];
            float ksc = 1.f;  // FP8: this key's K scale (0 past the sequence)
            if constexpr (!FP8) {
                tmem_ld2_sum_x32(tmem + lane_addr + C::TMEM_S0 + C::S_BUF * (i & 1) + col_wg, C::S_ACC, s);
                tc_fence_before_sync();
                __syncwarp();
                if (lane == 0) mbar_arrive(s_empty + 8 * (i & 1));
            } else {
                float sr[32];
                tmem_ld2_x32(tmem + lane_addr + C::TMEM_S0 + C::S_BUF * (i & 1) + col_wg, C::S_ACC, s, sr);
                tc_fence_before_sync();
                __syncwarp();
                if (lane == 0) mbar_arrive(s_empty + 8 * (i & 1));
                if (scaled) {
                    const int kse = i % C::KS;
                    mbar_wait(ks_full + 8 * kse, (i / C::KS) & 1, abort_flag, p.status, p.wait_limit_ns);
                    ksc = reinterpret_cast<const float*>(smem + C::OFF_KS)[kse * C::BN + my_lane];
                    __syncwarp();
                    if (lane == 0) mbar_arrive(ks_empty + 8 * kse);
                }
                // raw score: codes / (16 sigma_h) times the key's K scale, plus the rope part
                const float4* qinv = reinterpret_cast<const float4*>(smem + C::OFF_QINV) + (col_wg >> 2);
#pragma unroll
                for (int r4 = 0; r4 < 8; ++r4) {
                    const float4 qm = qinv[r4];
                    s[4 * r4 + 0] = fmaf(s[4 * r4 + 0], qm.x * ksc, sr[4 * r4 + 0]);
                    s[4 * r4 + 1] = fmaf(s[4 * r4 + 1], qm.y * ksc, sr[4 * r4 + 1]);
                    s[4 * r4 + 2] = fmaf(s[4 * r4 + 2], qm.z * ksc, sr[4 * r4 + 2]);
                    s[4 * r4 + 3] = fmaf(s[4 * r4 + 3], qm.w * ksc, sr[4 * r4 + 3]);
                }
            }

            const int key = (tile_begin + i) * C::BN + my_lane;
            if (key >= L) {
#pragma unroll
                for (int r = 0; r < 32; ++r) s[r] = -INFINITY;
                ksc = 0.f;
            }
            // Without short-circuit branches (one per head otherwise): a finite
            // score over an empty row, or one more than the threshold above the
            // row's max (a masked score compares false).
            bool need = false;
#pragma unroll
            for (int r = 0; r < 32; ++r) {
                const bool first = (m_run[r] == -INFINITY) & (s[r] != -INFINITY);
                const bool over = (s[r] - m_run[r]) * c2 > C::RESCALE;
                need = need | first | over;
            }
            if constexpr (FP8) {
                // a K scale above the bound, or a warp whose keys' scales all lie
                // more than 16x below it (the bound then follows them down, so
                // that P' keeps its precision)
                const bool low = __all_sync(0xffffffffu, ksc < sig_run * 0.0625f) && __any_sync(0xffffffffu, ksc > 0.f);
                need = need | (ksc > sig_run) | low;
            }
            seen_abort |= (*abort_flag != 0);
            if (named_barrier_or(wg_bar, 128, need || seen_abort)) {
                {
                    int row;
                    float v[32];
#pragma unroll
                    for (int r = 0; r < 32; ++r) v[r] = s[r];
                    // reduce-scatter: lane holds the max of head `row` over this warp's keys
                    row = 0;
#pragma unroll
                    for (int w = 16, n = 32; w >= 1; w >>= 1, n >>= 1) {
                        const bool up = (lane & w) != 0;
#pragma unroll
                        for (int k = 0; k < n / 2; ++k) {
                            const float send = up ? v[k] : v[k + n / 2];
                            const float keep = up ? v[k + n / 2] : v[k];
                            v[k] = fmaxf(keep, __shfl_xor_sync(0xffffffffu, send, w));
                        }
                        row += up ? n / 2 : 0;
                    }
                    red_w[quad * 32 + row] = v[0];
                }
                if constexpr (FP8) {
                    float km = ksc;
#pragma unroll
                    for (int o = 16; o >= 1; o >>= 1) km = fmaxf(km, __shfl_xor_sync(0xffffffffu, km, o));
                    if (lane == 0) sig_w[quad] = km;
                }
                seen_abort |= (*abort_flag != 0);
                if (named_barrier_or(wg_bar, 128, seen_abort)) break;
                bool moved = false;
                // FP8: a K scale above Sigma, or a tile whose largest scale km lies
                // more than 16x below it, sets Sigma to the power of two above km,
                // and O^T, which holds 16 / Sigma times its partial, is corrected by
                // Sigma_old / Sigma_new (nothing to correct before the first).
                float sig_ratio = 1.f;
                if constexpr (FP8) {
                    const float km = fmaxf(fmaxf(sig_w[0], sig_w[1]), fmaxf(sig_w[2], sig_w[3]));
                    if (km > sig_run || (km > 0.f && km < sig_run * 0.0625f)) {
                        int ex = 0;
                        frexpf(km, &ex);
                        const float sig_new = ldexpf(1.f, ex);
                        if (sig_run > 0.f) {
                            sig_ratio = sig_run / sig_new;
                            moved = true;
                        }
                        sig_run = sig_new;
                    }
                }
                float alpha[32];
#pragma unroll
                for (int r = 0; r < 32; ++r) {
                    const float tmax = fmaxf(fmaxf(red_w[r], red_w[32 + r]), fmaxf(red_w[64 + r], red_w[96 + r]));
                    const bool move = (m_run[r] == -INFINITY) ? (tmax != -INFINITY)
                                                              : ((tmax - m_run[r]) * c2 > C::RESCALE);
                    alpha[r] = sig_ratio;  // O^T's correction: the max's and (FP8) Sigma's
                    if (move) {
                        const float a_m = (m_run[r] == -INFINITY) ? 0.f : ex2_approx((m_run[r] - tmax) * c2);
                        m_run[r] = tmax;
                        l_part[r] *= a_m;
                        alpha[r] = a_m * sig_ratio;
                        moved = true;  // uniform: every thread sees the same maxima
                    }
                }
                if (moved && i > 0) {
                    // Correct O^T in place: its last product (tile i - 1) must
                    // have completed, and no later one is issued before this
                    // tile's P is published.
                    mbar_wait(o_full + 8 * ((i - 1) & 1), ((i - 1) >> 1) & 1, abort_flag, p.status,
                              p.wait_limit_ns);
                    tc_fence_after_sync();
#pragma unroll 1
                    for (int blk = 0; blk < 4; ++blk) {
                        float o[32];
                        const uint32_t ta = tmem + lane_addr + C::TMEM_O0 + 64 * blk + col_wg;
                        tmem_ld_32x32b_x32(ta, o);
#pragma unroll
                        for (int r = 0; r < 32; ++r) o[r] *= alpha[r];
                        tmem_st_32x32b_x32(ta, o);
                    }
                    tc_fence_before_sync();
                }
                named_barrier_sync(wg_bar, 128);  // red_w is read before the next tile's writes
            }
            // exp2(-inf) = +0 for masked scores (the select keeps an empty row's
            // -inf - -inf from giving NaN).
#pragma unroll
            for (int r = 0; r < 32; ++r) {
                const float x = (s[r] == -INFINITY) ? -INFINITY : (s[r] - m_run[r]) * c2;
                const float pr = ex2_approx(x);
                l_part[r] += pr;
                s[r] = pr;
            }
            // P buffer i % P_BUFS was last read by the O product of tile i - P_BUFS.
            if (i >= C::P_BUFS) {
                const int tp = i - C::P_BUFS;
                mbar_wait(o_full + 8 * (tp & 1), (tp >> 1) & 1, abort_flag, p.status, p.wait_limit_ns);
            }
            if constexpr (!FP8) {
                uint8_t* pb = smem + C::OFF_P + (i % C::P_BUFS) * C::P_BYTES + (my_lane >> 6) * C::P_ATOM;
                const int kk = my_lane & 63;
#pragma unroll
                for (int r = 0; r < 32; ++r) {
                    const int hr = col_wg + r;  // head row of P^T
                    *reinterpret_cast<__nv_bfloat16*>(pb + hr * 128 + (((kk >> 3) ^ (hr & 7)) << 4) + (kk & 7) * 2) =
                        __float2bfloat16_rn(s[r]);
                }
            } else {
                // 16 P' = 16 P k_scale / Sigma <= 256 as two E4M3 codes (h + l): P'_hi
                // in one atom [64 heads][128 keys], P'_lo in the next.
                uint8_t* pb = smem + C::OFF_P + (i % C::P_BUFS) * C::P_BYTES;
                const float f = sig_run > 0.f ? 16.f * ksc / sig_run : 0.f;
                const int kb = my_lane >> 4, kw = my_lane & 15;
#pragma unroll
                for (int r = 0; r < 32; r += 2) {
                    uint32_t hi, lo;
                    e4m3_split2(s[r] * f, s[r + 1] * f, hi, lo);
                    const int h0r = col_wg + r, h1r = h0r + 1;
                    const int o0 = h0r * 128 + ((kb ^ (h0r & 7)) << 4) + kw;
                    const int o1 = h1r * 128 + ((kb ^ (h1r & 7)) << 4) + kw;
                    pb[o0] = (uint8_t)(hi & 0xffu);
                    pb[o1] = (uint8_t)((hi >> 8) & 0xffu);
                    pb[C::P_ATOM + o0] = (uint8_t)(lo & 0xffu);
                    pb[C::P_ATOM + o1] = (uint8_t)((lo >> 8) & 0xffu);
                }
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(p_full + 8 * (i & 1));
        }
        // The sequence's last tile: zero the V rows past L in each of its V
        // items as it lands (P is already published: the O warp waits for
        // each item's v_zeroed barrier), so unused cache rows, whatever they
        // hold, meet P = 0 as exact zeros. Each warpgroup zeroes one of the
        // item's two 64-column atoms. Ring order: the item that held the slot
        // before has been consumed (both MMA warps' published progress).
        if (v_tail && !seen_abort) {
            const int t = tile_count - 1;
            const int j0 = mla_group_item<FP8>(mla_v_group(t, tile_count), tile_count);
            const bool past = (tile_begin + t) * C::BN + my_lane >= L;
            for (int e = 0; e < C::VITEMS; ++e) {
                const int j = j0 + e, slot = j % C::NSLOT;
                if (j >= C::NSLOT) {
                    counter_wait(s_next, (uint32_t)(j - C::NSLOT), abort_flag, p.status, p.wait_limit_ns);
                    counter_wait(o_next, (uint32_t)(j - C::NSLOT), abort_flag, p.status, p.wait_limit_ns);
                }
                mbar_wait(slot_full + 8 * slot, (j / C::NSLOT) & 1, abort_flag, p.status, p.wait_limit_ns);
                if (past) {
                    uint4* row = reinterpret_cast<uint4*>(smem + C::OFF_RING + slot * C::SLOT_BYTES +
                                                          wg * C::ATOM_BYTES + my_lane * 128);
#pragma unroll
                    for (int u = 0; u < 8; ++u) row[u] = make_uint4(0, 0, 0, 0);
                }
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(v_zeroed + 8 * e);
            }
        }
        if (wt == 0 && wg == 0) {
            stamp(4);  // unit 0: the tile loop is done
            if (trace) trace[10] = (unsigned long long)tile_count;
        }
        // All products complete.
        if (tile_count > 0)
            mbar_wait(o_full + 8 * ((tile_count - 1) & 1), ((tile_count - 1) >> 1) & 1, abort_flag, p.status,
                      p.wait_limit_ns);
        tc_fence_after_sync();
        if (wt == 0 && wg == 0) stamp(6);  // unit 0: last O product complete
        // Row sums of this warpgroup's 32 heads: reduce-scatter over the warp, then four warps.
        {
            float v[32];
#pragma unroll
            for (int r = 0; r < 32; ++r) v[r] = l_part[r];
            int row = 0;
#pragma unroll
            for (int w = 16, n = 32; w >= 1; w >>= 1, n >>= 1) {
                const bool up = (lane & w) != 0;
#pragma unroll
                for (int k = 0; k < n / 2; ++k) {
                    const float send = up ? v[k] : v[k + n / 2];
                    const float keep = up ? v[k + n / 2] : v[k];
                    v[k] = keep + __shfl_xor_sync(0xffffffffu, send, w);
                }
                row += up ? n / 2 : 0;
            }
            named_barrier_sync(wg_bar, 128);
            red_w[quad * 32 + row] = v[0];
            named_barrier_sync(wg_bar, 128);
        }
        // Row col_wg + wt's (max, sum) in mm, ll for threads wt < 32.
        float mm = -INFINITY, ll = 0.f;
        if (wt < 32) {
#pragma unroll
            for (int r = 0; r < 32; ++r)
                if (r == wt) mm = m_run[r];
            ll = red_w[wt] + red_w[32 + wt] + red_w[64 + wt] + red_w[96 + wt];
        }
        // Split-K epilogue (push). Rank q merges band q of the value columns,
        // [q BW, (q + 1) BW). Every rank pushes, straight from TMEM, its
        // unnormalised partial O for the columns of each other band, and each
        // row's (max, sum), into that band owner's shared memory with
        // st.async; the owner combines its own band from TMEM with what it
        // received. The receive area is this CTA's drained ring, so a rank
        // pushes to q only once q has announced (ready[q]) that all of its
        // own products are complete. Received partial of source s (the
        // source ranks other than q in order), column c, rows 4k .. 4k + 3 at
        // float ((s BW + c) 64 + 4 (k ^ (c & 7))): the XOR spreads a warp's 32
        // consecutive columns over every bank.
        const int BW = p.band_cols, OC = p.out_chunk_cols;
        const uint32_t recv_o = sbase + C::OFF_RECV, recv_ms = sbase + C::OFF_RECV_MS;
        const float o_unit = sig_run * 0.0625f;  // FP8: O^T holds 16 / Sigma times the partial
        if (P > 1) {
            cluster_wait();  // every rank's barriers are initialised
            if (wt == 0 && wg == 0 && !*abort_flag) {
                // This warpgroup has waited for the last O product, which
                // follows every product, every read of the ring, Q and P, and
                // the zeroing of the last tile's V rows.
                mbar_arrive_expect_tx(recv_ms_bar, (uint32_t)((P - 1) * C::ROWS * 8));
                mbar_arrive_expect_tx(recv_o_bar, (uint32_t)((P - 1) * C::ROWS * BW * 4));
                for (int q = 0; q < P; ++q)
                    if (q != rank) mbar_arrive_cluster(map_shared_rank(ready_bar + 8 * rank, q));
            }
            if (wt < 32) {
                for (int q = 0; q < P; ++q) {
                    if (q == rank) continue;
                    if (!mbar_wait<true>(ready_bar + 8 * q, 0, abort_flag, p.status, p.wait_limit_ns)) break;
                    const int src = rank < q ? rank : rank - 1;
                    st_async_f2(map_shared_rank(recv_ms + 8u * (uint32_t)(src * C::ROWS + col_wg + wt), q), mm, ll,
                                map_shared_rank(recv_ms_bar, q));
                }
            }
#pragma unroll 1
            for (int blk = 0; blk < 4; ++blk) {
                const int dv = 128 * blk + my_lane;
                const int q = dv / BW;
                if (q == rank) continue;
                if (!mbar_wait<true>(ready_bar + 8 * q, 0, abort_flag, p.status, p.wait_limit_ns)) break;
                float o[32];
                tmem_ld_32x32b_x32(tmem + lane_addr + C::TMEM_O0 + 64 * blk + col_wg, o);
                if (tile_count == 0) {  // no product was issued: the accumulator holds nothing of ours
#pragma unroll
                    for (int r = 0; r < 32; ++r) o[r] = 0.f;
                }
                if constexpr (FP8) {
#pragma unroll
                    for (int r = 0; r < 32; ++r) o[r] *= o_unit;
                }
                const int c = dv - q * BW, src = rank < q ? rank : rank - 1;
                const uint32_t dst = map_shared_rank(recv_o + 4u * (uint32_t)((src * BW + c) * C::ROWS), q);
                const uint32_t bar_q = map_shared_rank(recv_o_bar, q);
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const int k = (int)(col_wg >> 2) + i;
                    st_async_f4(dst + 16u * (uint32_t)(k ^ (c & 7)), o[4 * i], o[4 * i + 1], o[4 * i + 2],
                                o[4 * i + 3], bar_q);
                }
            }
        }
        if (wt == 0 && wg == 0) stamp(8);  // unit 0: partials pushed
        // Combine weights of row rr = col_wg + wt (threads wt < 32): Gmax over
        // the partials that saw keys, Gsum = sum_q sum_q 2^((max_q - Gmax) c),
        // and w_q = 2^((max_q - Gmax) c) / Gsum on each unnormalised partial
        // O_q (0 for a partial that saw no key), so O = sum_q w_q O_q.
        float* wtab = reinterpret_cast<float*>(smem + C::OFF_WTAB);  // [P][64]
        if (wt < 32) {
            const float2* ms_in = reinterpret_cast<const float2*>(smem + C::OFF_RECV_MS);
            const int rr = col_wg + wt;
            if (P > 1) mbar_wait<true>(recv_ms_bar, 0, abort_flag, p.status, p.wait_limit_ns);
            float gmax = ll > 0.f ? mm : -INFINITY;
            for (int s = 0; s < P - 1; ++s) {
                const float2 v = ms_in[s * C::ROWS + rr];
                if (v.y > 0.f) gmax = fmaxf(gmax, v.x);
            }
            const float e_own = ll > 0.f ? ex2_approx((mm - gmax) * c2) : 0.f;
            float gsum = ll * e_own;
            for (int s = 0; s < P - 1; ++s) {
                const float2 v = ms_in[s * C::ROWS + rr];
                gsum += v.y > 0.f ? v.y * ex2_approx((v.x - gmax) * c2) : 0.f;
            }
            const float ginv = gsum > 0.f ? 1.f / gsum : 0.f;
            wtab[rank * C::ROWS + rr] = e_own * ginv;
            for (int s = 0; s < P - 1; ++s) {
                const float2 v = ms_in[s * C::ROWS + rr];
                wtab[(s < rank ? s : s + 1) * C::ROWS + rr] = v.y > 0.f ? ex2_approx((v.x - gmax) * c2) * ginv : 0.f;
            }
            if (rank == 0 && rr < p.rows && p.lse != nullptr) {
                const int t = rr / p.heads_per_cta;
                const int h = kvh * p.group + row_block * p.heads_per_cta + rr % p.heads_per_cta;
                // natural-log LSE of the scaled scores: scale * Gmax + ln(Gsum)
                p.lse[((int64_t)b * p.num_q + t) * p.num_q_heads + h] =
                    gsum > 0.f ? p.scale * gmax + lg2_approx(gsum) * 0.6931471805599453f : -INFINITY;
            }
        }
        named_barrier_sync(wg_bar, 128);  // this warpgroup's rows' weights
        if (P > 1) mbar_wait<true>(recv_o_bar, 0, abort_flag, p.status, p.wait_limit_ns);
        uint16_t* out_s = reinterpret_cast<uint16_t*>(smem + C::OFF_OUT);  // [BW / OC][64][OC]
        const float* recv_f = reinterpret_cast<const float*>(smem + C::OFF_RECV);
#pragma unroll 1
        for (int blk = 0; blk < 4; ++blk) {
            const int dv = 128 * blk + my_lane;
            if (dv / BW != rank) continue;
            const int c = dv - rank * BW;
            float o[32];
            tmem_ld_32x32b_x32(tmem + lane_addr + C::TMEM_O0 + 64 * blk + col_wg, o);
            if (tile_count == 0) {
#pragma unroll
                for (int r = 0; r < 32; ++r) o[r] = 0.f;
            }
            if constexpr (FP8) {
#pragma unroll
                for (int r = 0; r < 32; ++r) o[r] *= o_unit;
            }
            const float* w_own = wtab + rank * C::ROWS + col_wg;
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const float4 w = *reinterpret_cast<const float4*>(w_own + 4 * i);
                o[4 * i] *= w.x;
                o[4 * i + 1] *= w.y;
                o[4 * i + 2] *= w.z;
                o[4 * i + 3] *= w.w;
            }
            for (int s = 0; s < P - 1; ++s) {
                const float* src = recv_f + (s * BW + c) * C::ROWS;
                const float* w_s = wtab + (s < rank ? s : s + 1) * C::ROWS + col_wg;
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const int k = (int)(col_wg >> 2) + i;
                    const float4 v = *reinterpret_cast<const float4*>(src + 4 * (k ^ (c & 7)));
                    const float4 w = *reinterpret_cast<const float4*>(w_s + 4 * i);
                    o[4 * i] = fmaf(w.x, v.x, o[4 * i]);
                    o[4 * i + 1] = fmaf(w.y, v.y, o[4 * i + 1]);
                    o[4 * i + 2] = fmaf(w.z, v.z, o[4 * i + 2]);
                    o[4 * i + 3] = fmaf(w.w, v.w, o[4 * i + 3]);
                }
            }
            uint16_t* dst = out_s + ((c / OC) * C::ROWS + col_wg) * OC + c % OC;
#pragma unroll
            for (int r = 0; r < 32; ++r) dst[r * OC] = __bfloat16_as_ushort(__float2bfloat16_rn(o[r]));
        }
        tc_fence_before_sync();
        fence_proxy_async_smem();
        named_barrier_sync(3, 256);
        if (wt == 0 && wg == 0) {
            for (int c0 = 0; c0 < BW; c0 += OC)
                tma_store_3d(&p.tm_out, smem_addr(out_s + (c0 / OC) * C::ROWS * OC), rank * BW + c0,
                             kvh * p.group + row_block * p.heads_per_cta, b * p.num_q);
            tma_store_commit();
            tma_store_wait_read();
            stamp(9);  // unit 0: band stored
        }
    }

    __syncthreads();
    if (warp == 1) {
        tc_fence_after_sync();
        tmem_dealloc(tmem, C::TMEM_COLS);
    }
    if (warp == 0 && lane == 0 && *abort_flag) {
        volatile int keep_waiting = 0;
        for (int j = issued > C::NSLOT ? issued - C::NSLOT : 0; j < issued; ++j)
            mbar_wait(slot_full + 8 * (j % C::NSLOT), (j / C::NSLOT) & 1, &keep_waiting, p.status, p.wait_limit_ns);
        for (int t = ks_issued > C::KS ? ks_issued - C::KS : 0; t < ks_issued; ++t)
            mbar_wait(ks_full + 8 * (t % C::KS), (t / C::KS) & 1, &keep_waiting, p.status, p.wait_limit_ns);
    }
    if (P > 1 && warp < C::WG0) cluster_wait();  // pairs with the early arrive
    __syncwarp();
    if (P > 1) cluster_sync_all();  // after a timed-out wait a peer may still push into this CTA until here
    if (tid == 0) stamp(3);
}

template <bool FP8>
static void mla_fill_geometry(KernelGeometry* g, const char* name)
{
    using C = MlaCfgT<FP8>;
    g->func = reinterpret_cast<const void*>(&mla_tc_decode_kernel<FP8>);
    g->threads = C::THREADS;
    g->keys_per_tile = C::BN;
    g->stages = C::NSLOT;
    g->rows_capacity = C::ROWS;
    g->smem_bytes = C::SMEM_BYTES;
    g->name = name;
}

bool mla_tc_geometry(int qk, int ov, int nope, int heads_per_kv, int num_q, KernelGeometry* g)
{
    using C = MlaCfgT<false>;
    if (qk != C::DK || ov != C::DV || nope != C::DV || num_q != 1 || heads_per_kv % C::ROWS) return false;
    mla_fill_geometry<false>(g, "mla_tc_d576_v512_bn128_n64_slots4");
    return true;
}

bool mla_tc_fp8_geometry(int qk, int ov, int nope, int rope, int heads_per_kv, int num_q, KernelGeometry* g)
{
    using C = MlaCfgT<true>;
    if (qk != C::DK || ov != C::DV || nope != C::DV || rope != C::DK - C::DV || num_q != 1 ||
        heads_per_kv % C::ROWS)
        return false;
    mla_fill_geometry<true>(g, "mla_tc_e4m3_d576_r64_v512_bn128_n64_slots4");
    return true;
}

}  // namespace fad
