// kernel_tc.cuh -- the tcgen05 (5th-generation tensor core) decode kernel for
// GQA rows of head dimension 128 (sm_103a), for a bf16 cache and for an fp8
// (OCP E4M3) cache with an optional per-token K scale. kernel_tc.cu and
// kernel_tc_fp8.cu instantiate it.
//
// The T*g <= 16 query rows of one kv head are too few to fill an MMA M
// dimension, so both products are issued transposed, with the keys (resp.
// the value columns) on M = 128 and the query rows on N = 16:
//   S^T [128 keys x 16 rows]  = K_tile [128 x 128] . Q^T          (A, B K-major)
//   O^T [128 dv x 16 rows]    = V_tile^T [128 dv x 128 keys] . P^T (A MN-major)
// with fp32 accumulators in tensor memory. This keeps the tile dense on the
// tensor pipe while HBM stays the bound.
//
// fp8 cache (FA4Config page: qkv_dtype E4M3, scale_dtype_ for the per-token K
// scale): the E4M3 tiles feed kind::f8f6f4 MMAs straight from the TMA ring
// (K = 32 per MMA). Q and P are bf16 / fp32 quantities, so each is carried
// as two E4M3 operands whose sum is 16 x to about 2^-8 (fp8.cuh: Q as
// 16 e4m3(x) + e4m3(16 (x - e4m3(x))) after a power-of-two scale per row;
// P <= 16 as e4m3(16 P) + e4m3(16 P - e4m3(16 P))), both accumulated into the
// same fp32 accumulator; this keeps about 8 bits of x, as bf16 does.
// S = acc / (16 sigma_r) times the key's scale, O = acc / 16.
// The per-token K scales reach the softmax threads through a small ring of
// bulk copies (one per page segment) with its own full / empty barriers.
//
// Warp roles (one CTA = one cluster rank; a cluster works on one
// (sequence, kv head) unit at a time, the deep-ring variant on several in turn):
//   warp 0     load: page-table walk (warp-wide blocks of entries fetched a
//              block ahead),
//              TMA loads of 128-key K and V tiles (two 64-column
//              128-byte-swizzled boxes per page segment, one lane per
//              segment) into a ring of NSLOT 32 KB slots, in the order the
//              MMA warps consume them (V lagging K by VLAG tiles, see k_item)
//   warp 1     MMA S: allocates 256 TMEM columns (two S buffers of four
//              accumulators, then one O fragment per softmax warpgroup) and
//              issues every S_i = K_i Q^T;
//   warp 2     MMA O: issues every O_t += V_t^T P_t^T into the fragment of the
//              tile's warpgroup; each MMA warp commits a tile's products to the
//              softmax warps and to the ring slot it read;
//   warps 3-6  softmax (and 7-10 for a second warpgroup on alternate tiles;
//              thread = TMEM lane = key for S, = value column for O): online
//              softmax in exp2 form with the running max in raw score units,
//              P^T to shared memory, and the correction O <- O * alpha applied
//              to the TMEM fragment in place when a row's max moves; then the
//              split-K epilogue (splitk_combine.cuh): in the shallow-ring
//              variant they merge themselves, in the deep-ring variant each
//              warpgroup pushes its partial to the band owners and goes on;
//   last warp  (deep ring) epilogue: merges the pushed partials, stores the band.
//
// Geometry and vocabulary follow the FA4Config page (Modular MAX docs):
// TMEM_S / TMEM_O / TMEM_P column maps, num_kv_stages, GQA fusion (field
// group), split-K clusters (splitk_partitions, with_splitk); the TMEM
// visibility rule of the fa4_lse_combine_write page (wait for the MMA's
// barrier, then tcgen05.fence::after_thread_sync, before reading TMEM) is
// applied to every TMEM read.
#pragma once

#include <type_traits>

#include "fa_decode_internal.h"
#include "fp8.cuh"
#include "splitk_combine.cuh"
#include "tcgen05.cuh"

namespace fad {

// NS32: the ring's size in 32 KB units (kTcSlotsShared or kTcSlotsAlone); a
// ring slot holds one K or V tile: 32 KB of bf16, 16 KB of E4M3.
template <int NS32, int NRV, bool FP8>
struct TcCfg {
    // The deep-ring variant (one CTA per SM) works through several
    // (sequence, kv head) units per cluster; it keeps dedicated Q, stage and
    // output buffers so that a unit's epilogue overlaps the next unit's
    // loads. The shallow-ring variant (two CTAs per SM) takes one unit per
    // cluster and stages its epilogue in the drained ring.
    static constexpr bool MULTI = NS32 > kTcSlotsShared;
    // Ring slots: the bf16 tile is 32 KB, the E4M3 tile 16 KB; the fp8 deep
    // ring gives one slot to the scale ring and its barriers (11 x 16 KB).
    static constexpr int NSLOT = FP8 ? 2 * NS32 - (MULTI ? 1 : 0) : NS32;
    // V tiles are issued VLAG tiles after their K (<= 3: rows_s ring). A lag
    // of 2 was measured slower than 1 on the deep ring: K tiles then wait in
    // the ring for an S buffer instead. A lag of 0 (V right behind its K) was
    // slower still (long_context 103 -> 111 us): the next tile's K then
    // queues behind a V that waits for its P anyway.
    static constexpr int VLAG = 1;
    static constexpr int D = 128;       // qk_depth == ov_depth
    static constexpr int BN = 128;      // keys per tile (M of S^T)
    static constexpr int NR = 16;       // padded query rows (N of both MMAs)
    static_assert(NRV == 4 || NRV == 8 || NRV == 16, "real rows per CTA");
    // Softmax warpgroups: two (taking alternate tiles) where the registers of
    // one CTA per SM allow it, else one.
    static constexpr int NWG = (MULTI && NRV <= 8) ? 2 : 1;
    static constexpr int WG0 = 3;       // first softmax warp (warps 3-6, 7-10 each cover TMEM quadrants 3, 0, 1, 2)
    static constexpr int EPI = WG0 + 4 * NWG;  // the multi-unit variant's epilogue warp
    static constexpr int THREADS = MULTI ? 32 * (EPI + 1) : 224;
    static constexpr int ELEM = FP8 ? 1 : 2;             // bytes per cache element
    static constexpr int BOXES = FP8 ? 1 : 2;            // 128-byte-wide TMA boxes per page segment
    static constexpr int TILE_BYTES = BN * D * ELEM;     // one K or V tile: 32 KB bf16, 16 KB fp8
    static constexpr int BOX_BYTES = BN * 128;           // one 128-byte-wide box of a tile
    // Q and P operands, 4 KB each: bf16 [2 atoms][16 rows][128 B]; fp8 the
    // high and low E4M3 parts, [2][16 rows][128 B].
    static constexpr int Q_BYTES = NR * D * 2;
    static constexpr int P_BYTES = NR * BN * 2;
    // Lazy-rescale threshold in exp2 units: P <= 2^threshold. The fp8 split
    // of P needs 16 e4m3(P) <= 448.
    static constexpr float RESCALE = FP8 ? 4.0f : 8.0f;
    // fp8 per-token K scales: a ring of KS entries of BN floats, by K tile.
    static constexpr int KS = FP8 ? (MULTI ? 8 : 4) : 0;
    // bf16: each product's 8 K-steps are spread over NACC = 4 independent
    // accumulators of N = 16 columns (K-step ks accumulates into ks % NACC),
    // so dependent MMAs form chains of depth 2. fp8: the high and low E4M3
    // parts of Q (of P) are the rows 0-15 and 16-31 of one N = 32 operand, so
    // a product is 4 K-steps of 32 over NACC = 2 accumulators of 32 columns,
    // half the MMA instructions (their issue bounds the tile rate). Either
    // way a buffer is 64 columns holding four 16-column partials, and readers
    // sum the four at a 16-column stride.
    static constexpr int NACC = FP8 ? 2 : 4;
    static constexpr int MMA_N = FP8 ? 32 : 16;
    static constexpr int ACC_COLS = MMA_N;                        // columns of one accumulator
    static constexpr int PART_COLS = 16;                          // reader stride between partials
    static constexpr int BUF_COLS = NACC * ACC_COLS;              // 64
    // P buffers (by global tile index): buffer gi % NPB, reused NPB tiles
    // later once the O product that read it has completed. Four with two
    // warpgroups on the fp8 kernel (whose smaller ring leaves room), else two.
    static constexpr int NPB = (NWG == 2 && FP8) ? 4 : 2;
    // O stays in tensor memory, one fragment per softmax warpgroup (the
    // TMEM_O fragments of the fa4_lse_combine_write page): the O MMA
    // accumulates a warpgroup's tiles straight into its fragment, a moved max
    // rescales the fragment in place, and the unit epilogue reads it once
    // (two warpgroups: each pushes its own fragment as a partial of the unit).
    // With one warpgroup the O barriers go by P buffer, so that writing P
    // waits only for the product two tiles back, and a rescale for the
    // previous one; with two they go by fragment.
    static constexpr bool O_BAR_BY_FRAG = NWG == 2;
    static constexpr int N_OBAR = O_BAR_BY_FRAG ? 2 : NPB;
    // Two warpgroups with four P buffers also count O products by P buffer
    // (o_buf), so that writing P(t) waits for O(t - 4), the buffer's previous
    // reader, and only a rescale waits for the fragment's previous product.
    static constexpr bool O_BUF_BAR = O_BAR_BY_FRAG && NPB > 2;
    static constexpr int TMEM_S0 = 0, TMEM_O0 = 2 * BUF_COLS;     // S [2], then O [NWG]
    static constexpr int TMEM_COLS = 256;
    // Units with at least this many tiles per rank are issued two items per
    // pass by the load warp (its per-item cost bounds them), shorter ones one
    // at a time; measured: pairs for every unit on the fp8 kernel and the
    // shallow ring, from 16 tiles on the bf16 deep ring.
    static constexpr int PAIR_TILES = (FP8 || !MULTI) ? 0 : 16;

    static constexpr int Q_BUFS = MULTI ? 2 : 1;                  // by unit parity
    static constexpr int OFF_RING = 0;                            // NSLOT x 32 KB
    static constexpr int OFF_Q = NSLOT * TILE_BYTES;              // K-major SW128 [Q_BUFS][2 boxes][16][128 B]
    static constexpr int OFF_P = OFF_Q + Q_BUFS * Q_BYTES;        // [2 buffers][2 atoms][16][128 B]
    static constexpr int OFF_RED = OFF_P + NPB * P_BYTES;         // float [2][4][NRV]
    static constexpr int OFF_MAXSUM = OFF_RED + 2 * 4 * NR * 4;   // float2 [NRV]
    static constexpr int OFF_BAR = OFF_MAXSUM + NR * 8;
    // barriers: slot_full[NSLOT], slot_empty[NSLOT], s_full[2], s_empty[2],
    // p_full[2], o_full[2], o_empty[2], q_full[2], q_empty[2], publish,
    // mma_done, tmem_ready, recv_full[2], recv_free[2], (spare)
    // then (fp8) ks_full[KS], ks_empty[KS], then p_full[NPB], o_full[NPB],
    // o_empty[NPB], (O_BUF_BAR) o_buf[NPB] (the pairs above at p_full /
    // o_full / o_empty are unused)
    static constexpr int NBAR = 2 * NSLOT + 22 + 2 * KS + 3 * NPB + (O_BUF_BAR ? NPB : 0);
    static constexpr int OFF_ROWS = OFF_BAR + NBAR * 8;          // int [4 tiles][16 segments]
    static constexpr int OFF_MISC = OFF_ROWS + 4 * 16 * 4;       // tmem base, abort, S next item, O next item
    static constexpr int OFF_KS = (OFF_MISC + 16 + 127) / 128 * 128;      // float [KS][BN]
    static constexpr int OFF_QINV = OFF_KS + KS * BN * 4;                 // fp8: float [2][NR], 1 / (16 sigma_r)
    static constexpr int MISC_END = OFF_QINV + (FP8 ? 2 * NR * 4 : 0);
    // Epilogue buffers. Single-unit variant: f32 stage [P][NRV][Dv / P] in the
    // drained ring (slot 0) that peers pull from, bf16 output band in slot 1.
    // Multi-unit variant: receive buffers that peers push into (one or two,
    // by unit, as space allows), each with one partial per (rank, softmax
    // warpgroup): float [NWG P][Dv / P][NRV] + float2 [NWG P][NRV]; the
    // combine weights float [NWG P][NRV] and the output band.
    static constexpr int OUT_BYTES = NRV * D * 2;
    static constexpr int RECV_BUFS = NWG * NRV <= 8 ? 2 : 1;
    static constexpr int RECV_O_BYTES = NWG * NRV * D * 4;       // [NWG P][Dv / P][NRV]
    static constexpr int RECV_BYTES = RECV_O_BYTES + NWG * kMaxSplit * NRV * 8;
    static constexpr int OFF_RECV = (MISC_END + 127) / 128 * 128;
    static constexpr int OFF_WTAB = OFF_RECV + RECV_BUFS * RECV_BYTES;
    static constexpr int OFF_STAGE = 0;
    static constexpr int OFF_OUT = MULTI ? (OFF_WTAB + NWG * kMaxSplit * NRV * 4 + 127) / 128 * 128 : TILE_BYTES;
    static constexpr int END_MULTI = OFF_OUT + OUT_BYTES;
    static constexpr int SMEM_BYTES = (MULTI ? END_MULTI : MISC_END) + 1024;
    static_assert(NSLOT >= 2, "ring of at least one K and one V tile");
    static_assert(OFF_Q % 1024 == 0 && OFF_P % 1024 == 0, "swizzle atoms on 1024 bytes");
    static_assert(OFF_OUT % 128 == 0, "TMA store source on 128 bytes");
    // 227 KB of dynamic shared memory per CTA; two CTAs of the shallow ring
    // share an SM's 228 KB, each with 1 KB reserved by the system.
    static_assert(SMEM_BYTES <= 232448, "dynamic shared memory per CTA");
    static_assert(MULTI || 2 * (SMEM_BYTES + 1024) <= 233472, "two CTAs per SM");
};

// One unit of work: the query rows of kv head `kvh` of sequence `b`, units
// numbered u = b * Hkv + kvh. Cluster c of G takes units c, c + G, c + 2G, ...
struct Unit {
    int u, b, kvh, L;
};

// Advances w.u to this cluster's next unit that this launch handles (with
// the per-sequence split rule, sequences of another split are skipped) and
// fills in the rest; false when none is left. Every role of the CTA walks
// the same sequence of units.
__device__ __forceinline__ bool next_unit(const DecodeParams& p, int stride, int n_units, Unit& w, bool report)
{
    for (; w.u < n_units; w.u += stride) {
        const int b = w.u / p.num_kv_heads;
        int L = p.seq_lens[b];
        if (L < 0) {
            if (report) atomicOr(p.status, FA_STATUS_BAD_PAGE);
            L = 0;
        }
        if (p.auto_split && auto_split_for_len(L) != p.splitk) continue;
        w.b = b;
        w.kvh = w.u - b * p.num_kv_heads;
        w.L = L;
        return true;
    }
    return false;
}

// The unit after w: advances w.u by one stride, then as next_unit.
__device__ __forceinline__ bool next_unit_after(const DecodeParams& p, int stride, int n_units, Unit& w, bool report)
{
    w.u += stride;
    return next_unit(p, stride, n_units, w, report);
}

// The per-sequence split in one launch (FA4Config page, field
// dynamic_cluster_dim: the cluster size a sequence uses is chosen at run
// time). Every cluster has 4 CTAs. The (sequence, kv head) units are ordered
// by the split their sequence takes (4, then 2, then 1; by unit index within
// a split) and cut into groups: one unit of split 4, two of split 2 or four of
// split 1; cluster c serves group c. Each CTA learns its unit, its split P,
// its partition index within the unit and the cluster rank of the unit's
// first partition; a CTA of a group that runs out of units is idle (it takes
// part in the cluster barriers only). Called by every lane of a warp; every
// warp of every CTA of the cluster reaches the same answer.
struct DynSlot {
    bool active;  // the cluster serves a group
    bool idle;    // this CTA serves no unit of it
    int P, rank, rbase, u;
};

__device__ __forceinline__ DynSlot dyn_group(const DecodeParams& p, int c, int x)
{
    const int lane = threadIdx.x & 31;
    // Sequences per split class, 32 at a time.
    int n4 = 0, n2 = 0, n1 = 0;
    for (int b0 = 0; b0 < p.batch; b0 += 32) {
        const int b = b0 + lane;
        const int P = b < p.batch ? auto_split_for_len(max(p.seq_lens[b], 0)) : 0;
        n4 += __popc(__ballot_sync(0xffffffffu, P == 4));
        n2 += __popc(__ballot_sync(0xffffffffu, P == 2));
        n1 += __popc(__ballot_sync(0xffffffffu, P == 1));
    }
    const int H = p.num_kv_heads;
    const int g4 = n4 * H, g2 = (n2 * H + 1) / 2, g1 = (n1 * H + 3) / 4;
    DynSlot d{false, true, 1, 0, 0, 0};
    int cls, k;  // split class and the index of this CTA's unit within it
    if (c < g4) {
        cls = 4; k = c;
    } else if (c < g4 + g2) {
        cls = 2; k = 2 * (c - g4) + x / 2;
    } else if (c < g4 + g2 + g1) {
        cls = 1; k = 4 * (c - g4 - g2) + x;
    } else {
        return d;  // the same for every CTA of the cluster
    }
    d.active = true;
    d.P = cls;
    d.rank = x % cls;
    d.rbase = x - d.rank;
    if (k >= (cls == 4 ? n4 : cls == 2 ? n2 : n1) * H) return d;  // idle
    // The (k / H)-th sequence of the class, kv head k % H.
    int want = k / H, b_sel = -1;
    for (int b0 = 0; b0 < p.batch && b_sel < 0; b0 += 32) {
        const int b = b0 + lane;
        const int P = b < p.batch ? auto_split_for_len(max(p.seq_lens[b], 0)) : 0;
        const unsigned m = __ballot_sync(0xffffffffu, P == cls);
        const int n = __popc(m);
        if (want < n) b_sel = b0 + (int)__fns(m, 0, want + 1);
        else want -= n;
    }
    d.idle = false;
    d.u = b_sel * H + k % H;
    return d;
}

// Warp reduce-scatter of N per-row values (max or sum over the warp's 32
// lanes): recursive halving exchanges half of the remaining rows at each of
// the first log2(N) steps, then a butterfly finishes. On return v[0] holds
// the reduction of row `row`; lanes whose low (32 / N) bits are zero hold
// distinct rows.
template <bool kMax>
__device__ __forceinline__ float rs_op(float a, float b) { return kMax ? fmaxf(a, b) : a + b; }

template <int N, int W, bool kMax, int M>
__device__ __forceinline__ void reduce_scatter_step(float (&v)[M], int lane, int& row)
{
    if constexpr (N > 1) {
        const bool up = (lane & W) != 0;
#pragma unroll
        for (int k = 0; k < N / 2; ++k) {
            const float send = up ? v[k] : v[k + N / 2];
            const float keep = up ? v[k + N / 2] : v[k];
            v[k] = rs_op<kMax>(keep, __shfl_xor_sync(0xffffffffu, send, W));
        }
        row += up ? N / 2 : 0;
        reduce_scatter_step<N / 2, W / 2, kMax, M>(v, lane, row);
    } else {
#pragma unroll
        for (int w = W; w >= 1; w >>= 1) v[0] = rs_op<kMax>(v[0], __shfl_xor_sync(0xffffffffu, v[0], w));
    }
}

template <int N, bool kMax>
__device__ __forceinline__ float warp_reduce_scatter(const float (&in)[N], int lane, int& row)
{
    float v[N];
#pragma unroll
    for (int k = 0; k < N; ++k) v[k] = in[k];
    row = 0;
    reduce_scatter_step<N, 16, kMax, N>(v, lane, row);
    return v[0];
}

// Load order of a unit's n tiles with V lagging D tiles behind K: K0 .. K_D,
// then V_t K_{t+D+1} for t = 0 .. n-D-2, then the remaining V in order; for
// D = 1: K0 K1 V0 K2 V1 ... K_{n-1} V_{n-2} V_{n-1}. A later V spends less
// time in the ring waiting for its P.
template <int D>
__device__ __forceinline__ int k_item(int i) { return i <= D ? i : 2 * i - D; }
template <int D>
__device__ __forceinline__ int v_item(int t, int n) { return t <= n - D - 2 ? D + 1 + 2 * t : n + t; }
// Inverse: the tile and kind of position j.
template <int D>
__device__ __forceinline__ void item_at(int j, int n, bool& is_v, int& t)
{
    if (j < min(n, D + 1)) {
        is_v = false;
        t = j;
        return;
    }
    const int m = j - (D + 1);
    if (m < 2 * (n - D - 1)) {
        is_v = (m & 1) == 0;
        t = is_v ? (m >> 1) : ((m - 1) >> 1) + D + 1;
    } else {
        is_v = true;
        t = j - n;
    }
}

// Lazy rescaling: the running max of a row moves only when a tile's max
// exceeds it by more than TcCfg::RESCALE exp2 units, so most tiles skip the
// correction; P then stays below 2^RESCALE (2^8 for bf16; 2^4 for the fp8
// split of P).


// SK: the stream-K partition (DecodeParams::sk_tiles; deep ring only).
// FP8: the E4M3 cache (DecodeParams::k_scale: per-token K scales or NULL).
template <int NS32, int NRV, bool SK, bool FP8>
__global__ void __launch_bounds__(TcCfg<NS32, NRV, FP8>::THREADS, TcCfg<NS32, NRV, FP8>::MULTI ? 1 : 2)
    tc_decode_kernel(const __grid_constant__ DecodeParams p)
{
    static_assert(!SK || TcCfg<NS32, NRV, FP8>::MULTI, "stream-K needs the multi-unit variant");
    using C = TcCfg<NS32, NRV, FP8>;
    constexpr int NSLOT = C::NSLOT;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
    const uint32_t sbase = smem_addr(smem);

    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;
    const int CL = p.splitk;  // CTAs per cluster
    // This CTA's split partition: P partitions of a unit, this one `rank`, the
    // unit's first partition at cluster rank rbase (0 unless the cluster
    // serves several units of a smaller split, see dyn_group).
    int P = CL, rank = (int)blockIdx.x, rbase = 0;
    const int n_units = p.batch * p.num_kv_heads;
    const int cluster_id = (int)(blockIdx.y + gridDim.y * blockIdx.z);
    const int n_clusters = (int)(gridDim.y * gridDim.z);
    // This cluster's units: c, c + G, ... or, under the stream-K partition,
    // the one or two its tile range touches.
    int u_first = cluster_id, u_step = n_clusters, u_end = n_units;
    int64_t sk_g0 = 0, sk_g1 = 0;  // the cluster's stream-K tile range
    if constexpr (SK) {
        sk_g0 = sk_begin(p.sk_total, p.sk_clusters, cluster_id);
        sk_g1 = sk_begin(p.sk_total, p.sk_clusters, cluster_id + 1);
        u_first = (int)(sk_g0 / p.sk_tiles);
        u_end = sk_g1 > sk_g0 ? (int)((sk_g1 - 1) / p.sk_tiles) + 1 : u_first;
        u_step = 1;
    }

    bool idle = false;  // (dynamic groups) this CTA serves no unit
    if constexpr (!C::MULTI) {
        if (p.dyn_split) {
            grid_dependency_wait();  // seq_lens may come from the previous kernel
            const DynSlot d = dyn_group(p, cluster_id, (int)blockIdx.x);
            if (!d.active) return;  // the same in every CTA of the cluster
            P = d.P;
            rank = d.rank;
            rbase = d.rbase;
            idle = d.idle;
            u_first = idle ? 0 : d.u;
            u_end = idle ? 0 : d.u + 1;
            u_step = 1;
        }
    }

    // Optional timeline trace (a profiling aid): one thread writes each event.
    const int64_t cta_lin = (int64_t)blockIdx.x + (int64_t)gridDim.x * (blockIdx.y + (int64_t)gridDim.y * blockIdx.z);
    unsigned long long* const trace =
        (p.trace != nullptr && cta_lin < p.trace_ctas) ? p.trace + cta_lin * FA_TRACE_WORDS_PER_CTA : nullptr;
    auto stamp = [&](int slot) {
        if (trace) trace[slot] = global_timer_ns();
    };
    constexpr int kTraceUnits = 7;
    auto unit_slot = [](int k, int e) { return 4 + 8 * k + e; };
    if (tid == 0) stamp(0);
    if (warp == 0 && lane == 0) {
        tma_prefetch_map(&p.tm_k);
        tma_prefetch_map(&p.tm_v);
    }

    // Tiles [tile_begin, tile_begin + tile_count) of unit u (length L) belong
    // to this rank: its share of all the unit's tiles or, under the stream-K
    // partition, of those in the cluster's range (clipped to L).
    auto rank_tiles = [&](int u, int L, int& tile_begin, int& tile_count) {
        int n_tiles = (L + C::BN - 1) / C::BN, t0 = 0;
        if constexpr (SK) {
            const int64_t base = (int64_t)u * p.sk_tiles;
            t0 = (int)min((int64_t)n_tiles, max(sk_g0, base) - base);
            n_tiles = max((int)min((int64_t)n_tiles, min(sk_g1, base + p.sk_tiles) - base) - t0, 0);
        }
        const int base = n_tiles / P, rem = n_tiles % P;
        tile_begin = t0 + rank * base + min(rank, rem);
        tile_count = base + (rank < rem ? 1 : 0);
    };
    // Page-table entries reach the load warp in warp-wide blocks: lane l
    // holds the entry of (tile tb + l / segs, page segment l % segs) of the
    // block starting at tile tb, fetched one block ahead, and a tile's entries
    // are shuffled out of it. The first block is fetched before the sequence
    // length is known, guessing that the sequence fills its page-table row;
    // the guess is checked once the length has arrived, so the two reads
    // overlap instead of following one another.
    const int segs = C::BN / p.box_rows;  // page segments per tile: 1, 2, 4, 8 or 16
    const int tpb = 32 / segs;            // tiles per block of page entries
    int spec_begin = -1, spec_count = 0, spec_raw = -1;
    grid_dependency_wait();  // inputs may come from the previous kernel in the stream
    grid_dependency_launch();
    if (warp == 0 && u_first < u_end && p.max_pages <= INT32_MAX / C::BN / p.page_size) {
        int gb, gc;
        rank_tiles(u_first, p.max_pages * p.page_size, gb, gc);
        spec_begin = gb;
        spec_count = gc;
        const int b0 = u_first / p.num_kv_heads;
        const int t = lane / segs;
        const int pslot = ((gb + t) * C::BN + (lane % segs) * p.box_rows) / p.page_size;
        if (t < gc && pslot < p.max_pages) spec_raw = p.page_table[(int64_t)b0 * p.max_pages + pslot];
    }
    if (u_first >= u_end && !idle) return;  // (grids never have more clusters than units or ranges)
    // The cluster's first unit (its sequence length), read by every thread
    // now: a role that read it later would wait behind the ring's first
    // copies, which the load warp is about to queue (measured: 6 us on the
    // MMA warp at the start of a cold launch).
    Unit first_unit{u_first, 0, 0, 0};
    const bool have_first = u_first < u_end && next_unit(p, u_step, u_end, first_unit, tid == 0 && rank == 0);
    // A cluster with no unit in this launch (the per-sequence split gives its
    // sequences to another launch) leaves at once; the decision is the same in
    // every CTA of the cluster.
    if (p.auto_split && !have_first) return;

    const uint32_t bar0 = sbase + C::OFF_BAR;
    const uint32_t slot_full = bar0, slot_empty = bar0 + 8 * NSLOT;
    const uint32_t s_full = bar0 + 16 * NSLOT, s_empty = s_full + 16;
    const uint32_t q_full = s_full + 80, q_empty = s_full + 96;
    const uint32_t publish_bar = s_full + 112, mma_done = s_full + 120, tmem_ready = s_full + 128;
    const uint32_t recv_full = s_full + 136, recv_free = s_full + 152;
    // fp8: the per-token K scale ring (entry = global K tile index % KS)
    const uint32_t ks_full = bar0 + 8 * (2 * NSLOT + 22), ks_empty = ks_full + 8 * C::KS;
    // P / O buffers, by global tile index gi: buffer gi % NPB, phase (gi / NPB) & 1
    const uint32_t p_full = ks_empty + 8 * C::KS, o_full = p_full + 8 * C::NPB, o_empty = o_full + 8 * C::NPB;
    const uint32_t o_buf = o_empty + 8 * C::NPB;  // O_BUF_BAR: O products by P buffer
    float* ks_s = reinterpret_cast<float*>(smem + C::OFF_KS);
    volatile uint32_t* tmem_slot = reinterpret_cast<volatile uint32_t*>(smem + C::OFF_MISC);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 4);
    // Ring-order progress of the two MMA warps: the global index of the next
    // K (resp. V) item each will consume; every earlier item of its kind has
    // been consumed.
    const uint32_t s_next = sbase + C::OFF_MISC + 8, o_next = sbase + C::OFF_MISC + 12;
    float* red_s = reinterpret_cast<float*>(smem + C::OFF_RED);  // [2][4][NRV]: by tile parity (= warpgroup)
    float2* maxsum_s = reinterpret_cast<float2*>(smem + C::OFF_MAXSUM);

    if (tid == 0) {
        for (int s = 0; s < NSLOT; ++s) {
            mbar_init(slot_full + 8 * s, 1);
            mbar_init(slot_empty + 8 * s, 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(s_full + 8 * i, 1);
            mbar_init(s_empty + 8 * i, 4);

            mbar_init(q_full + 8 * i, 4);  // one arrival per softmax warp
            mbar_init(q_empty + 8 * i, 1);
        }
        mbar_init(publish_bar, P);  // the unit's partitions
        mbar_init(mma_done, 2);
        mbar_init(tmem_ready, 1);
        for (int i = 0; i < 2; ++i) {
            // P > 1: the epilogue warp's expect_tx arrive plus the pushed bytes;
            // P == 1: the epilogue warp and the four softmax warps arrive.
            mbar_init(recv_full + 8 * i, P > 1 ? 1 : 1 + 4 * C::NWG);
            mbar_init(recv_free + 8 * i, P);  // one arrival per receiving rank
        }
        for (int i = 0; i < C::KS; ++i) {
            mbar_init(ks_full + 8 * i, 1);   // the load warp's expect_tx arrive plus the copied bytes
            mbar_init(ks_empty + 8 * i, 4);  // the four softmax warps that read the tile's scales
        }
        for (int i = 0; i < C::NPB; ++i) {
            mbar_init(p_full + 8 * i, 4);    // the four softmax warps that wrote P
            mbar_init(o_full + 8 * i, 1);    // the O warp's commit
            if (C::O_BUF_BAR) mbar_init(o_buf + 8 * i, 1);
            // o_empty[f]: the four warps of warpgroup f, once they have read its fragment at the end of a unit
            mbar_init(o_empty + 8 * i, 4);
        }
        *abort_flag = 0;
        *reinterpret_cast<volatile uint32_t*>(smem + C::OFF_MISC + 8) = 0;
        *reinterpret_cast<volatile uint32_t*>(smem + C::OFF_MISC + 12) = 0;
        fence_mbarrier_init_cluster();
    }
    __syncthreads();  // barriers initialised; the load warp may start at once
    // Peers arrive on this CTA's publish barrier only after the matching
    // cluster wait (before the first merge), so the prologue does not wait here.
    if (CL > 1) cluster_arrive_relaxed();
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

    // Softmax state (warps 3-6, 7-10), real rows only.
    float m_run[NRV], l_part[NRV];

    // Items (K or V tiles) and tiles are numbered globally over the units of
    // this cluster, so ring slots, buffers and barrier phases run on across
    // unit boundaries. Within a unit of n tiles the items come in the order
    // K0 K1 V0 K2 V1 ... K_{n-1} V_{n-2} V_{n-1}.
    int issued = 0;
    int ks_issued = 0;  // fp8: K tiles whose scale copies were issued
    if (warp == 0) {
        // ------------------------------------------------------------------ load warp
        // All 32 lanes run the loop; lane s owns page segment s of every tile.
        if (!(p.debug_flags & FA_DEBUG_SKIP_LOADS)) {
            const uint64_t policy = l2_policy_evict_first();
            int32_t* rows_s = reinterpret_cast<int32_t*>(smem + C::OFF_ROWS);
            constexpr int kNoSegment = INT32_MIN, kPastSequence = INT32_MIN + 1;
            int J0 = 0, lu = 0;
            int GT = 0;  // global index of the unit's first tile
            bool ok = true;
            Unit w = first_unit;
            for (bool on = have_first; ok && on; on = next_unit_after(p, u_step, u_end, w, tid == 0 && rank == 0), ++lu) {
                int tile_begin, tile_count;
                rank_tiles(w.u, w.L, tile_begin, tile_count);
                const int n_items = 2 * tile_count;
                // This lane's entry of the block starting at tile tb: the physical
                // page, or kNoSegment / kPastSequence (zero fill, no error); -1
                // past the page table. `raw` >= -1: that entry, already read.
                auto block_entry = [&](int tb, int raw = -2) -> int {
                    const int t = tb + lane / segs;
                    if (t >= tile_count) return kNoSegment;
                    const int key = (tile_begin + t) * C::BN + (lane % segs) * p.box_rows;
                    if (key >= w.L) return kPastSequence;
                    const int pslot = key / p.page_size;
                    if (pslot >= p.max_pages) return -1;
                    return raw >= -1 ? raw : p.page_table[(int64_t)w.b * p.max_pages + pslot];
                };
                // The guess holds when the unit's first tiles are the guessed ones
                // (then every entry block_entry needs below was read).
                const bool guessed =
                    lu == 0 && w.u == u_first && tile_begin == spec_begin && tile_count <= spec_count;
                int blk_cur = block_entry(0, guessed ? spec_raw : -2), blk_next = block_entry(tpb);
                // One pass issues one item (lanes 0-15) or, for a long unit, two
                // consecutive items (lanes 0-15 and 16-31; lane 16 h + s owns page
                // segment s), so the waits, barrier arms and copies of a pair share
                // their instructions: a long unit is bound by this warp's issue
                // rate, a short one by the ring.
                auto pass = [&](int j, auto two_tag) -> bool {
                    constexpr bool TWO = decltype(two_tag)::value;
                    // one item: every lane computes it, lane s owns segment s
                    const int half = TWO ? (lane >> 4) : 0, sl = TWO ? (lane & 15) : lane;
                    const int jh = j + half;  // this half's item in the unit
                    const bool valid = TWO ? (jh < n_items) : true;
                    const int jj = J0 + jh, slot = jj % NSLOT;
                    bool is_v = true;
                    int t = 0;
                    if (valid) item_at<C::VLAG>(jh, tile_count, is_v, t);
                    bool got = true;
                    if (valid && jj >= NSLOT)
                        got = mbar_wait(slot_empty + 8 * slot, ((jj / NSLOT) & 1) ^ 1, abort_flag, p.status,
                                        p.wait_limit_ns);
                    const bool k_here = valid && !is_v;
                    // fp8 with K scales: the K tile's scale-ring entry must have been read
                    const bool scaled = FP8 && p.k_scale != nullptr;
                    const int gk = GT + t, kse = scaled ? gk % max(C::KS, 1) : 0;
                    if (scaled && got && k_here && gk >= C::KS)
                        got = mbar_wait(ks_empty + 8 * kse, ((gk / max(C::KS, 1)) & 1) ^ 1, abort_flag, p.status,
                                        p.wait_limit_ns);
                    if (!__all_sync(0xffffffffu, got)) return false;
                    // A K tile of the pass that starts a new block of page entries.
                    int kt = k_here ? t : -1;
                    if (TWO) kt = max(kt, __shfl_xor_sync(0xffffffffu, kt, 16));  // one item: uniform already
                    if (kt > 0 && (kt & (tpb - 1)) == 0) {
                        // Waits only if the block fetched a block of tiles ago has not arrived.
                        blk_cur = blk_next;
                        blk_next = block_entry(kt + tpb);
                    }
                    const int e =
                        __shfl_sync(0xffffffffu, blk_cur, ((k_here ? t : 0) & (tpb - 1)) * segs + (sl & (segs - 1)));
                    int32_t row = p.oob_row;  // zero fill past the sequence or on a bad page
                    if (k_here) {
                        if (sl < segs) {
                            if (e >= 0 && e < p.num_pages) {
                                // the segment starts on a page boundary unless pages are longer than a tile
                                const int off = p.page_size > C::BN ? ((tile_begin + t) * C::BN) % p.page_size : 0;
                                row = (e * p.num_kv_heads + w.kvh) * p.page_size + off;
                            } else if (e != kNoSegment && e != kPastSequence) {
                                atomicOr(p.status, FA_STATUS_BAD_PAGE);
                            }
                        }
                        if (sl < 16) rows_s[(t & 3) * 16 + sl] = row;  // read by V_t, at most 3 tiles later
                    }
                    // A one-tile unit has K0 and V0 side by side, possibly in one pass:
                    // the K half's rows are written before the V half reads them.
                    if (TWO) __syncwarp();
                    if (valid && is_v) row = sl < 16 ? rows_s[(t & 3) * 16 + sl] : p.oob_row;
                    if constexpr (FP8) {
                        if (scaled) {
                            // The K tile's per-token scales: one bulk copy per page segment
                            // with a valid page; the other segments read zeros.
                            const bool seg_copy = k_here && sl < segs && row != p.oob_row;
                            const unsigned bal = __ballot_sync(0xffffffffu, seg_copy);
                            const unsigned half_mask = TWO ? (0xffffu << (16 * half)) : 0xffffffffu;
                            float* ks_dst = ks_s + kse * C::BN + sl * p.box_rows;
                            if (k_here && sl < segs && !seg_copy)
                                for (int i = 0; i < p.box_rows; i += 4)
                                    *reinterpret_cast<float4*>(ks_dst + i) = make_float4(0.f, 0.f, 0.f, 0.f);
                            __syncwarp();
                            if (k_here && sl == 0)
                                mbar_arrive_expect_tx(ks_full + 8 * kse,
                                                      (uint32_t)(__popc(bal & half_mask) * p.box_rows * 4));
                            __syncwarp();
                            if (seg_copy)
                                bulk_load(smem_addr(ks_dst), p.k_scale + row, (uint32_t)(p.box_rows * 4),
                                          ks_full + 8 * kse);
                            ks_issued = __reduce_max_sync(0xffffffffu, k_here ? gk + 1 : ks_issued);
                        }
                    }
                    if (valid && sl == 0) mbar_arrive_expect_tx(slot_full + 8 * slot, C::TILE_BYTES);
                    __syncwarp();
                    issued = J0 + (TWO ? min(j + 2, n_items) : j + 1);
                    if (valid && sl < segs) {
                        const CUtensorMap* map = is_v ? &p.tm_v : &p.tm_k;
                        const uint32_t dst = sbase + C::OFF_RING + slot * C::TILE_BYTES + sl * p.box_rows * 128;
                        tma_load_2d(dst, map, 0, row, slot_full + 8 * slot, policy);
                        if constexpr (C::BOXES == 2)
                            tma_load_2d(dst + C::BOX_BYTES, map, 64, row, slot_full + 8 * slot, policy);
                    }
                    return true;
                };
                if (n_items > 0 && lane == 0) {
                    if (J0 == 0) stamp(1);
                    if (lu < kTraceUnits) stamp(unit_slot(lu, 7));
                }
                if (tile_count >= C::PAIR_TILES) {
                    for (int j = 0; ok && j < n_items; j += 2) ok = pass(j, std::true_type{});
                } else {
                    for (int j = 0; ok && j < n_items; ++j) ok = pass(j, std::false_type{});
                }
                J0 += n_items;
                GT += tile_count;
            }
        }
    } else if (warp == 1 || warp == 2) {
        // ------------------------------------------------------------ MMA warps
        // One warp issues tcgen05.mma only every ~60 cycles, so the products go
        // to two warps: warp 1 issues every S_i = K_i Q^T, warp 2 every
        // O_t = V_t^T P_t^T. Each commits a tile's products twice: to the
        // softmax warps' barrier, and to the ring slot's empty barrier, which
        // frees the slot for the load warp as soon as the product completes.
        //
        // Ring-order rule: a slot's full barrier is waited on for item j only
        // after item j - NSLOT, which held the slot before, has been consumed
        // (a parity wait on a barrier whose previous phase has not completed
        // would alias with that phase). Each warp consumes its own kind in
        // order, so it waits for the other warp's published next-item index
        // to pass j - NSLOT.
        if (lane == 0) {
            const bool is_s = (warp == 1);
            const uint32_t other_next = is_s ? o_next : s_next;
            const uint32_t id_s = FP8 ? umma_idesc_e4m3_f32(128, C::MMA_N, false, false)
                                      : umma_idesc_bf16_f32(128, C::MMA_N, false, false);
            const uint64_t q_desc0 = umma_smem_desc(sbase + C::OFF_Q, 16, 1024, kLayoutSwizzle128);
            const uint64_t k_desc0 = umma_smem_desc(sbase + C::OFF_RING, 16, 1024, kLayoutSwizzle128);
            const uint32_t id_pv = FP8 ? umma_idesc_e4m3_f32(128, C::MMA_N, true, false)
                                       : umma_idesc_bf16_f32(128, C::MMA_N, true, false);
            // A = V^T, MN-major: 64-column atoms one box apart (LBO), 8-key groups 1024 B apart (SBO)
            const uint64_t v_desc0 = umma_smem_desc(sbase + C::OFF_RING, C::BOX_BYTES, 1024, kLayoutSwizzle128);
            // B = P, K-major: 64-key atoms of 16 rows x 128 B
            const uint64_t p_desc0 = umma_smem_desc(sbase + C::OFF_P, 16, 1024, kLayoutSwizzle128);
            if (!is_s) {
                mbar_wait(tmem_ready, 0, abort_flag, p.status, p.wait_limit_ns);
                tc_fence_after_sync();
                tmem = *tmem_slot;
            }
            auto ring_turn = [&](int j) -> bool {  // item j may wait on its slot
                return j < NSLOT ||
                       counter_wait(other_next, (uint32_t)(j - NSLOT), abort_flag, p.status, p.wait_limit_ns);
            };
            int J0 = 0, gt = 0, lu = 0;
            bool ok = true;
            Unit w = first_unit;
            for (bool on = have_first; ok && on; on = next_unit_after(p, u_step, u_end, w, false), ++lu) {
                int tile_begin, tile_count;
                rank_tiles(w.u, w.L, tile_begin, tile_count);
                if (is_s) {
                    ok = mbar_wait(q_full + 8 * (lu & 1), (lu >> 1) & 1, abort_flag, p.status, p.wait_limit_ns);
                    if (lu == 0) stamp(60);
                    const uint64_t qd = q_desc0 + (uint64_t)(((lu & 1) * C::Q_BYTES) >> 4);
                    for (int i = 0; ok && i < tile_count; ++i) {
                        const int gi = gt + i, j = J0 + k_item<C::VLAG>(i), slot = j % NSLOT;
                        ok = ring_turn(j) &&
                             mbar_wait(slot_full + 8 * slot, (j / NSLOT) & 1, abort_flag, p.status, p.wait_limit_ns) &&
                             (gi < 2 || mbar_wait(s_empty + 8 * (gi & 1), ((gi >> 1) - 1) & 1, abort_flag, p.status,
                                                  p.wait_limit_ns));
                        if (!ok) break;
                        if (gi == 0) stamp(61);
                        tc_fence_after_sync();
                        const uint64_t a0 = k_desc0 + (uint64_t)((slot * C::TILE_BYTES) >> 4);
                        const uint32_t d = tmem + C::TMEM_S0 + C::BUF_COLS * (gi & 1);
                        if constexpr (!FP8) {
#pragma unroll
                            for (int ks = 0; ks < C::D / 16; ++ks)
                                umma_f16_ss(d + C::ACC_COLS * (ks % C::NACC),
                                            a0 + (uint64_t)(((ks >> 2) * C::BOX_BYTES + (ks & 3) * 32) >> 4),
                                            qd + (uint64_t)(((ks >> 2) * 2048 + (ks & 3) * 32) >> 4), id_s,
                                            ks >= C::NACC);
                        } else {
                            // rows (16 Q_hi, Q_lo) x four K-steps of 32 depth columns
#pragma unroll
                            for (int ks = 0; ks < 4; ++ks)
                                umma_f8_ss(d + C::ACC_COLS * (ks % C::NACC), a0 + (uint64_t)((ks * 32) >> 4),
                                           qd + (uint64_t)((ks * 32) >> 4), id_s, ks >= C::NACC);
                        }
                        umma_commit(s_full + 8 * (gi & 1));
                        umma_commit(slot_empty + 8 * slot);  // K_i's slot is free once S_i has completed
                        st_release_u32(s_next, (uint32_t)(i + 1 < tile_count ? J0 + k_item<C::VLAG>(i + 1)
                                                                             : J0 + 2 * tile_count));
                    }
                    // Q buffer lu & 1 is read by no further product of this warp.
                    mbar_arrive(q_empty + 8 * (lu & 1));
                } else {
                    for (int t = 0; ok && t < tile_count; ++t) {
                        const int gi = gt + t, j = J0 + v_item<C::VLAG>(t, tile_count), slot = j % NSLOT;
                        // Tile t goes to the fragment of warpgroup t % NWG, whose first
                        // tile of a unit overwrites it once every warpgroup has read it
                        // for the previous unit (o_empty[f], one phase per unit).
                        const int frag = t % C::NWG;
                        const bool frag_first = t < C::NWG;
                        ok = ring_turn(j) &&
                             mbar_wait(slot_full + 8 * slot, (j / NSLOT) & 1, abort_flag, p.status, p.wait_limit_ns) &&
                             mbar_wait(p_full + 8 * (gi % C::NPB), (gi / C::NPB) & 1, abort_flag, p.status,
                                       p.wait_limit_ns) &&
                             (!frag_first || lu == 0 ||
                              mbar_wait(o_empty + 8 * frag, (lu - 1) & 1, abort_flag, p.status, p.wait_limit_ns));
                        if (!ok) break;
                        if (gi == 0) stamp(62);
                        tc_fence_after_sync();
                        const uint64_t a0 = v_desc0 + (uint64_t)((slot * C::TILE_BYTES) >> 4);
                        const uint64_t b0 = p_desc0 + (uint64_t)(((gi % C::NPB) * C::P_BYTES) >> 4);
                        const uint32_t d = tmem + C::TMEM_O0 + C::BUF_COLS * frag;
                        // Every tile but the fragment's first of the unit accumulates.
                        const bool acc_all = !frag_first;
                        if constexpr (!FP8) {
#pragma unroll
                            for (int ks = 0; ks < C::BN / 16; ++ks)
                                umma_f16_ss(d + C::ACC_COLS * (ks % C::NACC), a0 + (uint64_t)((ks * 2048) >> 4),
                                            b0 + (uint64_t)(((ks >> 2) * 2048 + (ks & 3) * 32) >> 4), id_pv,
                                            acc_all || ks >= C::NACC);
                        } else {
                            // rows (16 P_hi, P_lo) x four K-steps of 32 keys (four 8-key groups of V^T)
#pragma unroll
                            for (int ks = 0; ks < 4; ++ks)
                                umma_f8_ss(d + C::ACC_COLS * (ks % C::NACC), a0 + (uint64_t)((ks * 4096) >> 4),
                                           b0 + (uint64_t)((ks * 32) >> 4), id_pv, acc_all || ks >= C::NACC);
                        }
                        // O completion, for the softmax warps: by P buffer (o_buf with two
                        // warpgroups and four buffers, o_full with one), else by fragment
                        if constexpr (C::O_BUF_BAR)
                            umma_commit(o_buf + 8 * (gi % C::NPB));
                        else
                            umma_commit(o_full + 8 * (C::O_BAR_BY_FRAG ? frag : (gi % C::NPB)));
                        umma_commit(slot_empty + 8 * slot);  // V_t's slot is free once O_t has completed
                        st_release_u32(o_next, (uint32_t)(t + 1 < tile_count ? J0 + v_item<C::VLAG>(t + 1, tile_count)
                                                                             : J0 + 2 * tile_count));
                    }
                }
                gt += tile_count;
                J0 += 2 * tile_count;
            }
            st_release_u32(is_s ? s_next : o_next, 0xffffffffu);  // nothing more to wait for
            // mma_done expects one commit from each MMA warp: it fires once every
            // MMA of both warps has completed.
            umma_commit(mma_done);
            volatile int keep_waiting = 0;
            mbar_wait(mma_done, 0, &keep_waiting, p.status, p.wait_limit_ns);
        }
        __syncwarp();
    } else if (warp < C::EPI) {
        // ------------------------------------------------- softmax warps
        // NWG warpgroups; warpgroup g takes the unit's tiles whose index is g
        // modulo NWG and keeps its own running max, sum and TMEM O fragment; at
        // the end of a unit each pushes its own partial. Buffers of S and P are
        // indexed by the global tile index, so any warpgroup may consume any
        // buffer; the barrier phases order it.
        const int wg = (warp - C::WG0) >> 2;          // softmax warpgroup
        const int wt = tid - 32 * C::WG0 - 128 * wg;  // 0..127 within it
        const uint32_t wg_bar = 1 + wg;               // its named barrier
        const int quad = warp & 3;                    // TMEM lane quadrant of this warp
        const int my_lane = 32 * quad + lane;         // key (S) or value column (O) of this thread
        const uint32_t lane_addr = (uint32_t)(32 * quad) << 16;
        const float c2 = p.scale_log2e;
        const bool lead = wg == 0;                    // stores Q, stamps the trace, merges, pushes

        // Q rows of a unit -> K-major 128-byte-swizzled B operand; rows >= p.rows are zero.
        auto load_q = [&](const Unit& x, uint4 (&v)[2]) {
#pragma unroll
            for (int k = 0; k < 2; ++k) {
                const int idx = wt + 128 * k, r = idx >> 4, u = idx & 15;  // 16-byte chunk u of row r
                v[k] = make_uint4(0, 0, 0, 0);
                if (r < p.rows) {
                    const int t = r / p.heads_per_cta;
                    const int h = x.kvh * p.group + r % p.heads_per_cta;
                    v[k] = reinterpret_cast<const uint4*>(
                        p.q + (((int64_t)x.b * p.num_q + t) * p.num_q_heads + h) * C::D)[u];
                }
            }
        };
        // all_rows false: rows >= p.rows of the buffer hold zeros from its first
        // use, and warps whose two rows are both such rows skip them.
        auto store_q = [&](int buf, const uint4 (&v)[2], bool all_rows) {
#pragma unroll
            for (int k = 0; k < 2; ++k) {
                const int idx = wt + 128 * k, r = idx >> 4, u = idx & 15;
                if (!all_rows && (((wt & ~31) + 128 * k) >> 4) >= p.rows) continue;  // uniform over the warp
                if constexpr (!FP8) {
                    *reinterpret_cast<uint4*>(smem + C::OFF_Q + buf * C::Q_BYTES + (u >> 3) * 2048 + r * 128 +
                                              (((u & 7) ^ (r & 7)) << 4)) = v[k];
                } else {
                    // Row r scaled by sigma_r = a power of two with max |q_r| sigma_r <= 28,
                    // then split into 16 e4m3(x) and e4m3(16 (x - e4m3(x))): two K-major
                    // 128-byte-swizzled E4M3 operands [16 rows][128 B], 2 KB apart. The
                    // row's 16 chunks sit in one half-warp.
                    const uint32_t wv[4] = {v[k].x, v[k].y, v[k].z, v[k].w};
                    float x[8];
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const float2 f = bf16x2_to_float2(wv[e]);
                        x[2 * e] = f.x;
                        x[2 * e + 1] = f.y;
                    }
                    float amax = 0.f;
#pragma unroll
                    for (int e = 0; e < 8; ++e) amax = fmaxf(amax, fabsf(x[e]));
#pragma unroll
                    for (int o = 1; o < 16; o <<= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
                    const float sig = e4m3_split_scale(amax, 28.f);
                    uint32_t hi[4], lo[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        float h0, l0, h1, l1;
                        e4m3_split(x[2 * e] * sig, h0, l0);
                        e4m3_split(x[2 * e + 1] * sig, h1, l1);
                        hi[e] = e4m3x2(h0, h1);
                        lo[e] = e4m3x2(l0, l1);
                    }
                    const int off = r * 128 + ((((u >> 1) ^ (r & 7))) << 4) + (u & 1) * 8;
                    uint8_t* qb = smem + C::OFF_Q + buf * C::Q_BYTES;
                    *reinterpret_cast<uint2*>(qb + off) = make_uint2(hi[0] | (hi[1] << 16), hi[2] | (hi[3] << 16));
                    *reinterpret_cast<uint2*>(qb + 2048 + off) =
                        make_uint2(lo[0] | (lo[1] << 16), lo[2] | (lo[3] << 16));
                    if (u == 0) reinterpret_cast<float*>(smem + C::OFF_QINV)[buf * C::NR + r] = 0.0625f / sig;
                }
            }
        };

        Unit w = first_unit;
        bool have = have_first;
        if (have && lead) {
            uint4 qv[2];
            load_q(w, qv);
            store_q(0, qv, true);
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(q_full);
            if (wt == 0) stamp(63);
        }
        mbar_wait(tmem_ready, 0, abort_flag, p.status, p.wait_limit_ns);
        tc_fence_after_sync();
        tmem = *tmem_slot;

        // lanes holding distinct rows after a reduce-scatter of NRV values
        const bool row_writer = (lane & (32 / NRV - 1)) == 0;
        bool seen_abort = false;  // sticky: this thread has seen the abort flag
        bool cluster_waited = false;
        int J0 = 0, gt = 0, lu = 0;
        int wc = 0;  // two warpgroups: this warpgroup's tiles so far (phases of its o_full barrier)
        while (have) {
            const int L = w.L;
            int tile_begin, tile_count;
            rank_tiles(w.u, L, tile_begin, tile_count);
            if (lead && wt == 0 && lu < kTraceUnits) {
                stamp(unit_slot(lu, 0));
                if (trace) trace[unit_slot(lu, 6)] = (unsigned long long)tile_count;
            }
            // The next unit of this cluster: its Q rows are fetched now and
            // stored once the S warp has left the buffer's previous unit (at
            // this warpgroup's second tile of the unit), so the S warp runs
            // straight on into it.
            Unit nx = w;
            nx.u += u_step;
            const bool more = C::MULTI && next_unit(p, u_step, u_end, nx, false);
            uint4 qn[2];
            bool q_pending = more && lead;
            if (q_pending) load_q(nx, qn);
            auto put_next_q = [&]() {  // before a fence.proxy.async and the warp's q_full arrive
                if (lu >= 1)
                    mbar_wait(q_empty + 8 * ((lu + 1) & 1), ((lu - 1) >> 1) & 1, abort_flag, p.status,
                              p.wait_limit_ns);
                store_q((lu + 1) & 1, qn, lu == 0);
            };
#pragma unroll
            for (int r = 0; r < NRV; ++r) {
                m_run[r] = -INFINITY;
                l_part[r] = 0.f;
            }
            // Row r = t * heads + hh (query token t) sees keys < L - T + t + 1, so
            // the rows that see key k are a suffix: r >= (k - (L - T + 1) + 1) * heads.
            const int vis0 = L - p.num_q + 1;

            // fp8: this unit's S = acc / (16 sigma_r); its Q (and the multipliers,
            // read from shared memory at every tile) are published on the unit's
            // q_full phase.
            const float4* qinv = reinterpret_cast<const float4*>(smem + C::OFF_QINV) + (lu & 1) * (C::NR / 4);
            if constexpr (FP8) mbar_wait(q_full + 8 * (lu & 1), (lu >> 1) & 1, abort_flag, p.status, p.wait_limit_ns);
            // This warpgroup's tiles: local index i congruent to wg modulo NWG
            // (by local index, so a unit's arithmetic does not depend on the
            // units its cluster took before). Their global indices share a
            // parity, so within a unit a warpgroup uses one buffer of S, P, O
            // and red_s: (gt + wg) & 1 with two warpgroups.
            const int i0 = C::NWG == 2 ? wg : 0;
            const int gt0 = gt;
            int wc_unit = 0;   // this warpgroup's tiles of the unit so far
            for (int i = i0; i < tile_count; i += C::NWG) {
                const int gi = gt + i;
                mbar_wait(s_full + 8 * (gi & 1), (gi >> 1) & 1, abort_flag, p.status, p.wait_limit_ns);
                if (lead && wt == 0 && i == i0) {
                    if (gi == 0) stamp(2);
                    if (lu < kTraceUnits) stamp(unit_slot(lu, 1));
                }
                tc_fence_after_sync();
                float s[NRV];
                tmem_ld4_sum(tmem + lane_addr + C::TMEM_S0 + C::BUF_COLS * (gi & 1), C::PART_COLS, s);
                tc_fence_before_sync();
                __syncwarp();
                if (lane == 0) mbar_arrive(s_empty + 8 * (gi & 1));
                if constexpr (FP8) {
                    // raw scores: acc / (16 sigma_r) times this key's K scale
                    float ksc = 1.f;
                    if (p.k_scale != nullptr) {
                        const int kse = gi % C::KS;
                        mbar_wait(ks_full + 8 * kse, (gi / C::KS) & 1, abort_flag, p.status, p.wait_limit_ns);
                        ksc = ks_s[kse * C::BN + my_lane];
                        __syncwarp();
                        if (lane == 0) mbar_arrive(ks_empty + 8 * kse);
                    }
#pragma unroll
                    for (int r4 = 0; r4 < NRV / 4; ++r4) {
                        const float4 qm = qinv[r4];
                        s[4 * r4 + 0] *= qm.x * ksc;
                        s[4 * r4 + 1] *= qm.y * ksc;
                        s[4 * r4 + 2] *= qm.z * ksc;
                        s[4 * r4 + 3] *= qm.w * ksc;
                    }
                }

                const int key0 = (tile_begin + i) * C::BN;
                const int key = key0 + my_lane;
                // Causal and length mask; with 16 rows per thread, nothing to do
                // (uniformly) when every key of the tile is seen by every row and no
                // row is padding (measured: ragged_speculative_e4m3 199.7 -> 193.1 us;
                // with 4 or 8 rows the skip was no faster, long_context_e4m3 slower).
                if (NRV < 16 || key0 + C::BN > vis0 || p.rows < NRV) {
                    const int r_min = key < vis0 ? 0 : (key >= L ? NRV : (key - vis0 + 1) * p.heads_per_cta);
#pragma unroll
                    for (int r = 0; r < NRV; ++r) s[r] = ((r >= r_min) & (r < p.rows)) ? s[r] : -INFINITY;
                }

                // Lazy rescale: a row's running max moves only when some score
                // exceeds it by more than the threshold. In the common case a single
                // reducing barrier confirms that no thread needs it; otherwise the
                // tile max is exchanged and the rows that exceed are moved.
                // Evaluated without short-circuit branches: a finite score over an
                // empty row, or one more than the threshold above the row's max (a
                // masked score gives -inf or NaN there, which compares false).
                bool need = false;
#pragma unroll
                for (int r = 0; r < NRV; ++r) {
                    const bool first = (m_run[r] == -INFINITY) & (s[r] != -INFINITY);
                    const bool over = (s[r] - m_run[r]) * c2 > C::RESCALE;
                    need = need | first | over;
                }
                seen_abort |= (*abort_flag != 0);
                bool rescale = false;
                float alpha[NRV];
                if (named_barrier_or(wg_bar, 128, need || seen_abort)) {
                    {
                        int row;
                        const float wmax = warp_reduce_scatter<NRV, true>(s, lane, row);
                        if (row_writer) red_s[((gi & 1) * 4 + quad) * NRV + row] = wmax;
                    }
                    seen_abort |= (*abort_flag != 0);
                    // The abort decision is reduced over the warpgroup, so it is uniform.
                    if (named_barrier_or(wg_bar, 128, seen_abort)) {
                        seen_abort = true;
                        break;
                    }
                    float tmax[NRV];
                    const float* rq = red_s + (gi & 1) * 4 * NRV;
#pragma unroll
                    for (int r4 = 0; r4 < NRV / 4; ++r4) {
                        const float4 a0 = reinterpret_cast<const float4*>(rq)[r4];
                        const float4 a1 = reinterpret_cast<const float4*>(rq + NRV)[r4];
                        const float4 a2 = reinterpret_cast<const float4*>(rq + 2 * NRV)[r4];
                        const float4 a3 = reinterpret_cast<const float4*>(rq + 3 * NRV)[r4];
                        tmax[4 * r4 + 0] = fmaxf(fmaxf(a0.x, a1.x), fmaxf(a2.x, a3.x));
                        tmax[4 * r4 + 1] = fmaxf(fmaxf(a0.y, a1.y), fmaxf(a2.y, a3.y));
                        tmax[4 * r4 + 2] = fmaxf(fmaxf(a0.z, a1.z), fmaxf(a2.z, a3.z));
                        tmax[4 * r4 + 3] = fmaxf(fmaxf(a0.w, a1.w), fmaxf(a2.w, a3.w));
                    }
                    rescale = true;
#pragma unroll
                    for (int r = 0; r < NRV; ++r) {
                        const bool move = (m_run[r] == -INFINITY) ? (tmax[r] != -INFINITY)
                                                                  : ((tmax[r] - m_run[r]) * c2 > C::RESCALE);
                        alpha[r] = 1.f;
                        if (move) {
                            alpha[r] = (m_run[r] == -INFINITY) ? 0.f : ex2_approx((m_run[r] - tmax[r]) * c2);
                            m_run[r] = tmax[r];
                            l_part[r] *= alpha[r];
                        }
                    }
                }
                // exp2(-inf) = +0 for masked scores (a row whose max is still -inf
                // would give NaN from the difference, hence the select first).
#pragma unroll
                for (int r = 0; r < NRV; ++r) {
                    const float x = (s[r] == -INFINITY) ? -INFINITY : (s[r] - m_run[r]) * c2;
                    const float pr = ex2_approx(x);
                    l_part[r] += pr;
                    s[r] = pr;
                }

                // P -> K-major swizzled B operand of O^T = V^T P^T (rows >= NRV only
                // feed output columns that are never read). Buffer gi % NPB was last
                // read by O of global tile gi - NPB, which must have completed before
                // the store (and O(gi - 1) before a rescale of the fragment).
                if constexpr (C::O_BUF_BAR) {
                    // Four P buffers, O products counted by buffer (o_buf): the
                    // buffer's previous reader is O(gi - 4), this warpgroup's product
                    // before its previous one in the unit (earlier units' products
                    // have all been waited for at the unit's end); a rescale also
                    // waits for O(gi - 2), the fragment's previous product. Each wait
                    // is for the phase right after one already waited for on the same
                    // barrier, so no parity wait can alias.
                    if (wc_unit > 0) {
                        if (gi - C::NPB >= gt) {
                            const int gp = gi - C::NPB;
                            mbar_wait(o_buf + 8 * (gp % C::NPB), (gp / C::NPB) & 1, abort_flag, p.status,
                                      p.wait_limit_ns);
                        }
                        if (rescale) {
                            const int gp = gi - 2;
                            mbar_wait(o_buf + 8 * (gp % C::NPB), (gp / C::NPB) & 1, abort_flag, p.status,
                                      p.wait_limit_ns);
                            tc_fence_after_sync();
                            tmem_scale4<NRV>(tmem + lane_addr + C::TMEM_O0 + C::BUF_COLS * wg, C::PART_COLS, alpha);
                            tc_fence_before_sync();
                        }
                    }
                } else if constexpr (C::O_BAR_BY_FRAG) {
                    // Two P buffers: the fragment's previous O product read the buffer
                    // this tile reuses (and must finish before a rescale touches the
                    // fragment); waited for on every tile.
                    if (wc_unit > 0) {
                        mbar_wait(o_full + 8 * wg, (wc - 1) & 1, abort_flag, p.status, p.wait_limit_ns);
                        tc_fence_after_sync();
                        if (rescale) {
                            tmem_scale4<NRV>(tmem + lane_addr + C::TMEM_O0 + C::BUF_COLS * wg, C::PART_COLS, alpha);
                            tc_fence_before_sync();
                        }
                    }
                } else {
                    // One warpgroup: the product that read this P buffer, NPB tiles
                    // back, has to be complete (waited on every tile, which keeps each
                    // buffer's barrier at most one phase behind); a rescale also waits
                    // for the previous tile's O, and with it every earlier one.
                    if (gi >= C::NPB) {
                        const int gp = gi - C::NPB;
                        mbar_wait(o_full + 8 * (gp % C::NPB), (gp / C::NPB) & 1, abort_flag, p.status,
                                  p.wait_limit_ns);
                    }
                    if (rescale && i > 0) {
                        const int gp = gi - 1;
                        mbar_wait(o_full + 8 * (gp % C::NPB), (gp / C::NPB) & 1, abort_flag, p.status,
                                  p.wait_limit_ns);
                        tc_fence_after_sync();
                        tmem_scale4<NRV>(tmem + lane_addr + C::TMEM_O0, C::PART_COLS, alpha);
                        tc_fence_before_sync();
                    }
                }
                if constexpr (!FP8) {
                    uint8_t* pb = smem + C::OFF_P + (gi % C::NPB) * C::P_BYTES + (my_lane >> 6) * 2048;
                    const int kk = my_lane & 63;
#pragma unroll
                    for (int r = 0; r < NRV; ++r)
                        *reinterpret_cast<__nv_bfloat16*>(pb + r * 128 + ((((kk >> 3) ^ (r & 7))) << 4) +
                                                          (kk & 7) * 2) = __float2bfloat16_rn(s[r]);
                } else {
                    // P <= 16: the operands h = e4m3(16 P) and e4m3(16 P - h), [16 rows][128 keys],
                    // two rows per packed conversion
                    uint8_t* pb = smem + C::OFF_P + (gi % C::NPB) * C::P_BYTES + (my_lane & 15);
                    const int kc = my_lane >> 4;
#pragma unroll
                    for (int r = 0; r < NRV; r += 2) {
                        uint32_t hc, lc;
                        e4m3_split2(16.f * s[r], 16.f * s[r + 1], hc, lc);
                        const int off0 = r * 128 + ((kc ^ (r & 7)) << 4);
                        const int off1 = (r + 1) * 128 + ((kc ^ ((r + 1) & 7)) << 4);
                        pb[off0] = (uint8_t)(hc & 0xff);
                        pb[off1] = (uint8_t)(hc >> 8);
                        pb[2048 + off0] = (uint8_t)(lc & 0xff);
                        pb[2048 + off1] = (uint8_t)(lc >> 8);
                    }
                }
                // Last tile of the sequence: zero the V rows past L so that unused
                // cache rows (whatever they hold) meet P = 0 as exact zeros.
                if (key0 + C::BN > L) {
                    const int j = J0 + v_item<C::VLAG>(i, tile_count), slot = j % NSLOT;
                    mbar_wait(slot_full + 8 * slot, (j / NSLOT) & 1, abort_flag, p.status, p.wait_limit_ns);
                    if (key >= L) {
#pragma unroll
                        for (int bx = 0; bx < C::BOXES; ++bx) {
                            uint4* vrow = reinterpret_cast<uint4*>(smem + C::OFF_RING + slot * C::TILE_BYTES +
                                                                   bx * C::BOX_BYTES + my_lane * 128);
#pragma unroll
                            for (int u = 0; u < 8; ++u) vrow[u] = make_uint4(0, 0, 0, 0);
                        }
                    }
                }
                // Uniform: this warpgroup's second tile of the unit (its first when it
                // has one only), so that the next unit's Q rows, fetched at the unit's
                // start, have a tile's time to arrive.
                const bool q_now = q_pending && (i > i0 || i + C::NWG >= tile_count);
                if (q_now) put_next_q();
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive(p_full + 8 * (gi % C::NPB));
                    if (q_now) mbar_arrive(q_full + 8 * ((lu + 1) & 1));
                }
                q_pending = q_pending && !q_now;

                ++wc;
                ++wc_unit;
            }
            // Bounded even after an abort. After an abort the O of the tile
            // that broke the loop was never issued; the wait gives up at once.
            if (wc_unit > 0) {
                // The fragment's last product is complete. Counted by P buffer,
                // the warpgroup's last two products are waited for in order, so
                // that every product of the unit has been waited for on its
                // barrier before the next unit's first waits.
                if constexpr (C::O_BAR_BY_FRAG && !C::O_BUF_BAR) {
                    mbar_wait(o_full + 8 * wg, (wc - 1) & 1, abort_flag, p.status, p.wait_limit_ns);
                } else {
                    const int step = C::NWG;  // between a warpgroup's consecutive tiles
                    const uint32_t bars = C::O_BUF_BAR ? o_buf : o_full;
                    const int g_last = gt + (C::NWG == 2 ? wg : 0) + C::NWG * (wc_unit - 1);  // its last tile
                    for (int k = (wc_unit >= 2 ? 1 : 0); k >= 0; --k) {
                        const int gp = g_last - k * step;
                        mbar_wait(bars + 8 * (gp % C::NPB), (gp / C::NPB) & 1, abort_flag, p.status,
                                  p.wait_limit_ns);
                    }
                }
                tc_fence_after_sync();
            }
            if (lead && wt == 0 && lu < kTraceUnits) stamp(unit_slot(lu, 2));
            gt += tile_count;
            J0 += 2 * tile_count;
            if (q_pending) {  // no tile stored it (no tiles, or an abort in the first)
                put_next_q();
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(q_full + 8 * ((lu + 1) & 1));
            }

            // ---------------------------------------------------- unit epilogue
            // Row sums: per-thread partial sums -> warp reduce-scatter -> four
            // warps, in this warpgroup's half of red_s.
            float* red_w = red_s + (C::NWG == 2 ? ((gt0 + wg) & 1) : 0) * 4 * NRV;
            {
                int row;
                const float wsum = warp_reduce_scatter<NRV, false>(l_part, lane, row);
                named_barrier_sync(wg_bar, 128);  // red_s may still be read by the last tile's max step
                if (row_writer) red_w[quad * NRV + row] = wsum;
                named_barrier_sync(wg_bar, 128);
            }
            float lrow[NRV];
#pragma unroll
            for (int r = 0; r < NRV; ++r) lrow[r] = red_w[r] + red_w[NRV + r] + red_w[2 * NRV + r] + red_w[3 * NRV + r];
            {
                // This thread's value column of the warpgroup's O fragment (zero
                // when the warpgroup has no tiles of the unit: the fragment still
                // holds an earlier unit's O); then the O warp may overwrite it.
                // With two warpgroups each pushes its fragment as a partial of its
                // own, (O_w / l_w, m_w, l_w), and the epilogue warp's LSE combine
                // takes the 2P partials of the unit, so neither warpgroup waits for
                // the other at the end of a unit.
                float o_acc[NRV];
#pragma unroll
                for (int r = 0; r < NRV; ++r) o_acc[r] = 0.f;
                if (wc_unit > 0) {
                    tmem_ld4_sum(tmem + lane_addr + C::TMEM_O0 + C::BUF_COLS * wg, C::PART_COLS, o_acc);
                    if constexpr (FP8) {
#pragma unroll
                        for (int r = 0; r < NRV; ++r) o_acc[r] *= 0.0625f;  // the P split carries a factor 16
                    }
                }
                tc_fence_before_sync();
                __syncwarp();
                if (lane == 0) mbar_arrive(o_empty + 8 * wg);
                const int BW = p.ov_depth / P;  // this partition's output band
                const int dv = my_lane;
                if constexpr (C::MULTI) {
                    // Push this warpgroup's normalised partial (chunk NWG rank + wg)
                    // into the band owners' receive buffers (see
                    // splitk_merge_pushed) and go on with the next unit; the
                    // epilogue warp merges.
                    const int rb = lu % C::RECV_BUFS, rk = lu / C::RECV_BUFS;
                    // Every receiver has finished with this buffer's previous unit.
                    if (rk >= 1)
                        mbar_wait<true>(recv_free + 8 * rb, (rk - 1) & 1, abort_flag, p.status, p.wait_limit_ns);
                    if (P > 1 && !cluster_waited) {
                        cluster_wait();  // every rank's barriers are initialised
                        cluster_waited = true;
                    }
                    float v[NRV];
#pragma unroll
                    for (int r = 0; r < NRV; ++r) v[r] = lrow[r] > 0.f ? o_acc[r] * __frcp_rn(lrow[r]) : 0.f;
                    const uint32_t recv0 = sbase + C::OFF_RECV + rb * C::RECV_BYTES;
                    const int q = dv / BW, col = dv % BW;
                    const int chunk = C::NWG * rank + wg;
                    const uint32_t o_dst = recv0 + 4u * (uint32_t)((chunk * BW + col) * NRV);
                    if (P > 1) {
                        const uint32_t bar_q = map_shared_rank(recv_full + 8 * rb, q);
                        const uint32_t dst_q = map_shared_rank(o_dst, q);
#pragma unroll
                        for (int r4 = 0; r4 < NRV / 4; ++r4)
                            st_async_f4(dst_q + 16 * r4, v[4 * r4], v[4 * r4 + 1], v[4 * r4 + 2], v[4 * r4 + 3],
                                        bar_q);
                        for (int idx = wt; idx < P * NRV; idx += 128) {
                            const int qq = idx / NRV, rr = idx % NRV;
                            float mm = 0.f, ll = 0.f;
#pragma unroll
                            for (int r = 0; r < NRV; ++r)
                                if (r == rr) {
                                    mm = m_run[r];
                                    ll = lrow[r];
                                }
                            const uint32_t ms_dst = recv0 + C::RECV_O_BYTES + 8u * (uint32_t)(chunk * NRV + rr);
                            st_async_f2(map_shared_rank(ms_dst, qq), mm, ll, map_shared_rank(recv_full + 8 * rb, qq));
                        }
                    } else {
                        float* o_loc = reinterpret_cast<float*>(smem + (o_dst - sbase));
#pragma unroll
                        for (int r4 = 0; r4 < NRV / 4; ++r4)
                            reinterpret_cast<float4*>(o_loc)[r4] =
                                make_float4(v[4 * r4], v[4 * r4 + 1], v[4 * r4 + 2], v[4 * r4 + 3]);
                        if (wt == 0) {
                            float2* ms_loc = reinterpret_cast<float2*>(smem + (recv0 - sbase) + C::RECV_O_BYTES);
#pragma unroll
                            for (int r = 0; r < NRV; ++r) ms_loc[chunk * NRV + r] = make_float2(m_run[r], lrow[r]);
                        }
                        __syncwarp();
                        if (lane == 0) mbar_arrive(recv_full + 8 * rb);
                    }
                    if (lead && wt == 0 && lu < kTraceUnits) stamp(unit_slot(lu, 3));
                } else {
                    float* stage_s = reinterpret_cast<float*>(smem + C::OFF_STAGE);
                    const int q = dv / BW, jc = dv % BW;
#pragma unroll
                    for (int r = 0; r < NRV; ++r) {
                        if (wt == 0) maxsum_s[r] = make_float2(m_run[r], lrow[r]);
                        float inv = 0.f;
                        if (lrow[r] > 0.f) inv = __frcp_rn(lrow[r]);  // uniform: no divergence
                        stage_s[(q * NRV + r) * BW + jc] = o_acc[r] * inv;
                    }
                    if (wt == 0 && lu < kTraceUnits) stamp(unit_slot(lu, 3));
                    named_barrier_sync(wg_bar, 128);
                    if (CL > 1) {
                        cluster_wait();  // every rank's publish barrier is initialised
                        cluster_waited = true;
                    }
                    if (wt == 0 && lu < kTraceUnits) stamp(unit_slot(lu, 4));
                    splitk_merge_and_store<NRV>(p, P, rank, w.b, w.kvh, 0, stage_s, maxsum_s,
                                                reinterpret_cast<uint16_t*>(smem + C::OFF_OUT), publish_bar, 0u,
                                                0u, abort_flag, wt, 128, wg_bar, rbase, BW);
                    if (wt == 0 && lu < kTraceUnits) stamp(unit_slot(lu, 5));
                }
            }
            ++lu;
            // Uniform over the softmax warpgroups: stop after an abort.
            seen_abort |= (*abort_flag != 0);
            if (named_barrier_or(C::NWG == 2 ? 3 : wg_bar, 128 * C::NWG, seen_abort) || !more) break;
            w = nx;
        }
        if (CL > 1 && !cluster_waited) cluster_wait();  // pairs with the early arrive
        tc_fence_before_sync();
    } else {
        // ------------------------------------------- epilogue warp (multi-unit variant)
        // Merges each unit's pushed partials and stores the output band while
        // the softmax warps work on the next unit.
        bool cluster_waited = false;
        int lu = 0;
        Unit w = first_unit;
        const uint32_t expect = (uint32_t)pushed_bytes(C::NWG * P, p.band_cols, NRV);
        for (bool on = have_first; on; on = next_unit_after(p, u_step, u_end, w, false), ++lu) {
            const int rb = lu % C::RECV_BUFS, rk = lu / C::RECV_BUFS;
            if (P > 1 && !cluster_waited) {
                cluster_wait();  // every rank's barriers are initialised
                cluster_waited = true;
            }
            // This buffer's previous phase completed (this warp waited for it),
            // so the arrival belongs to this unit's phase; pushed bytes that
            // landed earlier are already counted against it.
            if (lane == 0) {
                if (P > 1)
                    mbar_arrive_expect_tx(recv_full + 8 * rb, expect);
                else
                    mbar_arrive(recv_full + 8 * rb);
            }
            const bool got = mbar_wait<true>(recv_full + 8 * rb, rk & 1, abort_flag, p.status, p.wait_limit_ns);
            if (!__all_sync(0xffffffffu, got)) break;
            if (lane == 0 && lu < kTraceUnits) stamp(unit_slot(lu, 4));
            const uint8_t* recv = smem + C::OFF_RECV + rb * C::RECV_BYTES;
            if constexpr (SK)
                splitk_merge_pushed_sk<NRV>(p, P, rank, w.b, w.kvh, w.u, cluster_id,
                                            reinterpret_cast<const float*>(recv),
                                            reinterpret_cast<const float2*>(recv + C::RECV_O_BYTES),
                                            reinterpret_cast<float*>(smem + C::OFF_WTAB),
                                            reinterpret_cast<uint16_t*>(smem + C::OFF_OUT), lane, C::NWG * P);
            else
                splitk_merge_pushed<NRV>(p, P, rank, w.b, w.kvh, reinterpret_cast<const float*>(recv),
                                         reinterpret_cast<const float2*>(recv + C::RECV_O_BYTES),
                                         reinterpret_cast<float*>(smem + C::OFF_WTAB),
                                         reinterpret_cast<uint16_t*>(smem + C::OFF_OUT), lane, C::NWG * P);
            // Release the buffer to every sender: all lanes' reads of it are
            // complete (their results are in the band); one fence orders them
            // ahead of the senders' next pushes, then relaxed arrives. Only a
            // unit RECV_BUFS later reuses the buffer: near the end there is
            // none, and the cluster-scope fence is left out.
            Unit later = w;
            bool reused = true;
            for (int k = 0; reused && k < C::RECV_BUFS; ++k) reused = next_unit_after(p, u_step, u_end, later, false);
            __syncwarp();
            if (lane == 0 && reused) {
                if (P > 1) {
                    fence_acq_rel_cluster();
                    for (int q = 0; q < P; ++q) mbar_arrive_cluster_relaxed(map_shared_rank(recv_free + 8 * rb, q));
                } else {
                    mbar_arrive(recv_free + 8 * rb);
                }
            }
            if (lane == 0 && lu < kTraceUnits) stamp(unit_slot(lu, 5));
        }
        if (lane == 0) tma_store_wait_read();  // the last band has been read out of shared memory
        __syncwarp();
        if (P > 1 && !cluster_waited) cluster_wait();  // pairs with the early arrive
    }

    // All TMEM reads and MMAs are complete (the MMA lanes waited for mma_done).
    __syncthreads();
    if (warp == 1) {
        tc_fence_after_sync();
        tmem_dealloc(tmem, C::TMEM_COLS);
    }
    if (warp == 0 && lane == 0 && *abort_flag) {
        // Gave up early: wait (bounded) until the copies of the last NSLOT
        // issued items have landed, so none is in flight when the CTA exits.
        volatile int keep_waiting = 0;
        for (int j = issued > NSLOT ? issued - NSLOT : 0; j < issued; ++j)
            mbar_wait(slot_full + 8 * (j % NSLOT), (j / NSLOT) & 1, &keep_waiting, p.status, p.wait_limit_ns);
        for (int g = ks_issued > C::KS ? ks_issued - C::KS : 0; g < ks_issued; ++g)
            mbar_wait(ks_full + 8 * (g % C::KS), (g / C::KS) & 1, &keep_waiting, p.status, p.wait_limit_ns);
    }
    if (CL > 1 && warp < C::WG0) cluster_wait();  // pairs with the early arrive (the other warps waited above)
    __syncwarp();
    if (CL > 1) cluster_sync_all();  // peers may still read this CTA's staged bands until here
    if (tid == 0) stamp(3);
}

// Geometry of the variant (NS32, NRV, FP8); stream_k selects the stream-K
// instantiation (deep ring only).
template <int NS32, int NRV, bool FP8>
inline void tc_variant(bool stream_k, const char* name, KernelGeometry* g)
{
    using C = TcCfg<NS32, NRV, FP8>;
    if constexpr (C::MULTI)
        g->func = stream_k ? reinterpret_cast<const void*>(&tc_decode_kernel<NS32, NRV, true, FP8>)
                           : reinterpret_cast<const void*>(&tc_decode_kernel<NS32, NRV, false, FP8>);
    else
        g->func = reinterpret_cast<const void*>(&tc_decode_kernel<NS32, NRV, false, FP8>);
    g->threads = C::THREADS;
    g->keys_per_tile = C::BN;
    g->stages = C::NSLOT;
    g->rows_capacity = NRV;
    g->smem_bytes = C::SMEM_BYTES;
    g->name = name;
}

}  // namespace fad
