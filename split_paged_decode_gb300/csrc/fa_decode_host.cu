// fa_decode_host.cu -- the C ABI of libfa_decode.so: argument validation, the
// launch plan, TMA tensor-map encoding and the cluster launches.
//
// The plan mirrors the FA4Config page (Modular MAX docs): a handle fixes the
// geometry of one shape family the way the FA4Config constructor and its
// with_num_q / with_splitk reconstructors do, `supported()` becomes the
// FA_ERR_UNSUPPORTED checks below, cluster_size() is the split-K partition
// count, and description() is fa_decode_describe().
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <string>
#include <vector>

#include "fa_decode_internal.h"
#include "stream_k_plan.h"

namespace {

thread_local std::string g_last_error;

// The one-launch per-sequence split reads every length in every CTA; above
// this batch the planner keeps one launch per cluster size.
constexpr int kDynSplitMaxBatch = 4096;

int fail(int code, const char* fmt, ...)
{
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    g_last_error = buf;
    return code;
}

int cuda_fail(cudaError_t e, const char* what)
{
    return fail(FA_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
}

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_tiled_fn()
{
    static std::once_flag once;
    static EncodeTiledFn fn = nullptr;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

bool is_aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// Cache of one encoded tensor map, keyed by what it was encoded from.
struct MapCache {
    bool valid = false;
    const void* ptr = nullptr;
    uint64_t key0 = 0, key1 = 0, key2 = 0;
    CUtensorMap map;
};

// Tensor map over the K (or V) rows of the paged cache: [num_pages*Hkv*PS][depth]
// elements of `elem` bytes (2: bf16, 1: E4M3 codes), boxes of 128 bytes x
// box_rows rows, 128-byte swizzle, zero fill.
int encode_cache_map(MapCache& c, const void* base, int depth, int64_t rows, int box_rows, int elem = 2)
{
    const uint64_t k2 = ((uint64_t)elem << 32) | (uint64_t)box_rows;
    if (c.valid && c.ptr == base && c.key0 == (uint64_t)depth && c.key1 == (uint64_t)rows && c.key2 == k2)
        return FA_OK;
    EncodeTiledFn enc = encode_tiled_fn();
    if (!enc) return fail(FA_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
    cuuint64_t dims[2] = {(cuuint64_t)depth, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)depth * elem};
    cuuint32_t box[2] = {(cuuint32_t)(128 / elem), (cuuint32_t)box_rows};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = enc(&c.map, elem == 2 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_UINT8, 2,
                     const_cast<void*>(base), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) {
        c.valid = false;
        return fail(FA_ERR_CUDA, "cuTensorMapEncodeTiled (cache view, depth %d, rows %lld) failed: %d", depth,
                    (long long)rows, (int)r);
    }
    c.valid = true;
    c.ptr = base;
    c.key0 = depth;
    c.key1 = rows;
    c.key2 = k2;
    return FA_OK;
}

// Tensor map over the output: 3-D {Dv, Hq, B*T} bf16, box {chunk, heads, tokens}.
int encode_out_map(MapCache& c, void* out, int dv, int hq, int64_t bt, int chunk, int heads, int tokens)
{
    uint64_t k1 = ((uint64_t)hq << 32) | (uint64_t)dv;
    uint64_t k2 = ((uint64_t)chunk << 40) | ((uint64_t)heads << 20) | (uint64_t)tokens;
    if (c.valid && c.ptr == out && c.key0 == (uint64_t)bt && c.key1 == k1 && c.key2 == k2) return FA_OK;
    EncodeTiledFn enc = encode_tiled_fn();
    if (!enc) return fail(FA_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
    cuuint64_t dims[3] = {(cuuint64_t)dv, (cuuint64_t)hq, (cuuint64_t)bt};
    cuuint64_t strides[2] = {(cuuint64_t)dv * 2, (cuuint64_t)hq * dv * 2};
    cuuint32_t box[3] = {(cuuint32_t)chunk, (cuuint32_t)heads, (cuuint32_t)tokens};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = enc(&c.map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, out, dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_NONE,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) {
        c.valid = false;
        return fail(FA_ERR_CUDA, "cuTensorMapEncodeTiled (output view) failed: %d", (int)r);
    }
    c.valid = true;
    c.ptr = out;
    c.key0 = bt;
    c.key1 = k1;
    c.key2 = k2;
    return FA_OK;
}

}  // namespace

struct fa_decode {
    int hq, hkv, group, dk, nope, dv, page_size, num_q, splitk;
    int kv_format;                   // FA_KV_BF16 or FA_KV_E4M3
    int rope_depth;                  // E4M3: trailing key columns kept in bf16 apart (0)
    int rows, row_blocks, heads_per_cta, tokens_per_cta, rows_capacity;
    int device;
    fad::KernelGeometry geo;         // SIMT kernel, separate V cache (or V = K rows)
    fad::KernelGeometry geo_latent;  // SIMT kernel, V = prefix of the K row
    fad::KernelGeometry geo_tc;      // tcgen05 kernel, 3-slot ring (two CTAs per SM)
    fad::KernelGeometry geo_tc_big;  // tcgen05 kernel, 6-slot ring (one CTA per SM, several units per cluster)
    fad::KernelGeometry geo_tc_sk;   // the same under the stream-K partition
    fad::KernelGeometry geo_mla;     // tcgen05 kernel of the MLA latent layout (64 heads per CTA)
    fad::KernelGeometry geo_latent8; // SIMT kernel, E4M3 latent cache with a bf16 rope cache
    bool has_simt, has_latent, has_tc, has_mla, has_latent8;
    int sm_count;
    int tc_big_clusters;             // clusters of geo_tc_big (fixed split) resident at once
    unsigned int* d_status;
    // Stream-K chunk scratch of geo_tc_big (fixed split): two slots per
    // resident cluster; null for plans made without a handle.
    void* d_chunk;
    size_t chunk_count_bytes;
    float* chunk_o;
    float2* chunk_ms;
    unsigned int* chunk_count;
    int64_t chunk_items;             // slots the scratch holds
    uint32_t debug_flags;
    uint64_t wait_limit_ns;
    uint64_t* trace;
    int64_t trace_words;
    MapCache k_map, v_map, rope_map, out_map[3];
    // Per-sequence split: the launches of the 2- and 4-CTA clusters run on two
    // side streams forked from the caller's stream (their sequences are
    // disjoint), so no launch waits for another's last wave. Owned by the
    // handle; absent (null) for plans made without a handle.
    cudaStream_t side[2];
    cudaEvent_t fork, join[2];
};

namespace {

int split_list(const fa_decode* h, int* list)
{
    if (h->splitk > 0) {
        list[0] = h->splitk;
        return 1;
    }
    list[0] = 1;
    list[1] = 2;
    list[2] = 4;
    return 3;
}

// Results of the per-kernel attribute calls and occupancy queries. They depend
// only on (device, kernel, cluster size), so each is made once per process and
// kept here: planning a call (fa_decode_run_noalloc plans every call) then
// costs no driver round trip. cluster_size 0 marks "attributes set".
struct PrepEntry {
    int dev;
    const void* func;
    int cluster_size;
    int clusters;
};
std::mutex g_prep_mutex;
std::vector<PrepEntry> g_prep;

bool prep_lookup(int dev, const void* func, int P, int* clusters)
{
    for (const PrepEntry& e : g_prep)
        if (e.dev == dev && e.func == func && e.cluster_size == P) {
            if (clusters) *clusters = e.clusters;
            return true;
        }
    return false;
}

// Clusters of P CTAs of kernel g (P == 1: single CTAs) that the device holds
// at once. Caller holds g_prep_mutex.
int query_clusters(int dev, int sm_count, const fad::KernelGeometry& g, int P, int* out)
{
    if (prep_lookup(dev, g.func, P, out)) return FA_OK;
    cudaError_t e;
    int n = 0;
    if (P <= 1) {
        int per_sm = 0;
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, g.func, g.threads, g.smem_bytes);
        if (e != cudaSuccess) return cuda_fail(e, "cudaOccupancyMaxActiveBlocksPerMultiprocessor");
        n = per_sm * sm_count;
    } else {
        cudaLaunchConfig_t cfg = {};
        cudaLaunchAttribute attr[1];
        cfg.gridDim = dim3(P, 1, 1);
        cfg.blockDim = dim3(g.threads, 1, 1);
        cfg.dynamicSmemBytes = g.smem_bytes;
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = P;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        e = cudaOccupancyMaxActiveClusters(&n, g.func, &cfg);
        if (e != cudaSuccess) return cuda_fail(e, "cudaOccupancyMaxActiveClusters");
    }
    if (n < 1)
        return fail(FA_ERR_UNSUPPORTED, "kernel %s: a cluster of %d CTAs with %d bytes of shared memory each "
                                        "cannot be scheduled on this device", g.name, P, g.smem_bytes);
    g_prep.push_back(PrepEntry{dev, g.func, P, n});
    *out = n;
    return FA_OK;
}

int prepare_kernel(const fa_decode* h, const fad::KernelGeometry& g)
{
    std::lock_guard<std::mutex> lock(g_prep_mutex);
    if (!prep_lookup(h->device, g.func, 0, nullptr)) {
        cudaError_t e = cudaFuncSetAttribute(g.func, cudaFuncAttributeMaxDynamicSharedMemorySize, g.smem_bytes);
        if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute(max dynamic shared memory)");
        // Clusters of 16 are beyond the portable size of 8.
        e = cudaFuncSetAttribute(g.func, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
        if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute(non-portable cluster size)");
        g_prep.push_back(PrepEntry{h->device, g.func, 0, 0});
    }
    int splits[3];
    int n = split_list(h, splits);
    for (int i = 0; i < n; ++i) {
        if (splits[i] <= 1) continue;
        int clusters = 0;
        int rc = query_clusters(h->device, h->sm_count, g, splits[i], &clusters);
        if (rc) return rc;
    }
    return FA_OK;
}

// Clusters of P CTAs of kernel g that the device holds at once.
int resident_clusters(const fa_decode* h, const fad::KernelGeometry& g, int P, int* out)
{
    std::lock_guard<std::mutex> lock(g_prep_mutex);
    return query_clusters(h->device, h->sm_count, g, P, out);
}

}  // namespace

static void release_side_streams(fa_decode& h)
{
    for (int i = 0; i < 2; ++i) {
        if (h.side[i]) cudaStreamDestroy(h.side[i]);
        if (h.join[i]) cudaEventDestroy(h.join[i]);
        h.side[i] = nullptr;
        h.join[i] = nullptr;
    }
    if (h.fork) cudaEventDestroy(h.fork);
    h.fork = nullptr;
}

// Validation, kernel choice and per-kernel attributes of a plan (the
// FA4Config constructor and supported() checks). Allocates nothing; the
// caller provides the status word.
static int plan_decode(fa_decode& tmp, int num_q_heads, int num_kv_heads, int qk_depth, int nope_depth, int ov_depth,
                       int page_size, int num_q, int splitk, int kv_format = FA_KV_BF16, int rope_depth = 0)
{
    if (kv_format != FA_KV_BF16 && kv_format != FA_KV_E4M3)
        return fail(FA_ERR_INVALID_ARG, "kv_format must be FA_KV_BF16 or FA_KV_E4M3 (got %d)", kv_format);
    if (rope_depth < 0 || rope_depth >= qk_depth || (kv_format == FA_KV_BF16 && rope_depth != 0))
        return fail(FA_ERR_INVALID_ARG, "rope_depth must be 0 for a bf16 cache and in [0, qk_depth) for E4M3 "
                                        "(got %d)", rope_depth);
    if (num_q_heads < 1 || num_kv_heads < 1)
        return fail(FA_ERR_INVALID_ARG, "head counts must be >= 1 (got %d q, %d kv)", num_q_heads, num_kv_heads);
    if (num_q_heads % num_kv_heads)
        return fail(FA_ERR_INVALID_ARG, "num_q_heads %d is not a multiple of num_kv_heads %d", num_q_heads,
                    num_kv_heads);
    if (qk_depth < 1 || ov_depth < 1) return fail(FA_ERR_INVALID_ARG, "depths must be >= 1");
    if (!(nope_depth == -1 || (nope_depth >= 1 && nope_depth <= qk_depth)))
        return fail(FA_ERR_INVALID_ARG, "nope_depth must be -1 or in [1, qk_depth] (got %d)", nope_depth);
    if (page_size < 1) return fail(FA_ERR_INVALID_ARG, "page_size must be >= 1");
    if (num_q < 1) return fail(FA_ERR_INVALID_ARG, "num_q must be >= 1");
    if (!(splitk == 0 || splitk == 1 || splitk == 2 || splitk == 4 || splitk == 8 || splitk == 16))
        return fail(FA_ERR_INVALID_ARG, "splitk must be 0 (per sequence), 1, 2, 4, 8 or 16 (got %d)", splitk);

    tmp = fa_decode{};
    tmp.hq = num_q_heads;
    tmp.hkv = num_kv_heads;
    tmp.group = num_q_heads / num_kv_heads;
    tmp.dk = qk_depth;
    tmp.nope = nope_depth < 0 ? qk_depth : nope_depth;
    tmp.dv = ov_depth;
    tmp.page_size = page_size;
    tmp.num_q = num_q;
    tmp.splitk = splitk;
    tmp.kv_format = kv_format;
    tmp.rope_depth = rope_depth;
    tmp.wait_limit_ns = fad::kDefaultWaitLimitNs;

    // Rows of one CTA: the T*g fused GQA rows, or 16-head blocks for wide groups.
    const int R = num_q * tmp.group;
    if (R <= 16) {
        tmp.rows = R;
        tmp.rows_capacity = R <= 4 ? 4 : (R <= 8 ? 8 : 16);
        tmp.row_blocks = 1;
        tmp.heads_per_cta = tmp.group;
        tmp.tokens_per_cta = num_q;
    } else if (num_q == 1 && tmp.group % 16 == 0) {
        tmp.rows = 16;
        tmp.rows_capacity = 16;
        tmp.row_blocks = tmp.group / 16;
        tmp.heads_per_cta = 16;
        tmp.tokens_per_cta = 1;
    } else {
        return fail(FA_ERR_UNSUPPORTED, "num_q * group = %d rows per kv head: built for <= 16, or num_q == 1 "
                                        "with group a multiple of 16", R);
    }
    if (page_size % 8)
        return fail(FA_ERR_UNSUPPORTED, "page_size %d is not a multiple of 8", page_size);
    auto page_fits = [&](int bn) { return page_size % bn == 0 || bn % page_size == 0; };
    if (kv_format == FA_KV_E4M3) {
        // The E4M3 cache: the tcgen05 GQA kernel (head dim 128, <= 16 rows per
        // CTA, separate V); for the MLA latent layout with a bf16 rope cache the
        // tcgen05 MLA kernel (64 heads per CTA) and the SIMT kernel (16).
        const auto geo = fad::tc_fp8_geometry;
        tmp.has_tc = tmp.row_blocks == 1 && rope_depth == 0 &&
                     geo(qk_depth, ov_depth, tmp.rows, fad::kTcSlotsShared, false, &tmp.geo_tc) &&
                     geo(qk_depth, ov_depth, tmp.rows, fad::kTcSlotsAlone, false, &tmp.geo_tc_big) &&
                     geo(qk_depth, ov_depth, tmp.rows, fad::kTcSlotsAlone, true, &tmp.geo_tc_sk) &&
                     page_fits(tmp.geo_tc.keys_per_tile);
        tmp.has_latent8 = fad::simt_fp8_latent_geometry(qk_depth, ov_depth, rope_depth, tmp.rows_capacity,
                                                        &tmp.geo_latent8) &&
                          page_fits(tmp.geo_latent8.keys_per_tile);
        tmp.has_mla = fad::mla_tc_fp8_geometry(qk_depth, ov_depth, tmp.nope, rope_depth, tmp.group, num_q,
                                               &tmp.geo_mla) &&
                      page_fits(tmp.geo_mla.keys_per_tile);
        if (!tmp.has_tc && !tmp.has_latent8 && !tmp.has_mla)
            return fail(FA_ERR_UNSUPPORTED, "no E4M3-cache kernel for (qk %d, ov %d, rope %d), %d rows per CTA and "
                                            "page_size %d (built: qk = ov = 128, rope 0, <= 16 rows per CTA; "
                                            "latent qk 576 = 512 + rope 64, ov 512, 16 rows per CTA)",
                        qk_depth, ov_depth, rope_depth, tmp.rows, page_size);
    } else {
        tmp.has_simt = fad::simt_geometry(qk_depth, ov_depth, false, tmp.rows_capacity, &tmp.geo) &&
                       page_fits(tmp.geo.keys_per_tile);
        tmp.has_latent = tmp.has_simt && fad::simt_geometry(qk_depth, ov_depth, true, tmp.rows_capacity,
                                                            &tmp.geo_latent);
        tmp.has_tc = tmp.row_blocks == 1 &&
                     fad::tc_geometry(qk_depth, ov_depth, tmp.rows, fad::kTcSlotsShared, false, &tmp.geo_tc) &&
                     fad::tc_geometry(qk_depth, ov_depth, tmp.rows, fad::kTcSlotsAlone, false, &tmp.geo_tc_big) &&
                     fad::tc_geometry(qk_depth, ov_depth, tmp.rows, fad::kTcSlotsAlone, true, &tmp.geo_tc_sk) &&
                     page_fits(tmp.geo_tc.keys_per_tile);
        tmp.has_mla = fad::mla_tc_geometry(qk_depth, ov_depth, tmp.nope, tmp.group, num_q, &tmp.geo_mla) &&
                      page_fits(tmp.geo_mla.keys_per_tile);
        if (!tmp.has_simt && !tmp.has_tc && !tmp.has_mla)
            return fail(FA_ERR_UNSUPPORTED, "no kernel for (qk %d, ov %d), %d rows per CTA and page_size %d "
                                            "(built: 64/64, 128/128, 576/512; page size and key tile must divide "
                                            "one another)", qk_depth, ov_depth, tmp.rows, page_size);
    }
    int splits[3];
    const int ns = split_list(&tmp, splits);
    for (int i = 0; i < ns; ++i) {
        const int bw = ov_depth / splits[i];
        if (ov_depth % splits[i] || bw % 8)
            return fail(FA_ERR_UNSUPPORTED, "ov_depth %d split %d ways gives bands that are not a multiple of 8 "
                                            "columns", ov_depth, splits[i]);
    }

    // Device: GB300 only (compute capability 10.3).
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    int major = 0, minor = 0;
    cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
    cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
    if (major != 10 || minor != 3)
        return fail(FA_ERR_UNSUPPORTED, "device %d has compute capability %d.%d; this library is built for "
                                        "sm_103a (GB300)", dev, major, minor);
    tmp.device = dev;
    cudaDeviceGetAttribute(&tmp.sm_count, cudaDevAttrMultiProcessorCount, dev);
    int rc = FA_OK;
    if (tmp.has_simt && (rc = prepare_kernel(&tmp, tmp.geo))) return rc;
    if (tmp.has_latent && (rc = prepare_kernel(&tmp, tmp.geo_latent))) return rc;
    if (tmp.has_tc && (rc = prepare_kernel(&tmp, tmp.geo_tc))) return rc;
    if (tmp.has_tc && (rc = prepare_kernel(&tmp, tmp.geo_tc_big))) return rc;
    if (tmp.has_tc && splitk > 0 && (rc = prepare_kernel(&tmp, tmp.geo_tc_sk))) return rc;
    if (tmp.has_mla && (rc = prepare_kernel(&tmp, tmp.geo_mla))) return rc;
    if (tmp.has_latent8 && (rc = prepare_kernel(&tmp, tmp.geo_latent8))) return rc;
    if (tmp.has_tc && splitk > 0 && (rc = resident_clusters(&tmp, tmp.geo_tc_big, splitk, &tmp.tc_big_clusters)))
        return rc;
    return FA_OK;
}

// Device memory for callers that cannot allocate (fa_decode_run_noalloc):
// status words in a file-scope device array, so no call ever needs
// cudaMalloc. Every GPU that loads this library holds the array until the
// process exits. On the host the name g_noalloc_status only stands for the
// symbol: its device address comes from cudaGetSymbolAddress, taken once per
// device with that device current.
static __device__ __align__(256) unsigned int g_noalloc_status[FA_NOALLOC_STATUS_SLOTS];

namespace {
constexpr int kMaxDevices = 64;
std::mutex g_noalloc_mutex;
unsigned int* g_noalloc_addr[kMaxDevices] = {};

int noalloc_status_base(int dev, unsigned int** out)
{
    if (dev < 0 || dev >= kMaxDevices) return fail(FA_ERR_UNSUPPORTED, "device ordinal %d beyond %d", dev, kMaxDevices);
    std::lock_guard<std::mutex> lock(g_noalloc_mutex);
    if (!g_noalloc_addr[dev]) {
        void* ptr = nullptr;
        cudaError_t e = cudaGetSymbolAddress(&ptr, g_noalloc_status);
        if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(static status array)");
        g_noalloc_addr[dev] = static_cast<unsigned int*>(ptr);
    }
    *out = g_noalloc_addr[dev];
    return FA_OK;
}
}  // namespace

extern "C" {

const char* fa_decode_last_error(void) { return g_last_error.c_str(); }

int fa_decode_create(fa_decode_t* out, int num_q_heads, int num_kv_heads, int qk_depth, int nope_depth,
                     int ov_depth, int page_size, int num_q, int splitk)
{
    return fa_decode_create_kv(out, num_q_heads, num_kv_heads, qk_depth, nope_depth, ov_depth, page_size, num_q,
                               splitk, FA_KV_BF16, 0);
}

int fa_decode_create_kv(fa_decode_t* out, int num_q_heads, int num_kv_heads, int qk_depth, int nope_depth,
                        int ov_depth, int page_size, int num_q, int splitk, int kv_format, int rope_depth)
{
    g_last_error.clear();
    if (!out) return fail(FA_ERR_INVALID_ARG, "out handle pointer is NULL");
    *out = nullptr;
    fa_decode tmp;
    int rc = plan_decode(tmp, num_q_heads, num_kv_heads, qk_depth, nope_depth, ov_depth, page_size, num_q, splitk,
                         kv_format, rope_depth);
    if (rc) return rc;

    cudaError_t e = cudaMalloc(&tmp.d_status, 256);
    if (e != cudaSuccess) return cuda_fail(e, "cudaMalloc(status word)");
    e = cudaMemset(tmp.d_status, 0, 256);
    if (e != cudaSuccess) {
        cudaFree(tmp.d_status);
        return cuda_fail(e, "cudaMemset(status word)");
    }
    if (splitk == 0) {
        bool made = cudaStreamCreateWithFlags(&tmp.side[0], cudaStreamNonBlocking) == cudaSuccess &&
                    cudaStreamCreateWithFlags(&tmp.side[1], cudaStreamNonBlocking) == cudaSuccess &&
                    cudaEventCreateWithFlags(&tmp.fork, cudaEventDisableTiming) == cudaSuccess &&
                    cudaEventCreateWithFlags(&tmp.join[0], cudaEventDisableTiming) == cudaSuccess &&
                    cudaEventCreateWithFlags(&tmp.join[1], cudaEventDisableTiming) == cudaSuccess;
        if (!made) {
            release_side_streams(tmp);
            cudaFree(tmp.d_status);
            return fail(FA_ERR_CUDA, "creating the side streams of the per-sequence split");
        }
    }
    if (tmp.has_tc && splitk > 0 && tmp.tc_big_clusters > 0) {
        // Stream-K scratch: per slot and rank, the band's fp32 rows and
        // per-row (max, sum), and one count per (slot, rank) for the shared
        // units, zero between launches.
        const size_t items = (size_t)tmp.tc_big_clusters * 2;
        const size_t rb = (size_t)tmp.geo_tc_big.rows_capacity;
        tmp.chunk_items = (int64_t)items;
        tmp.chunk_count_bytes = (items * splitk * sizeof(unsigned int) + 255) / 256 * 256;
        const size_t ms_bytes = (items * splitk * rb * sizeof(float2) + 255) / 256 * 256;
        const size_t o_bytes = items * rb * (size_t)ov_depth * sizeof(float);
        e = cudaMalloc(&tmp.d_chunk, tmp.chunk_count_bytes + ms_bytes + o_bytes);
        if (e == cudaSuccess) e = cudaMemset(tmp.d_chunk, 0, tmp.chunk_count_bytes);
        if (e != cudaSuccess) {
            if (tmp.d_chunk) cudaFree(tmp.d_chunk);
            release_side_streams(tmp);
            cudaFree(tmp.d_status);
            return cuda_fail(e, "allocating the key-range chunk scratch");
        }
        uint8_t* base = static_cast<uint8_t*>(tmp.d_chunk);
        tmp.chunk_count = reinterpret_cast<unsigned int*>(base);
        tmp.chunk_ms = reinterpret_cast<float2*>(base + tmp.chunk_count_bytes);
        tmp.chunk_o = reinterpret_cast<float*>(base + tmp.chunk_count_bytes + ms_bytes);
    }
    fa_decode* h = new (std::nothrow) fa_decode(tmp);
    if (!h) {
        release_side_streams(tmp);
        if (tmp.d_chunk) cudaFree(tmp.d_chunk);
        cudaFree(tmp.d_status);
        return fail(FA_ERR_CUDA, "out of host memory");
    }
    *out = h;
    return FA_OK;
}

int fa_decode_destroy(fa_decode_t h)
{
    if (!h) return FA_OK;
    release_side_streams(*h);
    if (h->d_chunk) cudaFree(h->d_chunk);
    cudaError_t e = cudaFree(h->d_status);
    delete h;
    if (e != cudaSuccess) return cuda_fail(e, "cudaFree(status word)");
    return FA_OK;
}

int fa_decode_set_debug(fa_decode_t h, uint32_t flags, int64_t wait_limit_ns)
{
    if (!h) return fail(FA_ERR_INVALID_ARG, "handle is NULL");
    if (wait_limit_ns < 0) return fail(FA_ERR_INVALID_ARG, "wait_limit_ns must be >= 0");
    h->debug_flags = flags;
    h->wait_limit_ns = wait_limit_ns ? (uint64_t)wait_limit_ns : fad::kDefaultWaitLimitNs;
    return FA_OK;
}

int fa_decode_set_trace(fa_decode_t h, uint64_t* buf, int64_t n_words)
{
    if (!h) return fail(FA_ERR_INVALID_ARG, "handle is NULL");
    if (buf && (n_words < 0 || !is_aligned(buf, 8)))
        return fail(FA_ERR_INVALID_ARG, "trace buffer must be 8-byte aligned with n_words >= 0");
    h->trace = buf;
    h->trace_words = buf ? n_words : 0;
    return FA_OK;
}

int fa_decode_check(fa_decode_t h, void* stream, uint32_t* status_out)
{
    if (!h) return fail(FA_ERR_INVALID_ARG, "handle is NULL");
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
    unsigned int st = 0;
    e = cudaMemcpy(&st, h->d_status, sizeof st, cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return cuda_fail(e, "reading the status word");
    e = cudaMemset(h->d_status, 0, sizeof st);
    if (e != cudaSuccess) return cuda_fail(e, "clearing the status word");
    if (st && h->chunk_count) {
        // A launch that gave up may have left chunk counts behind.
        e = cudaMemset(h->chunk_count, 0, h->chunk_count_bytes);
        if (e != cudaSuccess) return cuda_fail(e, "clearing the chunk counts");
    }
    if (status_out) *status_out = st;
    if (st) {
        return fail(FA_ERR_DEVICE, "device status 0x%x:%s%s", st, (st & FA_STATUS_TIMEOUT) ? " wait timed out" : "",
                    (st & FA_STATUS_BAD_PAGE) ? " page id or length out of range" : "");
    }
    return FA_OK;
}

int fa_decode_describe(fa_decode_t h, char* buf, int size)
{
    if (!h || !buf || size < 1) return fail(FA_ERR_INVALID_ARG, "handle or buffer is NULL");
    // The kernel a run takes by default: the MLA tcgen05 kernel for the latent
    // layout where it applies, the deep-ring tcgen05 kernel for a fixed split,
    // the shallow-ring one for the per-sequence split, else the SIMT kernel.
    const bool tc = h->has_mla || h->has_tc;
    const fad::KernelGeometry& g =
        h->has_mla ? h->geo_mla
                   : (h->has_tc ? (h->splitk > 0 ? h->geo_tc_big : h->geo_tc)
                                : (h->has_latent8 ? h->geo_latent8 : h->geo));
    const int rows = h->has_mla ? 64 : h->rows, row_blocks = h->has_mla ? h->group / 64 : h->row_blocks;
    const char* per_seq = h->splitk != 0 ? "" : (h->has_tc && !h->has_mla ? "(per sequence: 1/2/4, one launch)"
                                                                         : "(per sequence: 1/2/4)");
    snprintf(buf, (size_t)size,
             "path=%s kernel=%s simt_kernel=%s latent_kernel=%s splitk=%d%s threads=%d keys_per_tile=%d "
             "stages=%d rows=%d rows_capacity=%d row_blocks=%d smem=%d resident_clusters=%d",
             tc ? "tcgen05" : "simt", g.name, h->has_simt ? h->geo.name : "none",
             h->has_latent ? h->geo_latent.name : (h->has_latent8 ? h->geo_latent8.name : "none"), h->splitk, per_seq,
             g.threads, g.keys_per_tile, g.stages, rows, h->has_mla ? 64 : h->rows_capacity, row_blocks, g.smem_bytes,
             h->tc_big_clusters);
    return FA_OK;
}

int fa_decode_run(fa_decode_t h, const void* q, const void* k_pages, const void* v_pages,
                  const int32_t* page_table, const int32_t* seq_lens, float scale, void* out, float* lse,
                  void* stream, int batch, int max_pages_per_seq, int num_pages)
{
    if (h && h->kv_format != FA_KV_BF16)
        return fail(FA_ERR_INVALID_ARG, "this handle reads an E4M3 cache: call fa_decode_run_kv");
    return fa_decode_run_kv(h, q, k_pages, v_pages, nullptr, nullptr, page_table, seq_lens, scale, out, lse, stream,
                            batch, max_pages_per_seq, num_pages);
}

int fa_decode_run_kv(fa_decode_t h, const void* q, const void* k_pages, const void* v_pages, const void* k_rope_pages,
                     const float* k_scale, const int32_t* page_table, const int32_t* seq_lens, float scale,
                     void* out, float* lse, void* stream, int batch, int max_pages_per_seq, int num_pages)
{
    if (!h) return fail(FA_ERR_INVALID_ARG, "handle is NULL");
    const bool e4m3 = h->kv_format == FA_KV_E4M3;
    if (!e4m3 && (k_rope_pages || k_scale))
        return fail(FA_ERR_INVALID_ARG, "k_rope_pages and k_scale apply to an E4M3 cache only");
    if (e4m3 && (k_rope_pages != nullptr) != (h->rope_depth > 0))
        return fail(FA_ERR_INVALID_ARG, "k_rope_pages must be given exactly when rope_depth > 0 (rope_depth %d)",
                    h->rope_depth);
    if (k_scale && !is_aligned(k_scale, 16)) return fail(FA_ERR_INVALID_ARG, "k_scale must be 16-byte aligned");
    if (k_rope_pages && !is_aligned(k_rope_pages, 16))
        return fail(FA_ERR_INVALID_ARG, "k_rope_pages must be 16-byte aligned");
    if (batch < 0) return fail(FA_ERR_INVALID_ARG, "batch must be >= 0 (got %d)", batch);
    if (batch == 0) return FA_OK;
    if (!q || !k_pages || !page_table || !seq_lens || !out)
        return fail(FA_ERR_INVALID_ARG, "q, k_pages, page_table, seq_lens and out must not be NULL");
    if (!is_aligned(q, 16) || !is_aligned(k_pages, 16) || !is_aligned(out, 16) ||
        (v_pages && !is_aligned(v_pages, 16)))
        return fail(FA_ERR_INVALID_ARG, "q, k_pages, v_pages and out must be 16-byte aligned");
    if (!is_aligned(page_table, 4) || !is_aligned(seq_lens, 4) || (lse && !is_aligned(lse, 4)))
        return fail(FA_ERR_INVALID_ARG, "page_table, seq_lens and lse must be 4-byte aligned");
    if (max_pages_per_seq < 1 || num_pages < 1)
        return fail(FA_ERR_INVALID_ARG, "max_pages_per_seq and num_pages must be >= 1");
    if (!(scale >= 0.f) || scale == INFINITY) return fail(FA_ERR_INVALID_ARG, "scale must be finite and >= 0");
    if (batch > 65535) return fail(FA_ERR_UNSUPPORTED, "batch %d exceeds 65535 sequences per call", batch);
    const int64_t cache_rows = (int64_t)num_pages * h->hkv * h->page_size;
    if (cache_rows + 256 > INT32_MAX)
        return fail(FA_ERR_UNSUPPORTED, "cache of %lld rows exceeds the 2^31 TMA row coordinate range",
                    (long long)cache_rows);

    const bool latent = (v_pages == nullptr || v_pages == k_pages);
    if (e4m3 && latent && !h->has_latent8 && !h->has_mla)
        return fail(FA_ERR_UNSUPPORTED, "the E4M3 latent layout is built for qk 576 = 512 + rope 64, ov 512");
    if (e4m3 && !latent && !h->has_tc)
        return fail(FA_ERR_UNSUPPORTED, "this E4M3 handle reads the latent layout only (v_pages NULL)");
    if (latent && h->dv > h->dk)
        return fail(FA_ERR_INVALID_ARG, "latent layout (v_pages NULL or == k_pages) needs ov_depth <= qk_depth");
    // Kernel choice: for the MLA latent cache the MLA tcgen05 kernel (64 heads
    // per CTA) where it applies, else the latent-layout SIMT kernel; otherwise
    // the tcgen05 kernel where it applies, else the SIMT kernel.
    const bool force_simt = (h->debug_flags & FA_DEBUG_FORCE_SIMT) != 0;
    const bool use_mla = latent && h->has_mla && !(force_simt && (e4m3 ? h->has_latent8 : h->has_latent));
    const bool use_latent = latent && !use_mla && (e4m3 ? h->has_latent8 : h->has_latent);
    const bool use_tc = !use_mla && !use_latent && h->has_tc && !(force_simt && h->has_simt);
    if (!use_mla && !use_latent && !use_tc && !h->has_simt)
        return fail(FA_ERR_UNSUPPORTED, "no kernel for this call (latent layout %d)", (int)latent);
    // A fixed split takes the deep ring (one CTA per SM); when there are more
    // (sequence, kv head) units than clusters fit on the device at once, the
    // resident clusters work through the units in turn. The per-sequence
    // split (three launches) shares SMs two by two with the shallow ring.
    const bool tc_big = use_tc && h->splitk > 0;
    const int64_t units = (int64_t)h->hkv * batch;
    int64_t clusters = units;
    // Stream-K partition (see DecodeParams::sk_tiles): 0 = off.
    int sk_tiles = 0, sk_clusters = 0;
    int64_t sk_total = 0;
    if (tc_big) {
        const int64_t most = (h->debug_flags & FA_DEBUG_TWO_CLUSTERS) ? 2 : h->tc_big_clusters;
        if (h->chunk_count && !(h->debug_flags & FA_DEBUG_NO_STREAM_K)) {
            // Every cluster of the partition takes an equal share of all units'
            // tiles (a full page-table row each): with fewer units than resident
            // clusters, or with more when whole-unit rounds would leave some
            // clusters idle at the end.
            const int64_t nv = ((int64_t)max_pages_per_seq * h->page_size + 127) / 128;
            const int G = fad::sk_choose_clusters(units, nv, h->splitk, most, h->chunk_items);
            if (G > 0) {
                sk_tiles = (int)nv;
                sk_clusters = G;
                sk_total = units * nv;
                clusters = G;
            }
        }
        if (clusters > most) {
            // As many rounds as the resident clusters need, spread evenly: the
            // fewest clusters that still finish in that many rounds.
            const int64_t rounds = (units + most - 1) / most;
            clusters = (units + rounds - 1) / rounds;
        }
    }
    const fad::KernelGeometry& g = use_mla ? h->geo_mla
                                   : use_latent ? (e4m3 ? h->geo_latent8 : h->geo_latent)
                                                : (use_tc ? (tc_big ? (sk_tiles > 0 ? h->geo_tc_sk : h->geo_tc_big)
                                                                    : h->geo_tc)
                                                          : h->geo);
    // Heads per CTA: 64 for the MLA kernel, else the plan's rows.
    const int row_blocks = use_mla ? h->group / 64 : h->row_blocks;
    const int heads_per_cta = use_mla ? 64 : h->heads_per_cta;
    const int bn = g.keys_per_tile;
    const int box_rows = h->page_size < bn ? h->page_size : bn;

    const int elem = e4m3 ? 1 : 2;
    // An E4M3 key row holds the codes only; its rope columns come from their own cache.
    int rc = encode_cache_map(h->k_map, k_pages, h->dk - (e4m3 ? h->rope_depth : 0), cache_rows, box_rows, elem);
    if (rc) return rc;
    if (e4m3 && h->rope_depth > 0 &&
        (rc = encode_cache_map(h->rope_map, k_rope_pages, h->rope_depth, cache_rows, box_rows)))
        return rc;
    if (latent && !use_latent && !use_mla) {
        // V = K row prefix through a separate-V kernel (e.g. qk == ov): same rows, V width.
        rc = encode_cache_map(h->v_map, k_pages, h->dk, cache_rows, box_rows);
    } else if (!latent) {
        rc = encode_cache_map(h->v_map, v_pages, h->dv, cache_rows, box_rows, elem);
    }
    if (rc) return rc;

    fad::DecodeParams p;
    std::memset(&p, 0, sizeof p);
    p.tm_k = h->k_map.map;
    if (!use_latent && !use_mla) p.tm_v = h->v_map.map;
    if (e4m3 && h->rope_depth > 0) p.tm_rope = h->rope_map.map;
    p.q = static_cast<const uint16_t*>(q);
    p.page_table = page_table;
    p.seq_lens = seq_lens;
    p.lse = lse;
    p.status = h->d_status;
    p.batch = batch;
    p.num_q = h->num_q;
    p.num_q_heads = h->hq;
    p.num_kv_heads = h->hkv;
    p.group = h->group;
    p.qk_depth = h->dk;
    p.ov_depth = h->dv;
    p.page_size = h->page_size;
    p.max_pages = max_pages_per_seq;
    p.num_pages = num_pages;
    p.rows = use_mla ? heads_per_cta : h->rows;
    p.row_blocks = row_blocks;
    p.heads_per_cta = heads_per_cta;
    p.tokens_per_cta = h->tokens_per_cta;
    p.box_rows = box_rows;
    p.oob_row = (int32_t)cache_rows;
    p.scale = scale;
    p.scale_log2e = (float)((double)scale * 1.4426950408889634);
    p.debug_flags = h->debug_flags;
    p.wait_limit_ns = h->wait_limit_ns;
    p.auto_split = h->splitk == 0 ? 1 : 0;
    p.trace = reinterpret_cast<unsigned long long*>(h->trace);
    p.trace_ctas = h->trace_words / FA_TRACE_WORDS_PER_CTA;
    p.sk_tiles = sk_tiles;
    p.sk_clusters = sk_clusters;
    p.sk_total = sk_total;
    p.chunk_o = h->chunk_o;
    p.chunk_ms = h->chunk_ms;
    p.chunk_count = h->chunk_count;
    p.k_scale = k_scale;

    int splits[3];
    int ns = split_list(h, splits);
    // The per-sequence split on the tcgen05 shallow ring runs as one launch of
    // 4-CTA clusters, each serving one unit of split 4, two of split 2 or four
    // of split 1 (chosen on the device from the lengths; see dyn_group); the
    // other kernels launch once per cluster size.
    const bool dyn = h->splitk == 0 && use_tc && batch <= kDynSplitMaxBatch;
    if (dyn) {
        splits[0] = 4;
        ns = 1;
        p.auto_split = 0;
        p.dyn_split = 1;
    }
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    // Fork: launches after the first go to the side streams, which first wait
    // for everything queued on the caller's stream.
    const bool forked = ns > 1 && h->side[0] && h->side[1];
    if (forked) {
        cudaError_t e = cudaEventRecord(h->fork, s);
        for (int i = 0; e == cudaSuccess && i < 2; ++i) e = cudaStreamWaitEvent(h->side[i], h->fork, 0);
        if (e != cudaSuccess) return cuda_fail(e, "forking the per-sequence split launches");
    }
    for (int i = 0; i < ns; ++i) {
        const int P = splits[i];
        p.splitk = P;
        p.band_cols = h->dv / P;
        p.out_chunk_cols = p.band_cols < 256 ? p.band_cols : 256;
        if (dyn) p.out_chunk_cols = h->dv / 4;  // stores in boxes of the narrowest band (split 4)
        rc = encode_out_map(h->out_map[i], out, h->dv, h->hq, (int64_t)batch * h->num_q, p.out_chunk_cols,
                            heads_per_cta, h->tokens_per_cta);
        if (rc) return rc;
        p.tm_out = h->out_map[i].map;

        cudaLaunchConfig_t cfg = {};
        cudaLaunchAttribute attr[2];
        // Cluster c (= blockIdx.y + gridDim.y * blockIdx.z) takes units
        // c, c + G, ... of u = b * Hkv + kvh (with G = units that is one unit
        // each), or the units its stream-K range touches.
        cfg.gridDim = clusters == units ? dim3(P, h->hkv * row_blocks, batch) : dim3(P, (unsigned)clusters, 1);
        cfg.blockDim = dim3(g.threads, 1, 1);
        cfg.dynamicSmemBytes = g.smem_bytes;
        cfg.stream = forked && i > 0 ? h->side[i - 1] : s;
        // Programmatic dependent launch: the kernel may be scheduled while the
        // previous kernel in the stream finishes; it waits for that kernel's
        // completion (griddepcontrol.wait) before reading any input.
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        if (P > 1) {
            attr[1].id = cudaLaunchAttributeClusterDimension;
            attr[1].val.clusterDim.x = P;
            attr[1].val.clusterDim.y = 1;
            attr[1].val.clusterDim.z = 1;
            cfg.numAttrs = 2;
        }
        void* args[1] = {&p};
        cudaError_t e = cudaLaunchKernelExC(&cfg, g.func, args);
        if (e != cudaSuccess) return cuda_fail(e, "kernel launch");
    }
    if (forked) {
        // Join: the caller's stream continues once both side launches are done.
        cudaError_t e = cudaSuccess;
        for (int i = 0; e == cudaSuccess && i < 2; ++i) {
            e = cudaEventRecord(h->join[i], h->side[i]);
            if (e == cudaSuccess) e = cudaStreamWaitEvent(s, h->join[i], 0);
        }
        if (e != cudaSuccess) return cuda_fail(e, "joining the per-sequence split launches");
    }
    return FA_OK;
}

int fa_decode_run_noalloc(int num_q_heads, int num_kv_heads, int qk_depth, int nope_depth, int ov_depth,
                          int page_size, int num_q, int splitk, const void* q, const void* k_pages,
                          const void* v_pages, const int32_t* page_table, const int32_t* seq_lens, float scale,
                          void* out, float* lse, void* stream, int batch, int max_pages_per_seq, int num_pages,
                          int status_slot, uint32_t* status_out)
{
    g_last_error.clear();
    if (status_slot < 0 || status_slot >= FA_NOALLOC_STATUS_SLOTS)
        return fail(FA_ERR_INVALID_ARG, "status_slot %d is outside the %d status words of the static array",
                    status_slot, FA_NOALLOC_STATUS_SLOTS);
    // The plan lives on this stack frame; its tensor maps are encoded on the
    // host. Without the handle's scratch and side streams the plan takes no
    // stream-K partition and runs the per-sequence split's launches one after
    // another on `stream`.
    fa_decode plan{};
    int rc = plan_decode(plan, num_q_heads, num_kv_heads, qk_depth, nope_depth, ov_depth, page_size, num_q, splitk);
    if (rc) return rc;
    unsigned int* base = nullptr;
    if ((rc = noalloc_status_base(plan.device, &base))) return rc;
    plan.d_status = base + status_slot;
    // The array keeps whatever the previous call on this slot left: clear the
    // word this call reports into, in stream order before the launch.
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e = cudaMemsetAsync(plan.d_status, 0, sizeof(unsigned int), s);
    if (e != cudaSuccess) return cuda_fail(e, "clearing the static status word");
    if ((rc = fa_decode_run(&plan, q, k_pages, v_pages, page_table, seq_lens, scale, out, lse, stream, batch,
                            max_pages_per_seq, num_pages)))
        return rc;
    if (!status_out) return FA_OK;
    e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
    unsigned int st = 0;
    e = cudaMemcpy(&st, plan.d_status, sizeof st, cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return cuda_fail(e, "reading the static status word");
    *status_out = st;
    if (st)
        return fail(FA_ERR_DEVICE, "device status 0x%x:%s%s", st, (st & FA_STATUS_TIMEOUT) ? " wait timed out" : "",
                    (st & FA_STATUS_BAD_PAGE) ? " page id or length out of range" : "");
    return FA_OK;
}

}  // extern "C"
