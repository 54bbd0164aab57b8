// C ABI of the paged-attention library: argument checks, tensor-map set-up,
// the dispatch rule, and the device error word. No entry point allocates
// device memory; every launch goes on the caller's stream.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>
#include <math.h>
#include <stdint.h>
#include <string.h>

#include <algorithm>
#include <atomic>
#include <chrono>
#include <mutex>

#include "../../include/pagedattn.h"
#include "../../include/pagedattn_test.h"
#include "pa_internal.h"

namespace pa {

// Device error word: kernels OR PA_DEVERR_* bits into it; pa_get_device_error
// reads and clears it. One copy per device that loads the library.
__device__ unsigned int g_device_error;

uint64_t next_launch_stamp()
{
    static std::atomic<uint64_t> stamp{0};
    if (stamp.load(std::memory_order_relaxed) == 0) {
        const uint64_t seed = uint64_t(
            std::chrono::steady_clock::now().time_since_epoch().count()) * 0x9E3779B97F4A7C15ull;
        uint64_t expected = 0;
        stamp.compare_exchange_strong(expected, (seed >> 16) | 1ull);
    }
    uint64_t st = stamp.fetch_add(1, std::memory_order_relaxed) & ((uint64_t(1) << 48) - 1);
    return st == 0 ? 1 : st;
}

namespace {

constexpr int kMaxDevices = 64;

struct DeviceInfo {
    bool ready = false;
    int id = 0;
    int sm_count = 0;
    int max_smem_optin = 0;
    unsigned* err = nullptr;  // device address of g_device_error
};

std::mutex g_mutex;
thread_local bool t_arm_unset_wait = false;  // test support, see pa_debug_arm_wait_timeout
thread_local int t_prefill_variant = 0;      // see pa_debug_prefill_variant
DeviceInfo g_devices[kMaxDevices];
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

pa_status device_info(DeviceInfo** out)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
        return PA_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_mutex);
    DeviceInfo& d = g_devices[dev];
    if (!d.ready) {
        int sms = 0, smem = 0;
        if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&smem, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) !=
                cudaSuccess)
            return PA_ERR_CUDA;
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_device_error) != cudaSuccess)
            return PA_ERR_CUDA;
        d.id = dev;
        d.sm_count = sms;
        d.max_smem_optin = smem;
        d.err = static_cast<unsigned*>(p);
        d.ready = true;
    }
    *out = &d;
    return PA_OK;
}

pa_status get_encoder(PFN_cuTensorMapEncodeTiled_v12000* fn)
{
    std::lock_guard<std::mutex> lock(g_mutex);
    if (!g_encode) {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                             cudaEnableDefault, &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess || !p)
            return PA_ERR_CUDA;
        g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    }
    *fn = g_encode;
    return PA_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool pow2_in(int v, int lo, int hi) { return v >= lo && v <= hi && (v & (v - 1)) == 0; }

// Checks shared by the attention entry points.
pa_status check_attention(const void* query, const void* key_pages, const void* value_pages,
                          const int32_t* block_table, const int32_t* context_lens,
                          int32_t page_size, float scale, const void* out, const pa_shape& s)
{
    if (!query || !key_pages || !value_pages || !block_table || !context_lens || !out)
        return PA_ERR_INVALID_ARG;
    if (s.batch <= 0 || s.num_q_heads <= 0 || s.num_kv_heads <= 0 || s.q_len <= 0 ||
        s.num_pages <= 0 || s.max_pages <= 0 || s.head_dim <= 0)
        return PA_ERR_INVALID_ARG;
    if (!(scale > 0.f) || !isfinite(scale))
        return PA_ERR_INVALID_ARG;
    if (!aligned16(query) || !aligned16(key_pages) || !aligned16(value_pages) || !aligned16(out))
        return PA_ERR_INVALID_ARG;
    if (s.head_dim != 64 && s.head_dim != 128)
        return PA_ERR_UNSUPPORTED;
    if (s.num_q_heads % s.num_kv_heads != 0)
        return PA_ERR_UNSUPPORTED;
    if (!pow2_in(page_size, 1, 256))
        return PA_ERR_UNSUPPORTED;
    // TMA row coordinates and in-kernel page arithmetic are 32-bit.
    if (int64_t(s.num_pages) * s.num_kv_heads * page_size >= (int64_t(1) << 31))
        return PA_ERR_UNSUPPORTED;
    if (int64_t(s.max_pages) * page_size >= (int64_t(1) << 30))
        return PA_ERR_UNSUPPORTED;
    return PA_OK;
}

// Recently encoded tensor maps of this host thread (a map depends only on
// the pool's address and shape).
struct MapCacheEntry {
    CUtensorMap map;
    const void* pool;
    uint64_t rows;
    int32_t D, ps;
    bool fp8;
    bool valid;
};
constexpr int kMapCache = 8;
thread_local MapCacheEntry t_map_cache[kMapCache];
thread_local int t_map_next = 0;

pa_status encode_pool_map_uncached(CUtensorMap* map, const void* pool, const pa_shape& s,
                                   int32_t ps, bool fp8);

// 2-D view of a page pool: rows = P * H_kv * page_size, columns = D (bf16
// elements, or e4m3 codes of one byte when fp8).
pa_status encode_pool_map(CUtensorMap* map, const void* pool, const pa_shape& s, int32_t ps,
                          bool fp8 = false)
{
    const uint64_t rows = uint64_t(s.num_pages) * s.num_kv_heads * ps;
    for (int i = 0; i < kMapCache; ++i) {
        const MapCacheEntry& e = t_map_cache[i];
        if (e.valid && e.pool == pool && e.rows == rows && e.D == s.head_dim && e.ps == ps &&
            e.fp8 == fp8) {
            *map = e.map;
            return PA_OK;
        }
    }
    pa_status st = encode_pool_map_uncached(map, pool, s, ps, fp8);
    if (st == PA_OK) {
        MapCacheEntry& e = t_map_cache[t_map_next];
        t_map_next = (t_map_next + 1) % kMapCache;
        e.map = *map;
        e.pool = pool;
        e.rows = rows;
        e.D = s.head_dim;
        e.ps = ps;
        e.fp8 = fp8;
        e.valid = true;
    }
    return st;
}

pa_status encode_pool_map_uncached(CUtensorMap* map, const void* pool, const pa_shape& s,
                                   int32_t ps, bool fp8)
{
    PFN_cuTensorMapEncodeTiled_v12000 enc;
    pa_status st = get_encoder(&enc);
    if (st != PA_OK)
        return st;
    const cuuint64_t dims[2] = {cuuint64_t(s.head_dim),
                                cuuint64_t(s.num_pages) * s.num_kv_heads * ps};
    const cuuint64_t strides[1] = {cuuint64_t(s.head_dim) * (fp8 ? 1 : 2)};
    const int box_rows = ps < kDecodeTokens ? ps : kDecodeTokens;
    // a box row is 128 bytes: 64 bf16 or 128 e4m3 codes
    const cuuint32_t box[2] = {fp8 ? 128u : 64u, cuuint32_t(box_rows)};
    const cuuint32_t estr[2] = {1u, 1u};
    // Boxes of 8+ rows land on 1024-byte boundaries and use the 128-byte
    // swizzle; smaller pages use a linear layout (their destinations are only
    // 128-byte aligned).
    const CUtensorMapSwizzle swz =
        box_rows >= 8 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE;
    CUresult r = enc(map, fp8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
                     const_cast<void*>(pool), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? PA_OK : PA_ERR_CUDA;
}

// 2-D bf16 tensor map over `rows` rows of `cols` columns, boxes of 64 columns
// x box_rows rows, 128-byte swizzle (queries of both kernels, prefill K/V).
pa_status encode_rows_map(CUtensorMap* map, const void* base, uint64_t rows, uint32_t box_rows,
                          uint32_t cols = 128)
{
    PFN_cuTensorMapEncodeTiled_v12000 enc;
    pa_status st = get_encoder(&enc);
    if (st != PA_OK)
        return st;
    const cuuint64_t dims[2] = {cuuint64_t(cols), cuuint64_t(rows)};
    const cuuint64_t strides[1] = {cuuint64_t(cols) * 2};
    const cuuint32_t box[2] = {64u, box_rows};
    const cuuint32_t estr[2] = {1u, 1u};
    CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims,
                     strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                     CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? PA_OK : PA_ERR_CUDA;
}

// 3-D bf16 tensor map over the attention output [B * H_q, L, cols]: boxes of
// 64 columns x 32 rows of one (request, head), 128-byte swizzle (the pairs
// prefill kernel's output stores; rows past L are outside the map).
pa_status encode_out_map(CUtensorMap* map, void* base, uint64_t heads, uint64_t L, uint32_t cols)
{
    PFN_cuTensorMapEncodeTiled_v12000 enc;
    pa_status st = get_encoder(&enc);
    if (st != PA_OK)
        return st;
    const cuuint64_t dims[3] = {cuuint64_t(cols), cuuint64_t(L), cuuint64_t(heads)};
    const cuuint64_t strides[2] = {cuuint64_t(cols) * 2, cuuint64_t(cols) * 2 * L};
    const cuuint32_t box[3] = {64u, 32u, 1u};
    const cuuint32_t estr[3] = {1u, 1u, 1u};
    CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, base, dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? PA_OK : PA_ERR_CUDA;
}

// Workspace the split prefill kernel needs for this shape on this device, or
// 0 when the shape takes another prefill kernel (head_dim 64, pages of fewer
// than 8 tokens, one query head per KV group, or shared memory too small).
// (request, pair of query heads of one KV group, 128-row query tile) items of a
// prefill: ceil(G / 2) pairs per group (an odd group's last pair repeats its
// last head).
int64_t prefill_pair_items(const pa_shape& s)
{
    const int g = s.num_kv_heads > 0 ? s.num_q_heads / s.num_kv_heads : 0;
    return int64_t(s.batch) * ((int64_t(s.q_len) + 127) / 128) * s.num_kv_heads * ((g + 1) / 2);
}

size_t split_prefill_need(const pa_shape& s, int32_t page_size, const DeviceInfo* dev)
{
    if (s.head_dim != 128 || page_size < 8 || s.num_kv_heads <= 0 ||
        s.num_q_heads % s.num_kv_heads != 0 || s.num_q_heads / s.num_kv_heads < 2)
        return 0;
    if (prefill_split_smem_bytes() > size_t(dev->max_smem_optin))
        return 0;
    // the same workspace serves the pairs kernel's tail pieces
    const size_t split = prefill_split_workspace_bytes(dev->sm_count);
    const size_t pieces = prefill_pairs_workspace_bytes(dev->sm_count);
    return split > pieces ? split : pieces;
}

// Prefill on tcgen05 (D = 128 or 64; pages of fewer than 8 tokens on the
// pairs kernel, whose loaders then copy K/V row by row). With a workspace of at least split_prefill_need
// bytes: the split kernel (K/V tiles spread evenly over one block per SM);
// otherwise the persistent pairs kernel (whole (request, head pair, 128-row
// query tile) items) or one block per (request, query head, query tile).
pa_status run_prefill_tc(const void* query, const void* key_pages, const void* value_pages,
                         const int32_t* block_table, const int32_t* context_lens,
                         int32_t page_size, float scale, int causal, void* out,
                         const pa_shape& s, cudaStream_t stream, void* workspace = nullptr,
                         size_t workspace_bytes = 0, float out_scale = 1.f,
                         void* piece_ws = nullptr, size_t piece_ws_bytes = 0)
{
    DeviceInfo* dev;
    pa_status st = device_info(&dev);
    if (st != PA_OK)
        return st;
    const size_t split_need = split_prefill_need(s, page_size, dev);
    const bool split = t_prefill_variant == 0 && workspace && split_need > 0 &&
                       workspace_bytes >= split_need &&
                       (reinterpret_cast<uintptr_t>(workspace) & 255u) == 0;
    // Two query heads of one KV group per block when the group has at least
    // two (an odd group's last pair repeats its last head), unless the one-head
    // kernel is requested. An odd group with fewer pair items than SMs takes
    // the one-head kernel, whose more numerous blocks fill the GPU better
    // (group of 7, one 512-row chunk after a 16k prefix: 209.6 against 219.8
    // us; with 256 pair items the pairs kernel is 22-33 % faster).
    const int g = s.num_q_heads / s.num_kv_heads;
    const int64_t pair_items = prefill_pair_items(s);
    // Only the pairs kernel has the 64-column form and the row-by-row loads of
    // small pages. With one query head per KV group it takes that head twice,
    // as an odd group's last pair.
    const bool d64 = s.head_dim == 64;
    const bool small_pages = page_size < 8;
    bool pairs = d64 || small_pages ||
                 (g >= 2 && t_prefill_variant != 1 &&
                  (g % 2 == 0 || t_prefill_variant >= 2 || pair_items >= dev->sm_count));
    if (pairs && prefill_pairs_smem_bytes(s.head_dim) > size_t(dev->max_smem_optin))
        pairs = false;
    if ((d64 || small_pages) && !pairs)
        return PA_ERR_UNSUPPORTED;
    if (!pairs && prefill_smem_bytes() > size_t(dev->max_smem_optin))
        return PA_ERR_UNSUPPORTED;
    const int64_t n_qtiles = (int64_t(s.q_len) + 127) / 128;
    const int64_t grid = int64_t(s.batch) * s.num_q_heads * n_qtiles;
    const int64_t q_rows = int64_t(s.batch) * s.num_q_heads * s.q_len;
    if (grid >= (int64_t(1) << 31) || q_rows >= (int64_t(1) << 31))
        return PA_ERR_UNSUPPORTED;
    const uint32_t box = uint32_t(page_size < 128 ? page_size : 128);
    CUtensorMap qmap, kmap, vmap;
    const uint64_t kv_rows = uint64_t(s.num_pages) * s.num_kv_heads * page_size;
    const uint32_t cols = uint32_t(s.head_dim);
    CUtensorMap omap;
    if ((st = encode_rows_map(&qmap, query, uint64_t(q_rows), 128u, cols)) != PA_OK ||
        (st = encode_rows_map(&kmap, key_pages, kv_rows, box, cols)) != PA_OK ||
        (st = encode_rows_map(&vmap, value_pages, kv_rows, box, cols)) != PA_OK ||
        (st = encode_out_map(&omap, out, uint64_t(s.batch) * s.num_q_heads, uint64_t(s.q_len), cols)) !=
            PA_OK)
        return st;
    PrefillArgs a;
    memset(&a, 0, sizeof a);
    a.out = static_cast<uint16_t*>(out);
    a.block_table = block_table;
    a.context_lens = context_lens;
    a.err = dev->err;
    a.B = s.batch;
    a.H_q = s.num_q_heads;
    a.H_kv = s.num_kv_heads;
    a.L = s.q_len;
    a.ps = page_size;
    a.max_pages = s.max_pages;
    a.num_pages = s.num_pages;
    a.G = s.num_q_heads / s.num_kv_heads;
    a.n_qtiles = int32_t(n_qtiles);
    a.box_rows = int32_t(box);
    a.scale_log2 = scale * 1.4426950408889634f;
    a.causal = causal ? 1 : 0;
    a.out_scale = out_scale;
    a.D = s.head_dim;
    a.key_pages = static_cast<const uint16_t*>(key_pages);
    a.value_pages = static_cast<const uint16_t*>(value_pages);
    a.piece_last = t_prefill_variant == 5 ? 1 : 0;
    if (split) {
        SplitPrefillArgs sa;
        memset(&sa, 0, sizeof sa);
        sa.out = a.out;
        sa.block_table = a.block_table;
        sa.context_lens = a.context_lens;
        sa.err = a.err;
        sa.B = a.B;
        sa.H_q = a.H_q;
        sa.H_kv = a.H_kv;
        sa.L = a.L;
        sa.ps = a.ps;
        sa.max_pages = a.max_pages;
        sa.num_pages = a.num_pages;
        sa.G = a.G;
        sa.n_qtiles = a.n_qtiles;
        sa.box_rows = a.box_rows;
        sa.scale_log2 = a.scale_log2;
        sa.causal = a.causal;
        sa.out_scale = a.out_scale;
        // An error the caller left pending is not ours to clear: note it, so
        // that only a refused cooperative launch of this call is cleared.
        const bool pending = cudaPeekAtLastError() != cudaSuccess;
        cudaError_t e = launch_prefill_split(qmap, kmap, vmap, sa, dev->sm_count, workspace,
                                             dev->id, stream);
        if (e == cudaSuccess)
            return PA_OK;
        if (e != cudaErrorNotSupported && e != cudaErrorCooperativeLaunchTooLarge)
            return PA_ERR_CUDA;
        // The register split is not available, or not every block could be
        // resident (another client holds SMs): the kernels below.
        if (e == cudaErrorCooperativeLaunchTooLarge && !pending)
            (void)cudaGetLastError();
    }
    // The pairs kernel's tail pieces use the caller's workspace (pa_attention's).
    // Test setting 4: a grid of two thirds of the items, so that small shapes
    // have blocks of one item and of two, and get pieces.
    const bool small_grid = t_prefill_variant == 4 || t_prefill_variant == 5;
    const int grid_cap = small_grid ? int((2 * pair_items + 2) / 3) : dev->sm_count;
    cudaError_t e = pairs ? launch_prefill_pairs(qmap, kmap, vmap, omap, a, dev->id, grid_cap,
                                                 t_prefill_variant == 0 || small_grid ? piece_ws : nullptr,
                                                 piece_ws_bytes, stream)
                          : launch_prefill(qmap, kmap, vmap, a, dev->id, stream);
    if (pairs && e == cudaErrorNotSupported) {   // register split not available
        if (d64 || small_pages)
            return PA_ERR_UNSUPPORTED;
        e = launch_prefill(qmap, kmap, vmap, a, dev->id, stream);   // one head per block
    }
    return e == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

// (request, KV head, 16-row tile) count of a call: the limit kMaxSegments
// applies to it.
int64_t decode_segments(const pa_shape& s)
{
    const int64_t G = s.num_q_heads / s.num_kv_heads;
    const int64_t MT = (G * s.q_len + kDecodeRows - 1) / kDecodeRows;
    return int64_t(s.batch) * s.num_kv_heads * MT;
}

}  // namespace

DecodePlan decode_plan(const pa_shape& s, bool fp8)
{
    DecodePlan p;
    const int64_t G = s.num_q_heads / s.num_kv_heads;
    p.MT = int32_t((G * s.q_len + kDecodeRows - 1) / kDecodeRows);
    p.TG = fp8 || p.MT <= 1 ? 1 : p.MT == 2 ? 2 : 4;
    p.MS = (p.MT + p.TG - 1) / p.TG;
    p.nseg = int64_t(s.batch) * s.num_kv_heads * p.MS;
    return p;
}

namespace {

// Runs the split-KV kernel. whole_segments = 1 gives every block whole
// segments (no partial states, no workspace).
pa_status run_split_kv(const void* query, const void* key_pages, const void* value_pages,
                       const int32_t* block_table, const int32_t* context_lens,
                       int32_t page_size, float scale, int causal, void* out,
                       const pa_shape& s, int32_t max_context_len, void* workspace,
                       size_t workspace_bytes, int whole_segments, cudaStream_t stream,
                       int dense = 0, int fp8 = 0, float k_scale = 1.f, float v_scale = 1.f)
{
    DeviceInfo* dev;
    pa_status st = device_info(&dev);
    if (st != PA_OK)
        return st;
    const int G = s.num_q_heads / s.num_kv_heads;
    const int64_t R = int64_t(G) * s.q_len;
    if (R >= (int64_t(1) << 30) || decode_segments(s) > kMaxSegments)
        return PA_ERR_UNSUPPORTED;
    const DecodePlan plan = decode_plan(s, fp8 != 0);
    const int64_t nseg = plan.nseg;
    const size_t smem = decode_smem_bytes(s.head_dim, s.batch, fp8 != 0, plan.TG);
    if (smem > size_t(dev->max_smem_optin))
        return PA_ERR_UNSUPPORTED;  // batch too large for the per-block prefix table

    const int grid_max = decode_max_grid(dev->sm_count);
    int64_t grid = grid_max;
    if (whole_segments) {
        grid = nseg < grid_max ? nseg : grid_max;
    } else if (max_context_len > 0) {
        const int64_t gran = (int64_t(max_context_len) + kDecodeTokens - 1) / kDecodeTokens;
        const int64_t bound = nseg * (gran > 0 ? gran : 1);
        if (bound < grid)
            grid = bound;
    }
    if (grid < 1)
        grid = 1;

    DecodeArgs a;
    memset(&a, 0, sizeof a);
    if (!whole_segments) {
        const size_t need = decode_workspace_bytes(nseg, grid_max, s.head_dim, plan.TG);
        if (!workspace || workspace_bytes < need || (reinterpret_cast<uintptr_t>(workspace) & 15u))
            return PA_ERR_WORKSPACE;
        a.partials = static_cast<float*>(workspace);
    }
    CUtensorMap kmap, vmap;
    if ((st = encode_pool_map(&kmap, key_pages, s, page_size, fp8 != 0)) != PA_OK)
        return st;
    if ((st = encode_pool_map(&vmap, value_pages, s, page_size, fp8 != 0)) != PA_OK)
        return st;

    a.q = static_cast<const uint16_t*>(query);
    a.out = static_cast<uint16_t*>(out);
    a.block_table = block_table;
    a.context_lens = context_lens;
    a.err = dev->err;
    a.B = s.batch;
    a.H_q = s.num_q_heads;
    a.H_kv = s.num_kv_heads;
    a.L = s.q_len;
    a.D = s.head_dim;
    a.ps = page_size;
    a.max_pages = s.max_pages;
    a.num_pages = s.num_pages;
    a.G = G;
    a.R = int32_t(R);
    a.MS = plan.MS;
    a.TG = plan.TG;
    a.box_rows = page_size < kDecodeTokens ? page_size : kDecodeTokens;
    a.swz = a.box_rows >= 8 ? 7 : 0;
    a.whole_segments = whole_segments;
    a.dense = dense;
    // e4m3 pages: the kernel's K and V fragments hold the code values; the
    // per-tensor scales go into the softmax scale and the output
    a.scale_log2 = scale * 1.4426950408889634f * (fp8 ? k_scale : 1.f);
    a.causal = causal ? 1 : 0;
    a.fp8 = fp8 ? 1 : 0;
    a.v_scale = fp8 ? v_scale : 1.f;
    a.debug_unset_wait = t_arm_unset_wait ? 1 : 0;
    t_arm_unset_wait = false;
    CUtensorMap qmap;
    const uint64_t q_rows = uint64_t(s.batch) * s.num_q_heads * s.q_len;
    if ((st = encode_rows_map(&qmap, query, q_rows, uint32_t(kDecodeRows), uint32_t(s.head_dim))) !=
        PA_OK)
        return st;
    return launch_decode(kmap, vmap, qmap, a, int(grid), dev->id, stream) == cudaSuccess ? PA_OK
                                                                                   : PA_ERR_CUDA;
}

}  // namespace

pa_status validate_decode(const void* query, const void* key_pages, const void* value_pages,
                          const int32_t* block_table, const int32_t* context_lens,
                          int32_t page_size, float scale, const void* out, const pa_shape& s)
{
    pa_status st = check_attention(query, key_pages, value_pages, block_table, context_lens,
                                   page_size, scale, out, s);
    if (st != PA_OK)
        return st;
    DeviceInfo* dev;
    if ((st = device_info(&dev)) != PA_OK)
        return st;
    const int64_t R = int64_t(s.num_q_heads / s.num_kv_heads) * s.q_len;
    if (R >= (int64_t(1) << 30) || decode_segments(s) > kMaxSegments)
        return PA_ERR_UNSUPPORTED;
    const size_t smem = std::max(decode_smem_bytes(s.head_dim, s.batch),
                                 decode_smem_bytes(s.head_dim, s.batch, false,
                                                   decode_plan(s, false).TG));
    if (smem > size_t(dev->max_smem_optin))
        return PA_ERR_UNSUPPORTED;
    return PA_OK;
}

int64_t decode_segment_count(const pa_shape& s) { return decode_segments(s); }

}  // namespace pa

using namespace pa;

extern "C" {

pa_status pa_append_kv(const void* key, const void* value, void* key_pages, void* value_pages,
                       const int32_t* slot_mapping, int32_t page_size, pa_shape shape,
                       void* stream)
{
    if (!key || !value || !key_pages || !value_pages || !slot_mapping)
        return PA_ERR_INVALID_ARG;
    if (shape.batch <= 0 || shape.num_kv_heads <= 0 || shape.q_len < 0 || shape.num_pages <= 0 ||
        shape.head_dim <= 0)
        return PA_ERR_INVALID_ARG;
    if (!aligned16(key) || !aligned16(value) || !aligned16(key_pages) || !aligned16(value_pages))
        return PA_ERR_INVALID_ARG;
    if (shape.head_dim != 64 && shape.head_dim != 128)
        return PA_ERR_UNSUPPORTED;
    if (!pow2_in(page_size, 1, 256))
        return PA_ERR_UNSUPPORTED;
    if (2 * int64_t(shape.batch) * shape.q_len * shape.num_kv_heads * (shape.head_dim / 8) >=
        (int64_t(1) << 40))
        return PA_ERR_UNSUPPORTED;
    DeviceInfo* dev;
    pa_status st = device_info(&dev);
    if (st != PA_OK)
        return st;
    if (shape.q_len == 0)
        return PA_OK;
    AppendArgs a;
    memset(&a, 0, sizeof a);
    a.key = static_cast<const uint16_t*>(key);
    a.value = static_cast<const uint16_t*>(value);
    a.key_pages = static_cast<uint16_t*>(key_pages);
    a.value_pages = static_cast<uint16_t*>(value_pages);
    a.slot_mapping = slot_mapping;
    a.err = dev->err;
    a.B = shape.batch;
    a.L_new = shape.q_len;
    a.H_kv = shape.num_kv_heads;
    a.D = shape.head_dim;
    a.ps = page_size;
    a.num_pages = shape.num_pages;
    return launch_append(a, static_cast<cudaStream_t>(stream)) == cudaSuccess ? PA_OK
                                                                               : PA_ERR_CUDA;
}

size_t pa_decode_workspace_bytes(pa_shape shape)
{
    if (shape.batch <= 0 || shape.num_q_heads <= 0 || shape.num_kv_heads <= 0 ||
        shape.q_len <= 0 || shape.num_q_heads % shape.num_kv_heads != 0 ||
        (shape.head_dim != 64 && shape.head_dim != 128) ||
        decode_segments(shape) > kMaxSegments)
        return 0;
    DeviceInfo* dev;
    if (device_info(&dev) != PA_OK)
        return 0;
    // The bf16 plan's need; an e4m3 call's (one row tile per segment) is
    // never larger.
    const DecodePlan plan = decode_plan(shape, false);
    return decode_workspace_bytes(plan.nseg, decode_max_grid(dev->sm_count), shape.head_dim,
                                  plan.TG);
}

namespace {

// Prefill over e4m3 pools: the workspace holds the bf16 copies of K and V
// (B * P2 pages of [H_kv, 128, 128]), the copies' page table, then (256-byte
// aligned) the split prefill's workspace where that kernel serves the shape.
struct Fp8PrefillPlan {
    int64_t P2 = 0;
    pa_shape copy{};
    size_t kv_bytes = 0, table_off = 0, split_off = 0, split_bytes = 0, piece_bytes = 0, total = 0;
};

pa_status plan_prefill_fp8(const pa_shape& s, int32_t max_context_len, DeviceInfo* dev,
                           Fp8PrefillPlan* p)
{
    if (max_context_len < 0 || s.batch <= 0 || s.num_kv_heads <= 0 || s.num_q_heads <= 0)
        return PA_ERR_INVALID_ARG;
    p->P2 = fp8_copy_pages(max_context_len);
    const int64_t pages = int64_t(s.batch) * p->P2;
    if (pages * s.num_kv_heads * 128 >= (int64_t(1) << 31) || p->P2 * 128 >= (int64_t(1) << 30))
        return PA_ERR_UNSUPPORTED;
    p->copy = s;
    p->copy.head_dim = 128;
    p->copy.num_pages = int32_t(pages);
    p->copy.max_pages = int32_t(p->P2);
    p->kv_bytes = size_t(pages) * s.num_kv_heads * 128 * 128 * 2;
    p->table_off = 2 * p->kv_bytes;
    const size_t table_bytes = size_t(pages) * 4;
    p->split_off = (p->table_off + table_bytes + 255) & ~size_t(255);
    // the kernel choice of pa_attention's prefill route (split below 1.5
    // items per SM; from there to 2 items per SM the pairs kernel's tail
    // pieces, in the same place)
    const int64_t items = prefill_pair_items(s);
    const bool few = 2 * items < 3 * int64_t(dev->sm_count);
    p->split_bytes = few ? split_prefill_need(p->copy, 128, dev) : 0;
    p->piece_bytes = !few && items <= 2 * int64_t(dev->sm_count) && split_prefill_need(p->copy, 128, dev) > 0
                         ? prefill_pairs_workspace_bytes(dev->sm_count)
                         : 0;
    p->total = p->split_off + (p->split_bytes > p->piece_bytes ? p->split_bytes : p->piece_bytes);
    return PA_OK;
}

}  // namespace

size_t pa_prefill_fp8_workspace_bytes(pa_shape shape, int32_t max_context_len)
{
    if (shape.head_dim != 128)
        return 0;
    DeviceInfo* dev;
    if (device_info(&dev) != PA_OK)
        return 0;
    Fp8PrefillPlan p;
    if (plan_prefill_fp8(shape, max_context_len, dev, &p) != PA_OK)
        return 0;
    return p.total;
}

pa_status pa_prefill_fp8(const void* query, const void* key_pages, const void* value_pages,
                         const int32_t* block_table, const int32_t* context_lens,
                         int32_t page_size, float scale, float k_scale, float v_scale, int causal,
                         void* out, pa_shape shape, int32_t max_context_len, void* workspace,
                         size_t workspace_bytes, void* stream)
{
    pa_status st = check_attention(query, key_pages, value_pages, block_table, context_lens,
                                   page_size, scale, out, shape);
    if (st != PA_OK)
        return st;
    if (!(k_scale > 0.f) || !isfinite(k_scale) || !(v_scale > 0.f) || !isfinite(v_scale))
        return PA_ERR_INVALID_ARG;
    if (shape.head_dim != 128)
        return PA_ERR_UNSUPPORTED;
    DeviceInfo* dev;
    if ((st = device_info(&dev)) != PA_OK)
        return st;
    Fp8PrefillPlan p;
    if ((st = plan_prefill_fp8(shape, max_context_len, dev, &p)) != PA_OK)
        return st;
    if (!workspace || workspace_bytes < p.total || (reinterpret_cast<uintptr_t>(workspace) & 255u))
        return PA_ERR_WORKSPACE;
    uint8_t* w = static_cast<uint8_t*>(workspace);
    Fp8PagesArgs c;
    memset(&c, 0, sizeof c);
    c.key_pages = static_cast<const uint8_t*>(key_pages);
    c.value_pages = static_cast<const uint8_t*>(value_pages);
    c.block_table = block_table;
    c.context_lens = context_lens;
    c.key_out = reinterpret_cast<uint16_t*>(w);
    c.value_out = reinterpret_cast<uint16_t*>(w + p.kv_bytes);
    c.table_out = reinterpret_cast<int32_t*>(w + p.table_off);
    c.err = dev->err;
    c.B = shape.batch;
    c.H_kv = shape.num_kv_heads;
    c.ps = page_size;
    c.max_pages = shape.max_pages;
    c.num_pages = shape.num_pages;
    c.P2 = int32_t(p.P2);
    const cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (launch_fp8_pages_to_bf16(c, s) != cudaSuccess)
        return PA_ERR_CUDA;
    // k_scale into the softmax scale, v_scale into the output normalisation
    return run_prefill_tc(query, c.key_out, c.value_out, c.table_out, context_lens, 128,
                          scale * k_scale, causal, out, p.copy, s,
                          p.split_bytes ? w + p.split_off : nullptr, p.split_bytes, v_scale,
                          p.piece_bytes ? w + p.split_off : nullptr, p.piece_bytes);
}

namespace {

// Route of pa_attention_fp8: the e4m3 decode kernel carries one 16-row tile
// per segment (its K/V are read once per tile), so it takes query chunks of
// at most 8 rows per request, the rule of Week 3 Day 4, "Task 2".
int32_t route_fp8(const pa_shape& shape)
{
    if (shape.q_len <= 0)
        return -1;
    return shape.q_len <= 8 ? 0 : 1;
}

}  // namespace

size_t pa_attention_fp8_workspace_bytes(pa_shape shape, int32_t max_context_len)
{
    const int32_t route = route_fp8(shape);
    if (route < 0 || shape.head_dim != 128)
        return 0;
    return route == 0 ? pa_decode_workspace_bytes(shape)
                      : pa_prefill_fp8_workspace_bytes(shape, max_context_len);
}

pa_status pa_attention_fp8(const void* query, const void* key_pages, const void* value_pages,
                           const int32_t* block_table, const int32_t* context_lens,
                           int32_t page_size, float scale, float k_scale, float v_scale,
                           int causal, void* out, pa_shape shape, int32_t max_context_len,
                           void* workspace, size_t workspace_bytes, void* stream)
{
    const int32_t route = route_fp8(shape);
    if (route < 0)
        return PA_ERR_INVALID_ARG;
    if (route == 0)
        return pa_decode_fp8(query, key_pages, value_pages, block_table, context_lens, page_size,
                             scale, k_scale, v_scale, causal, out, shape, max_context_len,
                             workspace, workspace_bytes, stream);
    return pa_prefill_fp8(query, key_pages, value_pages, block_table, context_lens, page_size,
                          scale, k_scale, v_scale, causal, out, shape, max_context_len, workspace,
                          workspace_bytes, stream);
}

pa_status pa_append_kv_fp8(const void* key, const void* value, void* key_pages,
                           void* value_pages, const int32_t* slot_mapping, int32_t page_size,
                           float k_scale, float v_scale, pa_shape shape, void* stream)
{
    if (!key || !value || !key_pages || !value_pages || !slot_mapping)
        return PA_ERR_INVALID_ARG;
    if (shape.batch <= 0 || shape.num_kv_heads <= 0 || shape.q_len < 0 || shape.num_pages <= 0 ||
        shape.head_dim <= 0)
        return PA_ERR_INVALID_ARG;
    if (!(k_scale > 0.f) || !isfinite(k_scale) || !(v_scale > 0.f) || !isfinite(v_scale))
        return PA_ERR_INVALID_ARG;
    if (!aligned16(key) || !aligned16(value) || !aligned16(key_pages) || !aligned16(value_pages))
        return PA_ERR_INVALID_ARG;
    if (shape.head_dim != 128)
        return PA_ERR_UNSUPPORTED;
    if (!pow2_in(page_size, 1, 256))
        return PA_ERR_UNSUPPORTED;
    if (2 * int64_t(shape.batch) * shape.q_len * shape.num_kv_heads * (shape.head_dim / 8) >=
        (int64_t(1) << 40))
        return PA_ERR_UNSUPPORTED;
    DeviceInfo* dev;
    pa_status st = device_info(&dev);
    if (st != PA_OK)
        return st;
    if (shape.q_len == 0)
        return PA_OK;
    AppendArgs a;
    memset(&a, 0, sizeof a);
    a.key = static_cast<const uint16_t*>(key);
    a.value = static_cast<const uint16_t*>(value);
    a.key_pages = static_cast<uint16_t*>(key_pages);     // byte pages; the kernel casts back
    a.value_pages = static_cast<uint16_t*>(value_pages);
    a.slot_mapping = slot_mapping;
    a.err = dev->err;
    a.B = shape.batch;
    a.L_new = shape.q_len;
    a.H_kv = shape.num_kv_heads;
    a.D = shape.head_dim;
    a.ps = page_size;
    a.num_pages = shape.num_pages;
    a.fp8 = 1;
    a.k_scale = k_scale;
    a.v_scale = v_scale;
    return launch_append(a, static_cast<cudaStream_t>(stream)) == cudaSuccess ? PA_OK
                                                                               : PA_ERR_CUDA;
}

pa_status pa_decode_fp8(const void* query, const void* key_pages, const void* value_pages,
                        const int32_t* block_table, const int32_t* context_lens, int32_t page_size,
                        float scale, float k_scale, float v_scale, int causal, void* out,
                        pa_shape shape, int32_t max_context_len, void* workspace,
                        size_t workspace_bytes, void* stream)
{
    pa_status st = check_attention(query, key_pages, value_pages, block_table, context_lens,
                                   page_size, scale, out, shape);
    if (st != PA_OK)
        return st;
    if (!(k_scale > 0.f) || !isfinite(k_scale) || !(v_scale > 0.f) || !isfinite(v_scale))
        return PA_ERR_INVALID_ARG;
    if (shape.head_dim != 128)
        return PA_ERR_UNSUPPORTED;
    return run_split_kv(query, key_pages, value_pages, block_table, context_lens, page_size, scale,
                        causal, out, shape, max_context_len, workspace, workspace_bytes, 0,
                        static_cast<cudaStream_t>(stream), 0, 1, k_scale, v_scale);
}

pa_status pa_decode(const void* query, const void* key_pages, const void* value_pages,
                    const int32_t* block_table, const int32_t* context_lens, int32_t page_size,
                    float scale, int causal, void* out, pa_shape shape, int32_t max_context_len,
                    void* workspace, size_t workspace_bytes, void* stream)
{
    pa_status st = check_attention(query, key_pages, value_pages, block_table, context_lens,
                                   page_size, scale, out, shape);
    if (st != PA_OK)
        return st;
    return run_split_kv(query, key_pages, value_pages, block_table, context_lens, page_size,
                        scale, causal, out, shape, max_context_len, workspace, workspace_bytes,
                        0, static_cast<cudaStream_t>(stream));
}

pa_status pa_gather_kv(const void* key_pages, const void* value_pages, const int32_t* block_table,
                       const int32_t* context_lens, int32_t page_size, pa_shape shape,
                       int32_t dense_len, void* key_dense, void* value_dense, void* stream)
{
    if (!key_pages || !value_pages || !block_table || !context_lens || !key_dense || !value_dense)
        return PA_ERR_INVALID_ARG;
    if (shape.batch <= 0 || shape.num_kv_heads <= 0 || shape.num_pages <= 0 ||
        shape.max_pages <= 0 || shape.head_dim <= 0 || dense_len <= 0)
        return PA_ERR_INVALID_ARG;
    if (!aligned16(key_pages) || !aligned16(value_pages) || !aligned16(key_dense) ||
        !aligned16(value_dense))
        return PA_ERR_INVALID_ARG;
    if (shape.head_dim != 64 && shape.head_dim != 128)
        return PA_ERR_UNSUPPORTED;
    if (!pow2_in(page_size, 1, 256))
        return PA_ERR_UNSUPPORTED;
    if (int64_t(shape.num_pages) * shape.num_kv_heads * page_size >= (int64_t(1) << 31) ||
        int64_t(shape.max_pages) * page_size >= (int64_t(1) << 30) ||
        2 * int64_t(shape.batch) * shape.num_kv_heads * dense_len * (shape.head_dim / 8) >=
            (int64_t(1) << 40))
        return PA_ERR_UNSUPPORTED;
    DeviceInfo* dev;
    pa_status st = device_info(&dev);
    if (st != PA_OK)
        return st;
    GatherArgs a;
    a.key_pages = static_cast<const uint16_t*>(key_pages);
    a.value_pages = static_cast<const uint16_t*>(value_pages);
    a.block_table = block_table;
    a.context_lens = context_lens;
    a.key_dense = static_cast<uint16_t*>(key_dense);
    a.value_dense = static_cast<uint16_t*>(value_dense);
    a.err = dev->err;
    a.B = shape.batch;
    a.H_kv = shape.num_kv_heads;
    a.D = shape.head_dim;
    a.ps = page_size;
    a.num_pages = shape.num_pages;
    a.max_pages = shape.max_pages;
    a.dense_len = dense_len;
    return launch_gather(a, static_cast<cudaStream_t>(stream)) == cudaSuccess ? PA_OK
                                                                               : PA_ERR_CUDA;
}

pa_status pa_decode_dense(const void* query, const void* key_dense, const void* value_dense,
                          const int32_t* context_lens, int32_t dense_len, float scale, int causal,
                          void* out, pa_shape shape, int32_t max_context_len, void* workspace,
                          size_t workspace_bytes, void* stream)
{
    if (dense_len < 64 || dense_len % 64 != 0)
        return PA_ERR_UNSUPPORTED;
    // The dense buffers are a pool of B pages of dense_len tokens, request b
    // in page b (the kernel does not read a block table for them).
    pa_shape s = shape;
    s.num_pages = shape.batch;
    s.max_pages = 1;
    if (!query || !key_dense || !value_dense || !context_lens || !out)
        return PA_ERR_INVALID_ARG;
    if (s.batch <= 0 || s.num_q_heads <= 0 || s.num_kv_heads <= 0 || s.q_len <= 0 ||
        s.head_dim <= 0)
        return PA_ERR_INVALID_ARG;
    if (!(scale > 0.f) || !isfinite(scale))
        return PA_ERR_INVALID_ARG;
    if (!aligned16(query) || !aligned16(key_dense) || !aligned16(value_dense) || !aligned16(out))
        return PA_ERR_INVALID_ARG;
    if (s.head_dim != 64 && s.head_dim != 128)
        return PA_ERR_UNSUPPORTED;
    if (s.num_q_heads % s.num_kv_heads != 0)
        return PA_ERR_UNSUPPORTED;
    if (int64_t(s.batch) * s.num_kv_heads * dense_len >= (int64_t(1) << 31) ||
        int64_t(dense_len) >= (int64_t(1) << 30))
        return PA_ERR_UNSUPPORTED;
    return run_split_kv(query, key_dense, value_dense, nullptr, context_lens, dense_len, scale,
                        causal, out, s, max_context_len, workspace, workspace_bytes, 0,
                        static_cast<cudaStream_t>(stream), 1);
}

namespace {

// pa_prefill; piece_ws: room for the pairs kernel's tail pieces (pa_attention's
// workspace), or null.
pa_status prefill_route(const void* query, const void* key_pages, const void* value_pages,
                        const int32_t* block_table, const int32_t* context_lens, int32_t page_size,
                        float scale, int causal, void* out, pa_shape shape, void* stream,
                        void* piece_ws, size_t piece_ws_bytes)
{
    pa_status st = check_attention(query, key_pages, value_pages, block_table, context_lens,
                                   page_size, scale, out, shape);
    if (st != PA_OK)
        return st;
    if (shape.head_dim == 128 || shape.head_dim == 64) {
        st = run_prefill_tc(query, key_pages, value_pages, block_table, context_lens, page_size,
                            scale, causal, out, shape, static_cast<cudaStream_t>(stream), nullptr, 0,
                            1.f, piece_ws, piece_ws_bytes);
        if (st != PA_ERR_UNSUPPORTED || shape.head_dim == 128)
            return st;
    }
    // Without the pairs kernel's register split (head_dim 64, or pages of
    // fewer than 8 tokens): the split-KV kernel with whole segments per block.
    return run_split_kv(query, key_pages, value_pages, block_table, context_lens, page_size,
                        scale, causal, out, shape, 0, nullptr, 0, 1,
                        static_cast<cudaStream_t>(stream));
}

}  // namespace

pa_status pa_prefill(const void* query, const void* key_pages, const void* value_pages,
                     const int32_t* block_table, const int32_t* context_lens, int32_t page_size,
                     float scale, int causal, void* out, pa_shape shape, void* stream)
{
    return prefill_route(query, key_pages, value_pages, block_table, context_lens, page_size, scale,
                         causal, out, shape, stream, nullptr, 0);
}

size_t pa_prefill_workspace_bytes(pa_shape shape, int32_t page_size)
{
    DeviceInfo* dev;
    if (device_info(&dev) != PA_OK)
        return 0;
    return split_prefill_need(shape, page_size, dev);
}

pa_status pa_prefill_split(const void* query, const void* key_pages, const void* value_pages,
                           const int32_t* block_table, const int32_t* context_lens,
                           int32_t page_size, float scale, int causal, void* out, pa_shape shape,
                           void* workspace, size_t workspace_bytes, void* stream)
{
    pa_status st = check_attention(query, key_pages, value_pages, block_table, context_lens,
                                   page_size, scale, out, shape);
    if (st != PA_OK)
        return st;
    DeviceInfo* dev;
    if ((st = device_info(&dev)) != PA_OK)
        return st;
    const size_t need = split_prefill_need(shape, page_size, dev);
    if (need == 0)   // another prefill kernel serves this shape; no workspace used
        return pa_prefill(query, key_pages, value_pages, block_table, context_lens, page_size,
                          scale, causal, out, shape, stream);
    if (!workspace || workspace_bytes < need || (reinterpret_cast<uintptr_t>(workspace) & 255u))
        return PA_ERR_WORKSPACE;
    return run_prefill_tc(query, key_pages, value_pages, block_table, context_lens, page_size,
                          scale, causal, out, shape, static_cast<cudaStream_t>(stream), workspace,
                          workspace_bytes);
}

int32_t pa_attention_route(pa_shape shape, int32_t max_context_len)
{
    if (shape.q_len <= 0 || shape.num_q_heads <= 0 || shape.num_kv_heads <= 0)
        return -1;
    // The split-KV decode reads a KV group's K/V once per 64 of its query
    // rows (four 16-row tiles per segment) and its cost grows with the rows;
    // the persistent tile prefill pays a fixed cost per 128-row tile.
    // Measured crossover on GB300 (32 requests, contexts of 1k to 4k tokens,
    // page size 16, 1, 4 and 7 query heads per KV group): decode is faster up
    // to 24 rows per request (within 3 % at 1k contexts), the two tie at 32
    // rows from about 3k-token contexts on, and prefill is faster beyond.
    return shape.q_len <= 24 || (shape.q_len <= 32 && max_context_len >= 3072) ? 0 : 1;
}

pa_status pa_attention(const void* query, const void* key_pages, const void* value_pages,
                       const int32_t* block_table, const int32_t* context_lens, int32_t page_size,
                       float scale, int causal, void* out, pa_shape shape,
                       int32_t max_context_len, void* workspace, size_t workspace_bytes,
                       void* stream)
{
    const int32_t route = pa_attention_route(shape, max_context_len);
    if (route < 0)
        return PA_ERR_INVALID_ARG;
    if (route == 0)
        return pa_decode(query, key_pages, value_pages, block_table, context_lens, page_size,
                         scale, causal, out, shape, max_context_len, workspace, workspace_bytes,
                         stream);
    if (workspace && t_prefill_variant != 4 && t_prefill_variant != 5) {
        // The split kernel pays for its balance at every piece boundary; it
        // is the faster one when the (request, head pair, query tile) items
        // are too few to fill the SMs in whole waves (measured: 1.75x on one
        // 512-row chunk after a 16k prefix, 64 items; equal at 1.7 items per
        // SM; slower beyond).
        DeviceInfo* dev;
        pa_status st = device_info(&dev);
        if (st != PA_OK)
            return st;
        const size_t need = split_prefill_need(shape, page_size, dev);
        const int64_t items = prefill_pair_items(shape);
        if (need > 0 && workspace_bytes >= need && 2 * items < 3 * int64_t(dev->sm_count) &&
            (reinterpret_cast<uintptr_t>(workspace) & 255u) == 0)
            return pa_prefill_split(query, key_pages, value_pages, block_table, context_lens,
                                    page_size, scale, causal, out, shape, workspace,
                                    workspace_bytes, stream);
    }
    // the pairs kernel, which balances one to two items per block with tail
    // pieces in the workspace
    return prefill_route(query, key_pages, value_pages, block_table, context_lens, page_size, scale,
                         causal, out, shape, stream, workspace, workspace_bytes);
}

pa_status pa_get_device_error(void* stream, uint32_t* flags)
{
    DeviceInfo* dev;
    pa_status st = device_info(&dev);
    if (st != PA_OK)
        return st;
    if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess)
        return PA_ERR_CUDA;
    unsigned v = 0;
    const unsigned zero = 0;
    if (cudaMemcpyFromSymbol(&v, g_device_error, sizeof v) != cudaSuccess)
        return PA_ERR_CUDA;
    if (cudaMemcpyToSymbol(g_device_error, &zero, sizeof zero) != cudaSuccess)
        return PA_ERR_CUDA;
    if (flags)
        *flags = v;
    if (v & PA_DEVERR_TIMEOUT)
        return PA_ERR_DEVICE_TIMEOUT;
    return v ? PA_ERR_DEVICE_BOUNDS : PA_OK;
}

const char* pa_status_string(pa_status status)
{
    switch (status) {
    case PA_OK: return "PA_OK";
    case PA_ERR_INVALID_ARG: return "PA_ERR_INVALID_ARG: invalid argument";
    case PA_ERR_UNSUPPORTED: return "PA_ERR_UNSUPPORTED: unsupported shape or page size";
    case PA_ERR_WORKSPACE: return "PA_ERR_WORKSPACE: workspace missing, too small or misaligned";
    case PA_ERR_NO_PAGES: return "PA_ERR_NO_PAGES: page pool or block-table row full (nothing changed)";
    case PA_ERR_CUDA: return "PA_ERR_CUDA: CUDA call or launch failed";
    case PA_ERR_DEVICE_BOUNDS: return "PA_ERR_DEVICE_BOUNDS: kernel met an out-of-range index";
    case PA_ERR_DEVICE_TIMEOUT: return "PA_ERR_DEVICE_TIMEOUT: kernel wait gave up";
    }
    return "unknown pa_status";
}

const char* pa_version(void) { return "0.1.0"; }

void pa_debug_arm_wait_timeout(void) { t_arm_unset_wait = true; }

int pa_debug_prefill_variant(int variant)
{
    const int prev = t_prefill_variant;
    t_prefill_variant = (variant == 1 || variant == 2 || variant == 4 || variant == 5) ? variant : 0;
    return prev;
}

}  // extern "C"
