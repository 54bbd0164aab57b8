// Causal page-walking prefill attention on the 5th-generation tensor cores.
//
// What it computes: for request b, query head h_q and query rows i in
// [0, L) (absolute position n_b - L + i), softmax(scale * q . K^T + causal
// mask) . V over the keys 0..position, K/V resolved page by page through
// block_table (Week 3 Day 4: Direct Paged Attention, "Task 2": long queries
// take a page-walking schedule that resolves every K/V tile through the block
// table, one page id per page; tiled on the tensor cores as that chapter's
// next day plans).
//
// Schedule (one block per (request, query head, tile of 128 query rows);
// the tiles with the most keys are launched first):
//   * warps 0, 2, 3 (loaders): TMA loads of the Q tile (128 x 128, once)
//     and of K and V tiles of 128 keys, page by page (one box of
//     min(page_size, 128) rows x 64 columns per page and half, the boxes of a
//     tile split over the three warps), 128-byte swizzle, two K and two V
//     stages released separately (a K stage as soon as its scores are
//     computed);
//   * warp 1 (one thread): tcgen05.mma kind::f16 (bf16 in, fp32 accumulate)
//     S = Q K^T into one of two TMEM score buffers, then O += P V (P from
//     TMEM) into the TMEM output accumulator, completion signalled by
//     tcgen05.commit; a score buffer is reused once its P V is done;
//   * warps 4-7 (one thread per row, TMEM lanes 0..127): the online-softmax
//     fold. Scores are masked by select (never multiplied), kept in the log2
//     domain; the running maximum used for the exponentials moves only when
//     a tile's maximum exceeds it by more than 2^8, in which case O (TMEM)
//     and the running sum are rescaled (the result is the same softmax:
//     exponentials of a stale maximum stay below 2^8). P (bf16) is written
//     back into the tile's score buffer in TMEM and read from there as the A
//     operand of P V, so it never crosses shared memory (whose bandwidth the
//     MMAs and the TMA copies already share). V rows past the context are
//     zeroed before P V. At the end, O / l -> bf16.
#include <cuda.h>
#include <cuda_bf16.h>
#include <math.h>
#include <stdint.h>

#include <atomic>

#include "pa_device.cuh"
#include "pa_internal.h"
#include "pa_tcgen05.cuh"

namespace pa {
namespace {

constexpr int kTile = 128;            // query rows per block = keys per K/V tile
constexpr int kThreads = 256;
constexpr int kSoftmaxWarp0 = 4;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColS0 = 0, kColS1 = 128, kColO = 256;
constexpr float kRescaleLog2 = 8.f;   // stale-max slack of the exponentials

struct Layout {
    static constexpr int kHalf = kTile * 128;   // 128 rows x 64 bf16 (128 B)
    static constexpr int kMat = 2 * kHalf;      // 128 x 128 bf16
    static constexpr int kQ = 0;
    static constexpr int kK = kQ + kMat;        // 2 stages
    static constexpr int kV = kK + 2 * kMat;    // 2 stages
    static constexpr int kBar = kV + 2 * kMat;  // 16 mbarriers
    static constexpr int kTmemSlot = kBar + 16 * 8;
    static constexpr int kMisc = kTmemSlot + 16;
    static constexpr int kBytes = kMisc + 16 + 1024;  // + alignment slack
};

enum Bar { kQFull = 0, kKFull0 = 1, kKEmpty0 = 3, kVFull0 = 5, kVEmpty0 = 7, kSFull0 = 9,
           kPFull = 11, kPVDone = 12, kMmaDone = 13 };

// Operand descriptors (128B swizzle). K-major [half][128 rows][128 B] (Q, K):
// k-step kk (16 elements along K) starts kmajor_off(kk) bytes in. MN-major
// (V: rows = keys, 128 B of columns per row, two 64-column halves): k-step kk
// (16 keys) starts 16 rows in.
__host__ __device__ constexpr uint32_t kmajor_off(int kk)
{
    return uint32_t(kk >> 2) * Layout::kHalf + uint32_t(kk & 3) * 32u;
}
__host__ __device__ constexpr uint32_t mnmajor_off(int kk) { return uint32_t(kk) * 16u * 128u; }
__device__ __forceinline__ uint64_t kmajor_base(uint32_t saddr) { return smem_desc_sw128(saddr, 16u, 1024u); }
__device__ __forceinline__ uint64_t mnmajor_base(uint32_t saddr)
{
    return smem_desc_sw128(saddr, uint32_t(Layout::kHalf), 1024u);
}

__global__ void __launch_bounds__(kThreads, 1)
    prefill_kernel(const __grid_constant__ CUtensorMap q_map,
                   const __grid_constant__ CUtensorMap key_map,
                   const __grid_constant__ CUtensorMap value_map, const PrefillArgs a)
{
    grid_dependency_wait();  // the previous kernel's outputs are visible from here on
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* bar = reinterpret_cast<uint64_t*>(smem + Layout::kBar);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + Layout::kTmemSlot);
    volatile int* misc = reinterpret_cast<volatile int*>(smem + Layout::kMisc);
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    // ---- which tile -------------------------------------------------------
    const int bh_count = a.B * a.H_q;
    const int t = a.n_qtiles - 1 - int(blockIdx.x / bh_count);
    const int bh = int(blockIdx.x % bh_count);
    const int b = bh / a.H_q;
    const int hq = bh - b * a.H_q;
    const int hk = hq / a.G;
    const int cap = a.max_pages * a.ps;
    int n = a.context_lens[b];
    if (n < 0 || n > cap) {
        if (threadIdx.x == 0)
            atomicOr(a.err, PA_DEVERR_CONTEXT_LEN_BIT);
        n = n < 0 ? 0 : cap;
    }
    const int row0 = t * kTile;
    const int rows = min(kTile, a.L - row0);
    const int p_last = n - a.L + row0 + rows - 1;   // position of the tile's last row
    int n_keys = a.causal ? min(n, p_last + 1) : n;
    if (n_keys < 0)
        n_keys = 0;
    const int nt = (n_keys + kTile - 1) / kTile;     // K/V tiles to visit

    const uint32_t sQ = smem_u32(smem + Layout::kQ);
    const uint32_t sK = smem_u32(smem + Layout::kK);
    const uint32_t sV = smem_u32(smem + Layout::kV);

    if (threadIdx.x == 0) {
        misc[0] = 0;
        mbar_init(&bar[kQFull], 1);
        for (int s = 0; s < 2; ++s) {
            mbar_init(&bar[kKFull0 + s], 3);   // one arrival per loader warp
            mbar_init(&bar[kKEmpty0 + s], 1);
            mbar_init(&bar[kVFull0 + s], 3);
            mbar_init(&bar[kVEmpty0 + s], 1);
            mbar_init(&bar[kSFull0 + s], 1);
        }
        mbar_init(&bar[kPFull], 4);
        mbar_init(&bar[kPVDone], 1);
        mbar_init(&bar[kMmaDone], 1);
        fence_barrier_init();
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if ((warp == 0 || warp == 2 || warp == 3) && nt > 0) {
        // ===================== loaders: Q once (warp 0), then K and V page
        // by page. A tile's page boxes are split over the three loader warps
        // (box b to loader b mod 3), each arriving on the stage barrier with
        // its own byte count: issuing many small boxes is bound by the
        // issuing warp, so three warps issue them three times faster.
        const int li = warp == 0 ? 0 : warp - 1;  // 0, 1, 2
        // K/V tiles are read again by the other query tiles and heads of the
        // same request and KV group: keep them in L2.
        const uint64_t policy = l2_policy_evict_last();
        if (lane == 0 && li == 0) {
            prefetch_tensormap(&q_map);
            prefetch_tensormap(&key_map);
            prefetch_tensormap(&value_map);
            const int qrow = (b * a.H_q + hq) * a.L + row0;
            mbar_arrive_expect_tx(&bar[kQFull], 2u * Layout::kHalf);
            tma_load_2d(smem + Layout::kQ, &q_map, 0, qrow, &bar[kQFull], policy);
            tma_load_2d(smem + Layout::kQ + Layout::kHalf, &q_map, 64, qrow, &bar[kQFull], policy);
        }
        const int box = a.box_rows;
        const int32_t* bt = a.block_table + int64_t(b) * a.max_pages;
        const int my_box = li + 3 * lane;              // this lane's box of a tile
        auto n_boxes = [&](int j) {
            const int key0 = j * kTile;
            return (min(n, key0 + kTile) - key0 + box - 1) / box;
        };
        // Raw block-table entry of this lane's box in tile j (loaded ahead of
        // use, so the load latency overlaps the waits; checked at use).
        // The load is unconditional (index clamped to entry 0 when the box
        // does not exist) so that nothing waits for its result before use.
        auto fetch_page = [&](int j) -> int {
            const bool live = j < nt && my_box < n_boxes(j);
            return bt[live ? (j * kTile + my_box * box) / a.ps : 0];
        };
        auto pool_row = [&](int j, int phys) -> int {
            if (unsigned(phys) >= unsigned(a.num_pages)) {
                atomicOr(a.err, PA_DEVERR_PAGE_ID_BIT);
                phys = 0;
            }
            const int tok = j * kTile + my_box * box;
            return (phys * a.H_kv + hk) * a.ps + (tok - (tok / a.ps) * a.ps);
        };
        // This warp's part of tile j's K (is_v = false) or V.
        auto load = [&](int j, bool is_v, int phys) {
            const int nbox = n_boxes(j);
            const int mine = nbox > li ? (nbox - li + 2) / 3 : 0;  // boxes of this warp
            const int s = j & 1;
            const int full = (is_v ? kVFull0 : kKFull0) + s;
            const int empty = (is_v ? kVEmpty0 : kKEmpty0) + s;
            const bool ok = mbar_wait_warp(&bar[empty], ((j >> 1) & 1) ^ 1u, misc, a.err);
            if (ok) {
                if (lane == 0)
                    mbar_arrive_expect_tx(&bar[full], uint32_t(mine) * box * 128u * 2u);
                __syncwarp();
                if (my_box < nbox) {
                    const int row = pool_row(j, phys);
                    uint8_t* d = smem + (is_v ? Layout::kV : Layout::kK) + s * Layout::kMat +
                                 my_box * box * 128;
                    const CUtensorMap* m = is_v ? &value_map : &key_map;
                    tma_load_2d(d, m, 0, row, &bar[full], policy);
                    tma_load_2d(d + Layout::kHalf, m, 64, row, &bar[full], policy);
                }
            }
            __syncwarp();
        };
        // Order of need: S_j = Q K_j^T is issued before P_{j-1} V_{j-1}, so
        // the loads go K_0, K_1, V_0, K_2, V_1, ...; a K stage is free again
        // as soon as its S is computed, a V stage once its P V is. Page ids
        // are fetched two tiles ahead.
        // Page ids two tiles ahead in a ring of three registers (slot = tile
        // mod 3). The loop is unrolled over the ring so that no pending load
        // result is ever copied (a copy would wait for the load).
        int pg[3];
        pg[0] = fetch_page(0);
        pg[1] = fetch_page(1);
        load(0, false, pg[0]);
        for (int j0 = 0; j0 < nt; j0 += 3) {
#pragma unroll
            for (int u = 0; u < 3; ++u) {
                const int j = j0 + u;
                if (j < nt) {
                    pg[(u + 2) % 3] = fetch_page(j + 2);
                    if (j + 1 < nt)
                        load(j + 1, false, pg[(u + 1) % 3]);
                    load(j, true, pg[u]);
                }
            }
        }
        // No copy may still be landing when the block exits: the last (up to)
        // two stages' phases have completed once they were consumed; wait for
        // them again (bounded) in case a consumer gave up.
        for (int j = max(0, nt - 2); j < nt; ++j) {
            mbar_wait_bounded(&bar[kKFull0 + (j & 1)], (j >> 1) & 1, misc, a.err);
            mbar_wait_bounded(&bar[kVFull0 + (j & 1)], (j >> 1) & 1, misc, a.err);
        }
    } else if (warp == 1 && nt > 0) {
        // ===================== MMA issue (one thread) ======================
        if (lane == 0) {
            const uint32_t idesc_s = idesc_bf16_f32(kTile, kTile, 0);
            const uint32_t idesc_pv = idesc_bf16_f32(kTile, 128, 1);
            // Base descriptors built once; every k-step is one add.
            const uint64_t dq = kmajor_base(sQ);
            const uint64_t dk0 = kmajor_base(sK), dk1 = desc_advance(dk0, Layout::kMat);
            const uint64_t dv0 = mnmajor_base(sV), dv1 = desc_advance(dv0, Layout::kMat);
            bool ok = mbar_wait_bounded(&bar[kQFull], 0, misc, a.err);
            tc_fence_after();
            for (int j = 0; j <= nt && ok; ++j) {
                if (j < nt) {
                    const int s = j & 1;
                    ok = mbar_wait_bounded(&bar[kKFull0 + s], (j >> 1) & 1, misc, a.err);
                    // The buffer S_j overwrites holds P_{j-2} until P_{j-2} V is done.
                    if (ok && j >= 2)
                        ok = mbar_wait_bounded(&bar[kPVDone], (j - 2) & 1, misc, a.err);
                    if (!ok)
                        break;
                    tc_fence_after();
                    const uint32_t d = tmem + (s ? kColS1 : kColS0);
                    const uint64_t db = s ? dk1 : dk0;
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk)
                        tc_mma_bf16(d, desc_advance(dq, kmajor_off(kk)),
                                    desc_advance(db, kmajor_off(kk)), idesc_s, kk > 0);
                    tc_commit(&bar[kSFull0 + s]);
                    tc_commit(&bar[kKEmpty0 + s]);
                }
                if (j >= 1) {
                    const int jp = j - 1;
                    const int sp = jp & 1;
                    ok = mbar_wait_bounded(&bar[kPFull], jp & 1, misc, a.err);
                    if (ok)
                        ok = mbar_wait_bounded(&bar[kVFull0 + sp], (jp >> 1) & 1, misc, a.err);
                    if (!ok)
                        break;
                    tc_fence_after();
                    const uint64_t db = sp ? dv1 : dv0;
                    const uint32_t pcol = tmem + (sp ? kColS1 : kColS0);  // P_jp in TMEM
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk)
                        tc_mma_bf16_ts(tmem + kColO, pcol + 8u * kk, desc_advance(db, mnmajor_off(kk)),
                                       idesc_pv, (jp > 0 || kk > 0) ? 1u : 0u);
                    tc_commit(&bar[kPVDone]);
                    tc_commit(&bar[kVEmpty0 + sp]);
                }
            }
            // Every MMA this thread issued completes before the block ends.
            tc_commit(&bar[kMmaDone]);
            mbar_wait_bounded(&bar[kMmaDone], 0, misc, a.err);
        }
        __syncwarp();
    } else if (warp >= kSoftmaxWarp0) {
        // ===================== softmax: one thread per query row ===========
        const int w4 = warp - kSoftmaxWarp0;
        const int r = w4 * 32 + lane;                 // row of the tile = TMEM lane
        const uint32_t trow = tmem + (uint32_t(w4 * 32) << 16);
        const int i = row0 + r;
        const bool valid = r < rows;
        const int lim = a.causal ? min(n - a.L + i, n - 1) : n - 1;  // last visible key
        float m_used = -INFINITY;
        float l = 0.f;
        const float c = a.scale_log2;
        uint16_t* orow = a.out + ((int64_t(b) * a.H_q + hq) * a.L + i) * 128;

        for (int j = 0; j < nt; ++j) {
            const int sb = j & 1;
            const bool ok = mbar_wait_warp(&bar[kSFull0 + sb], (j >> 1) & 1, misc, a.err);
            tc_fence_after();
            uint32_t sv[128];
#pragma unroll
            for (int q4 = 0; q4 < 4; ++q4)
                tmem_ld32(trow + (sb ? kColS1 : kColS0) + 32u * q4, sv + 32 * q4);
            tmem_wait_ld();
            float* s = reinterpret_cast<float*>(sv);
            const int key0 = j * kTile;
            if (key0 + kTile - 1 > lim) {
#pragma unroll
                for (int k = 0; k < kTile; ++k)
                    if (key0 + k > lim)
                        s[k] = -INFINITY;
            }
            float m8[8];
#pragma unroll
            for (int u = 0; u < 8; ++u)
                m8[u] = s[u];
#pragma unroll
            for (int k = 8; k < kTile; k += 8)
#pragma unroll
                for (int u = 0; u < 8; ++u)
                    m8[u] = fmaxf(m8[u], s[k + u]);
            const float mx = fmaxf(fmaxf(fmaxf(m8[0], m8[1]), fmaxf(m8[2], m8[3])),
                                   fmaxf(fmaxf(m8[4], m8[5]), fmaxf(m8[6], m8[7])));
            const float mxs = mx * c;
            const bool need = mxs > m_used + kRescaleLog2 || (m_used == -INFINITY && mxs > -INFINITY);
            float factor = 1.f;
            if (need) {
                factor = m_used == -INFINITY ? 0.f : fast_exp2(m_used - mxs);
                m_used = mxs;
                l *= factor;
            }
            const float mu = m_used == -INFINITY ? 0.f : m_used;
            uint32_t pk[64];
#pragma unroll
            for (int k = 0; k < 64; ++k) {
                const float p0 = fast_exp2(fmaf(s[2 * k], c, -mu));
                const float p1 = fast_exp2(fmaf(s[2 * k + 1], c, -mu));
                l += p0 + p1;
                pk[k] = pack_bf16x2(p0, p1);
            }
            // P buffer and O are free once the previous P V has completed.
            if (j >= 1)
                mbar_wait_bounded(&bar[kPVDone], (j - 1) & 1, misc, a.err);
            if (j >= 1 && __any_sync(0xffffffffu, need)) {
                tc_fence_after();
#pragma unroll
                for (int q4 = 0; q4 < 4; ++q4) {
                    uint32_t ov[32];
                    tmem_ld32(trow + kColO + 32u * q4, ov);
                    tmem_wait_ld();
#pragma unroll
                    for (int k = 0; k < 32; ++k)
                        ov[k] = __float_as_uint(__uint_as_float(ov[k]) * factor);
                    tmem_st32(trow + kColO + 32u * q4, ov);
                }
                tmem_wait_st();
            }
            // P row r (bf16, two per 32-bit column) over the first 64 columns of
            // this tile's score buffer: the A operand of P V, read from TMEM.
            tmem_st32(trow + (sb ? kColS1 : kColS0), pk);
            tmem_st32(trow + (sb ? kColS1 : kColS0) + 32u, pk + 32);
            tmem_wait_st();
            // V rows past the context hold stale bytes: zero them (P is 0
            // there, but 0 * NaN is not).
            if (n < key0 + kTile) {
                mbar_wait_bounded(&bar[kVFull0 + sb], (j >> 1) & 1, misc, a.err);  // V_j landed
                const int z0 = max(0, n - key0);
                const int nz = (kTile - z0) * 16;   // 16-byte chunks
                uint8_t* vb = smem + Layout::kV + sb * Layout::kMat;
                for (int idx = r; idx < nz; idx += 128) {
                    const int zr = z0 + idx / 16, ch = idx % 16;
                    *reinterpret_cast<uint4*>(vb + (ch >> 3) * Layout::kHalf + zr * 128 +
                                              (((ch & 7) ^ (zr & 7)) << 4)) = make_uint4(0, 0, 0, 0);
                }
            }
            fence_proxy_async_smem();
            tc_fence_before();
            __syncwarp();
            if (lane == 0)
                mbar_arrive(&bar[kPFull]);
            (void)ok;
        }
        // ---- epilogue: O / l -> bf16 --------------------------------------
        const float inv = l > 0.f ? a.out_scale / l : 0.f;
        if (nt > 0) {
            mbar_wait_bounded(&bar[kPVDone], (nt - 1) & 1, misc, a.err);
            tc_fence_after();
        }
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4) {
            uint32_t ov[32];
            if (nt > 0) {
                tmem_ld32(trow + kColO + 32u * q4, ov);
                tmem_wait_ld();
            } else {
#pragma unroll
                for (int k = 0; k < 32; ++k)
                    ov[k] = 0u;
            }
            if (valid && misc[0] == 0) {
#pragma unroll
                for (int k = 0; k < 32; k += 8) {
                    uint4 w;
                    w.x = pack_bf16x2(__uint_as_float(ov[k]) * inv, __uint_as_float(ov[k + 1]) * inv);
                    w.y = pack_bf16x2(__uint_as_float(ov[k + 2]) * inv, __uint_as_float(ov[k + 3]) * inv);
                    w.z = pack_bf16x2(__uint_as_float(ov[k + 4]) * inv, __uint_as_float(ov[k + 5]) * inv);
                    w.w = pack_bf16x2(__uint_as_float(ov[k + 6]) * inv, __uint_as_float(ov[k + 7]) * inv);
                    *reinterpret_cast<uint4*>(orow + 32 * q4 + k) = w;
                }
            }
        }
        tc_fence_before();
    }

    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

}  // namespace

size_t prefill_smem_bytes() { return size_t(Layout::kBytes); }

cudaError_t launch_prefill(const CUtensorMap& q_map, const CUtensorMap& key_map,
                           const CUtensorMap& value_map, const PrefillArgs& a, int device,
                           cudaStream_t stream)
{
    constexpr int kMaxDev = 64;
    static std::atomic<int> smem_set[kMaxDev];
    if (device < 0 || device >= kMaxDev)
        return cudaErrorInvalidDevice;
    const int smem = Layout::kBytes;
    if (smem_set[device].load(std::memory_order_relaxed) < smem) {
        cudaError_t e = cudaFuncSetAttribute(prefill_kernel,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess)
            return e;
        smem_set[device].store(smem, std::memory_order_relaxed);
    }
    const int64_t grid = int64_t(a.B) * a.H_q * a.n_qtiles;
    // Programmatic stream serialization: the blocks may be scheduled while the
    // previous kernel in the stream finishes; each waits for it
    // (griddepcontrol.wait) before reading anything.
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(unsigned(grid));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = size_t(smem);
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const cudaError_t e = cudaLaunchKernelEx(&cfg, prefill_kernel, q_map, key_map, value_map, a);
    return e;
}

}  // namespace pa
