// Causal page-walking prefill attention on the 5th-generation tensor cores,
// with the K/V tiles of all query tiles split evenly over the SMs.
//
// Computes the same as the other prefill kernels: for request b, query head
// h_q and query rows i in [0, L) (absolute position n_b - L + i),
// softmax(scale * q . K^T + causal mask) . V over keys 0..position, K/V
// resolved page by page through block_table (Week 3 Day 4: Direct Paged
// Attention, "Task 2"; the two query heads of a block share every K/V tile,
// the grouped-query schedule of "Checkpoint 2").
//
// Why split: with one block per (request, head pair, 128-row query tile) the
// blocks visit from a few to many K/V tiles (a tile near the end of a long
// prefix sees the most keys), and whole blocks cannot be packed onto the SMs
// evenly: on a chunk of 512 rows after prefixes of 200 to 1800 tokens the
// best greedy packing leaves the SMs a quarter idle at the end. Here every
// (request, head pair, query tile) is an item of nt K/V tiles (one unit per
// tile; an item with no visible key is one unit that writes zeros); the items
// form one stream of U units that a persistent grid of one block per SM cuts
// into equal ranges (block c takes units [c U / G, (c + 1) U / G)). The piece
// of an item inside one block runs exactly as in the pairs kernel. An item
// cut by range boundaries is finished by the block holding its first tiles
// (the end of that block's range); its later pieces lie at the starts of the
// following blocks' ranges, so they are done early and have left their
// unnormalised states (O, running maximum m, running sum l) in the
// workspace. The first block merges them into its own O: M = max m_k,
// l = sum l_k 2^(m_k - M), o = sum O_k 2^(m_k - M) / l (the split-KV
// combination of the pages' decode schedule, "Choose a Schedule for Each
// Query Shape", applied to the long-query tiles), in a fixed order.
//
// Per block (384 threads, as the pairs kernel):
//   * warps 0, 2, 3: TMA loads of the K and V tiles of 128 keys page by page
//     (two K and two V stages, the stream running on across pieces); warps 0
//     and 2 also load head 0's and head 1's Q tile of each piece, into a
//     buffer per head that is free once that head's last S of the piece
//     before has completed. At the start, every piece's Q tiles are
//     prefetched into L2;
//   * warp 1 (one elected thread): the tcgen05.mma chain P_0 V_j, S_0(j + 1),
//     P_1 V_j, S_1(j + 1), across piece boundaries;
//   * warps 4-7 (head 0) and 8-11 (head 1): the online-softmax fold (lazy
//     rescale at 2^8), P written over the upper half of the score columns,
//     and per piece the epilogue (store O / l; or leave the state; or merge).
// TMEM (512 columns): S_0, S_1, O_0, O_1 (128 each).
//
// Workspace (per block c of the grid): the state of c's first piece when the
// item started in an earlier block, per head O as [32 column quads][128
// rows][4 floats] (a warp's stores and loads contiguous) and (m, l) per row;
// and per head and softmax warp one 64-bit flag that holds the launch's stamp
// once that warp's rows are written (so the workspace needs no clearing).
// The wait for a flag is bounded; the launch is cooperative, so every block
// is resident and the wait normally ends at once.
#include <cuda.h>
#include <cuda_bf16.h>
#include <math.h>
#include <stdint.h>
#include <string.h>

#include <atomic>

#include "pa_device.cuh"
#include "pa_internal.h"
#include "pa_tcgen05.cuh"

namespace pa {
namespace {

constexpr int kRows = 128;            // query rows per head and block
constexpr int kKeys = 128;            // keys per K/V tile
constexpr int kThreads = 384;
constexpr int kWarps = kThreads / 32;
constexpr uint32_t kTmemCols = 512;
constexpr float kRescaleLog2 = 8.f;
constexpr int kRegsProducer = 128;
constexpr int kRegsSoftmax = 184;
static_assert(128 * kRegsProducer + 256 * kRegsSoftmax <= 65536, "register split");

__host__ __device__ constexpr uint32_t col_s(int head) { return uint32_t(head * 128); }
__host__ __device__ constexpr uint32_t col_o(int head) { return uint32_t(256 + head * 128); }
constexpr uint32_t kPCol = 64;

struct Layout {
    static constexpr int kHalf = 128 * 128;        // 128 rows x 64 bf16 (128 B)
    static constexpr int kMat = 2 * kHalf;         // 128 x 128 bf16, [half][row][128 B]
    static constexpr int kQ = 0;                   // [head] matrices
    static constexpr int kK = kQ + 2 * kMat;       // 2 stages
    static constexpr int kV = kK + 2 * kMat;       // 2 stages
    static constexpr int kStage = kV + 2 * kMat;   // output staging, 4 KiB per softmax warp
    static constexpr int kStageWarp = 4096;
    static constexpr int kBar = kStage + 8 * kStageWarp;
    static constexpr int kNumBars = 20;
    static constexpr int kTmemSlot = kBar + kNumBars * 8;
    static constexpr int kMisc = kTmemSlot + 16;
    static constexpr int kBytes = kMisc + 16 + 1024;   // + alignment slack
};

// Barrier indices.
constexpr int kQFull = 0;     // + head (2)
constexpr int kQEmpty = 2;    // + head
constexpr int kKFull = 4;     // + stage (2)
constexpr int kKEmpty = 6;    // + stage
constexpr int kVFull = 8;     // + stage
constexpr int kVEmpty = 10;   // + stage
constexpr int kSFull = 12;    // + head (2)
constexpr int kPFull = 14;    // + head
constexpr int kPVDone = 16;   // + head
constexpr int kMmaDone = 18;
static_assert(kMmaDone < Layout::kNumBars, "barrier count");

// Workspace per block: the state of its first piece when that piece belongs
// to an item started by an earlier block.
constexpr int64_t kStateFloats = 2 * 128 * 128;   // [head][32][128][4]
constexpr int64_t kMlEntries = 2 * 128;           // [head][128] float2
constexpr int64_t kFlags = 2 * 4;                 // [head][warp]

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

// K/V tiles visited by query tile t of request b (and its clamped context
// length). Every role of every block evaluates the same function, so all of
// them see the same item stream.
__device__ __forceinline__ int combo_tiles(const SplitPrefillArgs& a, int m, int* n_out)
{
    const int b = m / a.n_qtiles;
    const int t = m - b * a.n_qtiles;
    const int cap = a.max_pages * a.ps;
    int n = a.context_lens[b];
    n = n < 0 ? 0 : (n > cap ? cap : n);
    const int row0 = t * kRows;
    const int rows = min(kRows, a.L - row0);
    const int p_last = n - a.L + row0 + rows - 1;
    int nk = a.causal ? min(n, p_last + 1) : n;
    nk = nk < 0 ? 0 : nk;
    *n_out = n;
    return (nk + kKeys - 1) / kKeys;
}

// Units of the stream: a K/V tile weighs kTileUnits, and an item adds
// kItemUnits ahead of its first tile for what a piece costs besides its
// tiles (its Q tiles, the epilogue, the restart of the chain: about two
// tiles' time, measured per piece on the 512-row batch); an item with no
// visible key weighs kEmptyUnits. A tile belongs to the block whose range
// holds its first unit.
constexpr int kTileUnits = 4;
constexpr int kItemUnits = 8;
constexpr int kEmptyUnits = 1;

__device__ __forceinline__ int64_t item_units(int nt)
{
    return nt > 0 ? int64_t(nt) * kTileUnits + kItemUnits : kEmptyUnits;
}

// Tiles [k0, k1) of an item (first unit us, nt > 0 tiles) whose first units
// lie in [s, e).
__device__ __forceinline__ void tiles_in(int64_t us, int nt, int64_t s, int64_t e, int& k0, int& k1)
{
    auto first_at = [&](int64_t x) -> int {      // first tile starting at or after unit x
        const int64_t d = x - us - kItemUnits;
        if (d <= 0)
            return 0;
        const int64_t k = (d + kTileUnits - 1) / kTileUnits;
        return k > nt ? nt : int(k);
    };
    k0 = first_at(s);
    k1 = first_at(e);
}

// One item's piece inside this block's unit range.
struct Piece {
    int b, t, hp, n;
    int nt;              // K/V tiles of the whole item
    int k0, k1;          // its tiles [k0, k1) run here (may be none)
    int zero;            // 1: an item with no visible key whose unit is here
    int64_t us, ue;      // the item's units [us, ue)
};

// Walks the items that intersect [s, e), in stream order.
struct Cursor {
    int m, hp;
    int64_t us;
    __device__ __forceinline__ bool next(const SplitPrefillArgs& a, int pairs, int64_t s, int64_t e,
                                         Piece& p)
    {
        if (us >= e)
            return false;
        int n;
        const int nt = combo_tiles(a, m, &n);
        p.b = m / a.n_qtiles;
        p.t = m - p.b * a.n_qtiles;
        p.hp = hp;
        p.n = n;
        p.nt = nt;
        p.us = us;
        p.ue = us + item_units(nt);
        if (nt > 0) {
            tiles_in(us, nt, s, e, p.k0, p.k1);
            p.zero = 0;
        } else {
            p.k0 = p.k1 = 0;
            p.zero = us >= s ? 1 : 0;
        }
        us = p.ue;
        if (++hp == pairs) {
            hp = 0;
            ++m;
        }
        return true;
    }
};

// One K/V tile of the block's tile stream (pieces without tiles skipped).
struct TileDesc {
    int b, t, hp, n, k;
    bool first;          // first tile of its piece
    bool last;           // last tile of its piece
    bool valid;
};

struct TileIter {
    Cursor cur;
    Piece p;
    int k;               // next tile of p
    bool have;           // p is loaded
    __device__ __forceinline__ TileDesc next(const SplitPrefillArgs& a, int pairs, int64_t s,
                                             int64_t e)
    {
        TileDesc d;
        d.valid = false;
        for (;;) {
            if (have && k < p.k1) {
                d.b = p.b;
                d.t = p.t;
                d.hp = p.hp;
                d.n = p.n;
                d.k = k;
                d.first = k == p.k0;
                d.last = k + 1 == p.k1;
                d.valid = true;
                ++k;
                return d;
            }
            if (!cur.next(a, pairs, s, e, p))
                return d;
            have = true;
            k = p.k0;
        }
    }
};

// Block c's range starts at unit (c U) / G; the block holding unit x is the
// largest c with c U / G <= x.
__device__ __forceinline__ int64_t range_start(int64_t c, int64_t U, int64_t G) { return c * U / G; }
__device__ __forceinline__ int block_of_unit(int64_t x, int64_t U, int64_t G)
{
    return int(((x + 1) * G - 1) / U);
}

// kOdd: the group size is odd; the last head pair of each group holds its
// last head twice (computed by both softmax warpgroups, written by the
// first only), a separate instantiation so that even groups keep their code.
template <bool kOdd>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_split_kernel(const __grid_constant__ CUtensorMap q_map,
                         const __grid_constant__ CUtensorMap key_map,
                         const __grid_constant__ CUtensorMap value_map, const SplitPrefillArgs a)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* bar = reinterpret_cast<uint64_t*>(smem + Layout::kBar);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + Layout::kTmemSlot);
    volatile int* misc = reinterpret_cast<volatile int*>(smem + Layout::kMisc);
    __shared__ long long warp_sum[kWarps];
    __shared__ long long start_cursor[3];
    __shared__ long long blk_range[3];            // s, e, U of this block
    __shared__ Piece warp_piece[8];               // softmax warps: current piece
    __shared__ Cursor warp_cursor[8];             // softmax warps: next item
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int per_group = kOdd ? (a.G + 1) / 2 : a.G / 2;   // head pairs per KV group
    const int pairs = a.H_kv * per_group;
    // Query head h (0, 1) of head pair hp, and whether hp repeats its head.
    auto head_of = [&](int hp, int h) -> int {
        if constexpr (kOdd) {
            const int hk = hp / per_group;
            const int hq0 = hk * a.G + 2 * (hp - hk * per_group);
            return h == 1 && hq0 + 1 == (hk + 1) * a.G ? hq0 : hq0 + h;
        } else {
            return 2 * hp + h;
        }
    };
    auto repeats = [&](int hp) -> bool {
        if constexpr (kOdd)
            return head_of(hp, 1) == head_of(hp, 0);
        else
            return false;
    };
    const int64_t G = gridDim.x;
    const int c = int(blockIdx.x);

    // ---- this block's range of the unit stream ----------------------------
    // Each thread sums the units of a contiguous run of (request, query tile)
    // combinations; a block-wide exclusive scan gives every run its offset.
    const int M = a.B * a.n_qtiles;
    const int per = (M + kThreads - 1) / kThreads;
    const int m_lo = min(M, int(threadIdx.x) * per);
    const int m_hi = min(M, m_lo + per);
    long long mine = 0;
    for (int m = m_lo; m < m_hi; ++m) {
        int n;
        const int nt = combo_tiles(a, m, &n);
        mine += item_units(nt);
        if (blockIdx.x == 0 && m % a.n_qtiles == 0) {
            const int raw = a.context_lens[m / a.n_qtiles];
            if (raw < 0 || raw > a.max_pages * a.ps)
                atomicOr(a.err, PA_DEVERR_CONTEXT_LEN_BIT);
        }
    }
    long long incl = mine;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const long long v = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o)
            incl += v;
    }
    if (lane == 31)
        warp_sum[warp] = incl;
    if (threadIdx.x == 0) {                       // overwritten by the run holding unit s
        start_cursor[0] = 0;
        start_cursor[1] = 0;
        start_cursor[2] = 0;
    }
    __syncthreads();
    long long before = 0, total = 0;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) {
        before += w < warp ? warp_sum[w] : 0;
        total += warp_sum[w];
    }
    const long long excl = before + incl - mine;   // units of combos before m_lo (per head pair)
    const int64_t U = int64_t(total) * pairs;
    const int64_t s = range_start(c, U, G);
    const int64_t e = range_start(c + 1, U, G);
    if (s < e && excl * pairs <= s && s < (excl + mine) * pairs) {
        long long pre = excl;
        for (int m = m_lo; m < m_hi; ++m) {
            int n;
            const int nt = combo_tiles(a, m, &n);
            const int64_t w = item_units(nt);
            if ((pre + w) * pairs > s) {
                const int64_t hp = (s - pre * pairs) / w;
                start_cursor[0] = m;
                start_cursor[1] = hp;
                start_cursor[2] = pre * pairs + hp * w;
                break;
            }
            pre += w;
        }
    }
    if (s >= e)
        return;                                   // an empty range (the whole block)
    if (threadIdx.x == 0) {
        blk_range[0] = s;
        blk_range[1] = e;
        blk_range[2] = U;
    }
    __syncthreads();
    Cursor start;
    start.m = int(start_cursor[0]);
    start.hp = int(start_cursor[1]);
    start.us = start_cursor[2];

    const uint32_t sQ = smem_u32(smem + Layout::kQ);
    const uint32_t sK = smem_u32(smem + Layout::kK);
    const uint32_t sV = smem_u32(smem + Layout::kV);

    if (threadIdx.x == 0) {
        misc[0] = 0;
        for (int h = 0; h < 2; ++h) {
            mbar_init(&bar[kQFull + h], 1);
            mbar_init(&bar[kQEmpty + h], 1);
        }
        for (int st = 0; st < 2; ++st) {
            mbar_init(&bar[kKFull + st], 3);   // one arrival per loader warp
            mbar_init(&bar[kKEmpty + st], 1);
            mbar_init(&bar[kVFull + st], 3);
            mbar_init(&bar[kVEmpty + st], 1);
        }
        for (int h = 0; h < 2; ++h) {
            mbar_init(&bar[kSFull + h], 1);
            mbar_init(&bar[kPFull + h], 4);   // one arrival per softmax warp
            mbar_init(&bar[kPVDone + h], 1);
        }
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

    // Registers from the loader / MMA warpgroup (warps 0-3) to the two softmax
    // warpgroups, each change at the top of its warpgroup's branch so that the
    // code of the branch is compiled to the new limit.
    if (warp < 4) {
        setmaxnreg_dec<kRegsProducer>();
        if (warp != 1) {
            // ===================== loaders =====================================
            const int li = warp == 0 ? 0 : warp - 1;     // 0, 1, 2
            const uint64_t policy = l2_policy_evict_last();
            if (lane == 0 && li == 0) {
                prefetch_tensormap(&q_map);
                prefetch_tensormap(&key_map);
                prefetch_tensormap(&value_map);
                // Every piece's Q tiles into L2 now, so that a piece boundary
                // waits for an L2 read rather than a DRAM one.
                Cursor pc = start;
                Piece pp;
                while (pc.next(a, pairs, s, e, pp)) {
                    if (pp.k1 > pp.k0) {
                        for (int h = 0; h < 2; ++h) {
                            const int qrow = (pp.b * a.H_q + head_of(pp.hp, h)) * a.L + pp.t * kRows;
                            tma_prefetch_l2_2d(&q_map, 0, qrow);
                            tma_prefetch_l2_2d(&q_map, 64, qrow);
                        }
                    }
                }
            }
            const int box = a.box_rows;                  // min(ps, 128)
            const int my_box = li + 3 * lane;
            TileIter it;
            it.cur = start;
            it.have = false;
            it.k = 0;
            int qp = 0;                                  // pieces whose Q this warp loaded
            auto n_boxes = [&](const TileDesc& d) {
                const int key0 = d.k * kKeys;
                return (min(d.n, key0 + kKeys) - key0 + box - 1) / box;
            };
            auto load_q = [&](const TileDesc& d, int h) {
                // Head h's Q tile of a new piece, once head h's last S of the
                // piece before has completed (loader h only).
                const bool ok = mbar_wait_warp(&bar[kQEmpty + h], (qp & 1) ^ 1u, misc, a.err);
                if (ok && lane == 0) {
                    mbar_arrive_expect_tx(&bar[kQFull + h], uint32_t(Layout::kMat));
                    const int qrow = (d.b * a.H_q + head_of(d.hp, h)) * a.L + d.t * kRows;
                    uint8_t* dst = smem + Layout::kQ + h * Layout::kMat;
                    tma_load_2d(dst, &q_map, 0, qrow, &bar[kQFull + h], policy);
                    tma_load_2d(dst + Layout::kHalf, &q_map, 64, qrow, &bar[kQFull + h], policy);
                }
                __syncwarp();
                ++qp;
            };
            // Order of need: K_g then V_g for every tile g of the block's stream,
            // the Q tiles of a piece around its first K and V. A tile's page ids
            // are loaded just before the wait for its K stage, which hides the
            // load (consecutive tiles' entries share cache lines).
            int n_tiles = 0;
            for (TileDesc d = it.next(a, pairs, s, e); d.valid; d = it.next(a, pairs, s, e)) {
                const int g = n_tiles++;
                // Head 0's Q is needed with the first K, head 1's only after
                // both heads' work on the previous tile: loader 1 issues its K/V
                // boxes before it waits to refill Q_1.
                if (d.first && li == 0)
                    load_q(d, 0);
                const int nbox = n_boxes(d);
                const int mine_boxes = nbox > li ? (nbox - li + 2) / 3 : 0;
                const bool live = my_box < nbox;
                int phys = live ? a.block_table[int64_t(d.b) * a.max_pages + (d.k * kKeys + my_box * box) / a.ps]
                                : 0;
                const int st = g & 1;
    #pragma unroll 1
                for (int is_v = 0; is_v < 2; ++is_v) {
                    const int full = (is_v ? kVFull : kKFull) + st;
                    const int empty = (is_v ? kVEmpty : kKEmpty) + st;
                    const bool ok = mbar_wait_warp(&bar[empty], ((g >> 1) & 1) ^ 1u, misc, a.err);
                    if (ok) {
                        if (lane == 0)
                            mbar_arrive_expect_tx(&bar[full], uint32_t(mine_boxes) * box * 128u * 2u);
                        __syncwarp();
                        if (live) {
                            if (unsigned(phys) >= unsigned(a.num_pages)) {
                                atomicOr(a.err, PA_DEVERR_PAGE_ID_BIT);
                                phys = 0;
                            }
                            const int tok = d.k * kKeys + my_box * box;
                            const int hk = d.hp / per_group;
                            const int row = (phys * a.H_kv + hk) * a.ps + (tok - (tok / a.ps) * a.ps);
                            uint8_t* dst = smem + (is_v ? Layout::kV : Layout::kK) + st * Layout::kMat +
                                           my_box * box * 128;
                            const CUtensorMap* mp = is_v ? &value_map : &key_map;
                            tma_load_2d(dst, mp, 0, row, &bar[full], policy);
                            tma_load_2d(dst + Layout::kHalf, mp, 64, row, &bar[full], policy);
                        }
                    }
                    __syncwarp();
                }
                if (d.first && li == 1)
                    load_q(d, 1);
            }
            // No copy may still be landing when the block exits.
            for (int g = max(0, n_tiles - 2); g < n_tiles; ++g) {
                mbar_wait_bounded(&bar[kKFull + (g & 1)], (g >> 1) & 1, misc, a.err);
                mbar_wait_bounded(&bar[kVFull + (g & 1)], (g >> 1) & 1, misc, a.err);
            }
            if (qp > 0 && li < 2)
                mbar_wait_bounded(&bar[kQFull + li], (qp - 1) & 1, misc, a.err);
        } else {
            // ===================== MMA issue (one elected thread) ==============
            const bool leader = elect_one();
            const uint32_t idesc_s = idesc_bf16_f32(kRows, kKeys, 0);
            const uint32_t idesc_pv = idesc_bf16_f32(kRows, 128, 1);
            const uint64_t dq0 = kmajor_base(sQ), dq1 = desc_advance(dq0, Layout::kMat);
            const uint64_t dk0 = kmajor_base(sK), dk1 = desc_advance(dk0, Layout::kMat);
            const uint64_t dv0 = mnmajor_base(sV), dv1 = desc_advance(dv0, Layout::kMat);
            auto s_mmas = [&](int h, int g) {
                if (leader) {
                    const uint64_t da = h ? dq1 : dq0;
                    const uint64_t db = (g & 1) ? dk1 : dk0;
                    const uint32_t dd = tmem + col_s(h);
    #pragma unroll
                    for (int kk = 0; kk < 8; ++kk)
                        tc_mma_bf16(dd, desc_advance(da, kmajor_off(kk)), desc_advance(db, kmajor_off(kk)),
                                    idesc_s, kk > 0);
                }
                __syncwarp();
            };
            auto pv_mmas = [&](int h, int g, bool first) {
                if (leader) {
                    const uint64_t db = (g & 1) ? dv1 : dv0;
                    const uint32_t dd = tmem + col_o(h);
                    const uint32_t pa = tmem + col_s(h) + kPCol;
    #pragma unroll
                    for (int kk = 0; kk < 8; ++kk)
                        tc_mma_bf16_ts(dd, pa + 8u * kk, desc_advance(db, mnmajor_off(kk)), idesc_pv,
                                       (!first || kk > 0) ? 1u : 0u);
                }
                __syncwarp();
            };
            auto commit = [&](int bi) {
                if (leader)
                    tc_commit(&bar[bi]);
                __syncwarp();
            };
            auto wait = [&](int bi, uint32_t parity) {
                return __all_sync(0xffffffffu, mbar_wait_lean(&bar[bi], parity, misc, a.err));
            };
            TileIter it;
            it.cur = start;
            it.have = false;
            it.k = 0;
            TileDesc cur, nxt;
    #pragma unroll 1
            for (int u = 0; u < 2; ++u) {
                const TileDesc d = it.next(a, pairs, s, e);
                if (u == 0)
                    cur = d;
                else
                    nxt = d;
            }
            int qp = 1;                                  // Q phase of the next new piece
            bool ok = cur.valid;
            if (ok) {
                ok = wait(kQFull, 0) && wait(kKFull, 0);
                if (ok) {
                    tc_fence_after();
                    s_mmas(0, 0);
                    if (cur.last)
                        commit(kQEmpty);
                    commit(kSFull);
                    ok = wait(kQFull + 1, 0);
                }
                if (ok) {
                    tc_fence_after();
                    s_mmas(1, 0);
                    if (cur.last)
                        commit(kQEmpty + 1);
                    ok = wait(kVFull, 0) && (!nxt.valid || wait(kKFull + 1, 0));
                    commit(kSFull + 1);
                    commit(kKEmpty);
                }
            }
            for (int g = 0; ok; ++g) {
                const bool more = nxt.valid;
                // head 0: P_0 V_g, then S_0 for tile g + 1 once P_0 V_g is done
                // (S_0 overwrites P_0); a new piece's S also waits for its Q.
                if (!wait(kPFull, g & 1))
                    break;
                tc_fence_after();
                pv_mmas(0, g, cur.first);
                commit(kPVDone);
                if (!wait(kPVDone, g & 1) || (more && nxt.first && !wait(kQFull, qp & 1)))
                    break;
                tc_fence_after();
                if (more) {
                    s_mmas(0, g + 1);
                    if (nxt.last)
                        commit(kQEmpty);
                }
                ok = wait(kPFull + 1, g & 1);
                if (more)
                    commit(kSFull);
                if (!ok)
                    break;
                // head 1: P_1 V_g, then S_1 for tile g + 1
                tc_fence_after();
                pv_mmas(1, g, cur.first);
                commit(kPVDone + 1);
                commit(kVEmpty + (g & 1));
                if (!wait(kPVDone + 1, g & 1) || !more || (nxt.first && !wait(kQFull + 1, qp & 1)))
                    break;
                if (nxt.first)
                    ++qp;
                const TileDesc nn = it.next(a, pairs, s, e);   // tile g + 2
                tc_fence_after();
                s_mmas(1, g + 1);
                if (nxt.last)
                    commit(kQEmpty + 1);
                // the next tile's V and the tile after's K, before the commit
                ok = wait(kVFull + ((g + 1) & 1), ((g + 1) >> 1) & 1) &&
                     (!nn.valid || wait(kKFull + (g & 1), ((g + 2) >> 1) & 1));
                commit(kSFull + 1);
                commit(kKEmpty + ((g + 1) & 1));
                cur = nxt;
                nxt = nn;
            }
            commit(kMmaDone);
            wait(kMmaDone, 0);
        }
    } else {
        setmaxnreg_inc<kRegsSoftmax>();
        // ===================== softmax: one warpgroup per head =============
        const int head = (warp - 4) >> 2;
        const int w4 = warp & 3;
        const int r = w4 * 32 + lane;
        const uint32_t trow = tmem + (uint32_t(w4 * 32) << 16);
        const uint32_t ts = trow + col_s(head);
        const uint32_t to = trow + col_o(head);
        const float c2l = a.scale_log2;
        // The piece walk lives in shared memory (one slot per warp, read
        // back where needed): the fold below needs every register it has.
        const int w8 = warp - 4;
        volatile Piece* vp = &warp_piece[w8];
        volatile long long* vr = blk_range;
        if (lane == 0)
            warp_cursor[w8] = start;
        __syncwarp();
        // Output rows leave through a per-warp staging buffer, 64 columns at a
        // time: each thread puts its row's 128 bytes in (16-byte chunks
        // swizzled by row), then the warp stores four whole 128-byte row
        // segments per instruction.
        uint8_t* stage = smem + Layout::kStage + w8 * Layout::kStageWarp;
        auto store_half = [&](int hf, const uint32_t* pk, uint16_t* out_warp, int rows_ok) {
#pragma unroll
            for (int cq = 0; cq < 8; ++cq)
                *reinterpret_cast<uint4*>(stage + lane * 128 + ((cq ^ (lane & 7)) << 4)) =
                    make_uint4(pk[4 * cq], pk[4 * cq + 1], pk[4 * cq + 2], pk[4 * cq + 3]);
            __syncwarp();
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const int idx = j * 32 + lane;
                const int row = idx >> 3, cq = idx & 7;
                const uint4 v = *reinterpret_cast<const uint4*>(stage + row * 128 + ((cq ^ (row & 7)) << 4));
                if (row < rows_ok)
                    *reinterpret_cast<uint4*>(out_warp + int64_t(row) * 128 + hf * 64 + cq * 8) = v;
            }
            __syncwarp();
        };
        // A later piece's state is handed over with the fence and the flag
        // one tile later, when its stores have drained.
        bool flag_pending = false;
        auto raise_flag = [&]() {
            __threadfence();
            __syncwarp();
            if (lane == 0)
                st_release_gpu(a.flags + (int64_t(c) * 2 + head) * 4 + w4, a.stamp);
            flag_pending = false;
        };
        int g = 0;                                   // tiles of this block so far
        for (;;) {
            int more = 0;
            if (lane == 0) {
                Cursor cur = warp_cursor[w8];
                Piece pc;
                more = cur.next(a, pairs, vr[0], vr[1], pc) ? 1 : 0;
                warp_piece[w8] = pc;
                warp_cursor[w8] = cur;
            }
            more = __shfl_sync(0xffffffffu, more, 0);
            __syncwarp();
            if (!more)
                break;
            if (vp->k1 <= vp->k0 && !vp->zero)
                continue;                            // none of this item's tiles is here
            const int i = vp->t * kRows + r;
            const int n = vp->n;
            const int lim = a.causal ? min(n - a.L + i, n - 1) : n - 1;
            const int k_first = vp->k0, k_end = vp->k1;
            // The first piece of an item cut at this block's end reads the
            // next block's flag now and tests it at the end, so that the
            // read costs nothing (it is normally long set).
            unsigned long long early_flag = 0;
            if (k_first == 0 && k_end < vp->nt && c + 1 < G)
                early_flag = ld_relaxed_gpu(a.flags + (int64_t(c + 1) * 2 + head) * 4 + w4);
            float m_used = -INFINITY;
            float l = 0.f;
            for (int k = k_first; k < k_end; ++k, ++g) {
                mbar_wait_warp(&bar[kSFull + head], g & 1, misc, a.err);
                tc_fence_after();
                const int key0 = k * kKeys;
                const bool edge = key0 + kKeys - 1 > lim;
                // All 128 scores of the row in registers (four loads, one wait).
                uint32_t sv[128];
                float* sc = reinterpret_cast<float*>(sv);
#pragma unroll
                for (int w = 0; w < 4; ++w)
                    tmem_ld32(ts + 32u * w, sv + 32 * w);
                tmem_wait_ld();
                if (edge) {
#pragma unroll
                    for (int w = 0; w < 4; ++w) {
                        const int nv = lim - (key0 + 32 * w) + 1;
                        const uint32_t vis = nv >= 32 ? 0xffffffffu : nv <= 0 ? 0u : (1u << nv) - 1u;
#pragma unroll
                        for (int kq = 0; kq < 32; ++kq)
                            sc[32 * w + kq] = (vis >> kq) & 1u ? sc[32 * w + kq] : -INFINITY;
                    }
                }
                float m8[8];
#pragma unroll
                for (int u = 0; u < 8; ++u)
                    m8[u] = -INFINITY;
#pragma unroll
                for (int kq = 0; kq < 128; kq += 8)
#pragma unroll
                    for (int u = 0; u < 8; ++u)
                        m8[u] = fmaxf(m8[u], sc[kq + u]);
                const float mx = fmaxf(fmaxf(fmaxf(m8[0], m8[1]), fmaxf(m8[2], m8[3])),
                                       fmaxf(fmaxf(m8[4], m8[5]), fmaxf(m8[6], m8[7])));
                const float mxs = mx * c2l;
                const bool need =
                    mxs > m_used + kRescaleLog2 || (m_used == -INFINITY && mxs > -INFINITY);
                float factor = 1.f;
                if (need) {
                    factor = m_used == -INFINITY ? 0.f : fast_exp2(m_used - mxs);
                    m_used = mxs;
                    l *= factor;
                }
                const float mu = m_used == -INFINITY ? 0.f : m_used;
                const float2 cc = make_float2(c2l, c2l), nmu2 = make_float2(-mu, -mu);
                float2 lsum[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f),
                                  make_float2(0.f, 0.f)};
                auto exp_store = [&](int hf) {
                    uint32_t pk[32];
#pragma unroll
                    for (int kq = 0; kq < 32; ++kq) {
                        const float2 x =
                            __ffma2_rn(make_float2(sc[64 * hf + 2 * kq], sc[64 * hf + 2 * kq + 1]), cc, nmu2);
                        const float2 pp = make_float2(fast_exp2(x.x), fast_exp2(x.y));
                        lsum[kq & 3] = __fadd2_rn(lsum[kq & 3], pp);
                        pk[kq] = pack_bf16x2(pp.x, pp.y);
                    }
                    tmem_st32(ts + kPCol + 32u * hf, pk);
                };
                exp_store(1);
                exp_store(0);
                {
                    const float2 t2 =
                        __fadd2_rn(__fadd2_rn(lsum[0], lsum[1]), __fadd2_rn(lsum[2], lsum[3]));
                    l += t2.x + t2.y;
                }
                // O_h holds the piece's earlier tiles, complete (the commit of
                // S_h for this tile covers them): rescale if the maximum moved.
                if (k > k_first && __any_sync(0xffffffffu, need)) {
#pragma unroll
                    for (int q4 = 0; q4 < 4; ++q4) {
                        uint32_t ov[32];
                        tmem_ld32(to + 32u * q4, ov);
                        tmem_wait_ld();
#pragma unroll
                        for (int kq = 0; kq < 32; ++kq)
                            ov[kq] = __float_as_uint(__uint_as_float(ov[kq]) * factor);
                        tmem_st32(to + 32u * q4, ov);
                    }
                }
                tmem_wait_st();
                // V rows past the context hold stale bytes: zero them before
                // either head's P V.
                if (head == 0 && n < key0 + kKeys) {
                    mbar_wait_bounded(&bar[kVFull + (g & 1)], (g >> 1) & 1, misc, a.err);
                    const int z0 = max(0, n - key0);
                    const int nz = (kKeys - z0) * 16;
                    uint8_t* vb = smem + Layout::kV + (g & 1) * Layout::kMat;
                    for (int idx = r; idx < nz; idx += 128) {
                        const int zr = z0 + idx / 16, ch = idx % 16;
                        *reinterpret_cast<uint4*>(vb + (ch >> 3) * Layout::kHalf + zr * 128 +
                                                  (((ch & 7) ^ (zr & 7)) << 4)) = make_uint4(0, 0, 0, 0);
                    }
                    fence_proxy_async_smem();
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0)
                    mbar_arrive(&bar[kPFull + head]);
                if (flag_pending)
                    raise_flag();
            }
            // ---- epilogue of the piece -----------------------------------
            const bool has_tiles = k_end > k_first;
            if (has_tiles) {
                mbar_wait_warp(&bar[kPVDone + head], (g - 1) & 1, misc, a.err);
                tc_fence_after();
            }
            const int hq = head_of(vp->hp, head);
            const int wrow0 = vp->t * kRows + w4 * 32;            // this warp's first row
            uint16_t* out_warp = a.out + ((int64_t(vp->b) * a.H_q + hq) * a.L + wrow0) * 128;
            const int rows_ok =
                misc[0] == 0 && !(head == 1 && repeats(vp->hp)) ? min(32, a.L - wrow0) : 0;
            const int64_t s = vr[0], e = vr[1], U = vr[2];
            const int64_t p_us = vp->us;
            const int p_nt = vp->nt;
            const bool split = has_tiles && (k_first > 0 || k_end < p_nt);
            if (!split) {
                const float inv = l > 0.f ? a.out_scale / l : 0.f;
#pragma unroll 1
                for (int hf = 0; hf < 2; ++hf) {
                    uint32_t ov[64];
                    if (has_tiles) {
                        tmem_ld32(to + 64u * hf, ov);
                        tmem_ld32(to + 64u * hf + 32u, ov + 32);
                        tmem_wait_ld();
                    } else {
#pragma unroll
                        for (int kq = 0; kq < 64; ++kq)
                            ov[kq] = 0u;
                    }
                    uint32_t pk[32];
#pragma unroll
                    for (int kq = 0; kq < 32; ++kq)
                        pk[kq] = pack_bf16x2(__uint_as_float(ov[2 * kq]) * inv,
                                             __uint_as_float(ov[2 * kq + 1]) * inv);
                    store_half(hf, pk, out_warp, rows_ok);
                }
            } else if (k_first > 0) {
                // A later piece of an item that started in an earlier block:
                // leave the state (O relative to m_used, m_used, l) for the
                // item's first block; the flag follows one tile later.
                float4* st_o = reinterpret_cast<float4*>(a.state + (int64_t(c) * 2 + head) * 128 * 128);
#pragma unroll
                for (int q4 = 0; q4 < 4; ++q4) {
                    uint32_t ov[32];
                    tmem_ld32(to + 32u * q4, ov);
                    tmem_wait_ld();
#pragma unroll
                    for (int qq = 0; qq < 8; ++qq)
                        __stcg(st_o + (q4 * 8 + qq) * 128 + r,
                               make_float4(__uint_as_float(ov[4 * qq]), __uint_as_float(ov[4 * qq + 1]),
                                           __uint_as_float(ov[4 * qq + 2]), __uint_as_float(ov[4 * qq + 3])));
                }
                __stcg(a.state_ml + (int64_t(c) * 2 + head) * 128 + r, make_float2(m_used, l));
                flag_pending = true;
            } else {
                // The item's first piece, cut at this block's end: merge the
                // states of its later pieces (blocks c + 1 .. c_end, each at
                // the start of its range, so normally long done) into O_h.
                // This warp needs only its own 32 rows, written by the same
                // warp index there.
                if (flag_pending)
                    raise_flag();
                const int c_end = block_of_unit(p_us + kItemUnits + int64_t(kTileUnits) * (p_nt - 1), U, G);
                auto live = [&](int cc) {
                    int k0c, k1c;
                    tiles_in(p_us, p_nt, range_start(cc, U, G), range_start(cc + 1, U, G), k0c, k1c);
                    return k0c < k1c;
                };
                bool ready = true;
                int n_live = 0;
                for (int cc = c + 1; cc <= c_end && ready; ++cc) {
                    if (!live(cc))
                        continue;
                    ++n_live;
                    const unsigned long long* f = a.flags + (int64_t(cc) * 2 + head) * 4 + w4;
                    bool got = cc == c + 1 && early_flag == a.stamp;
                    if (!got)
                        got = ld_acquire_gpu(f) == a.stamp;
                    if (!got) {
                        const uint64_t t0 = global_timer_ns();
                        const uint64_t limit = misc[0] ? kShortWaitLimitNs : kWaitLimitNs;
                        for (uint32_t it = 1; !got; ++it) {
                            got = ld_acquire_gpu(f) == a.stamp;
                            if (!got && (it & 15u) == 0 && global_timer_ns() - t0 > limit)
                                break;
                        }
                    }
                    ready = __all_sync(0xffffffffu, got);
                }
                if (!ready) {
                    if (lane == 0 && !misc[0]) {
                        misc[0] = 1;
                        atomicOr(a.err, PA_DEVERR_TIMEOUT_BIT);
                    }
                    __syncwarp();
                }
                __threadfence();
                if (n_live == 1 && live(c + 1)) {
                    // One later piece (the usual case): its (m, l) and the
                    // first two 32-column quarters in one round trip, each
                    // further quarter fetched while the one before is used.
                    const int64_t sl = (int64_t(c + 1) * 2 + head);
                    const float2 ml = __ldcg(a.state_ml + sl * 128 + r);
                    const float4* so = reinterpret_cast<const float4*>(a.state + sl * 128 * 128) + r;
                    float4 va[8], vb[8];
#pragma unroll
                    for (int qq = 0; qq < 8; ++qq) {
                        va[qq] = __ldcg(so + qq * 128);
                        vb[qq] = __ldcg(so + (8 + qq) * 128);
                    }
                    const float mx = fmaxf(m_used, ml.x);
                    const float f_own = m_used == -INFINITY ? 0.f : fast_exp2(m_used - mx);
                    const float f = ml.x == -INFINITY ? 0.f : fast_exp2(ml.x - mx);
                    const float lt = l * f_own + ml.y * f;
                    const float inv = lt > 0.f ? a.out_scale / lt : 0.f;
                    uint32_t pk[32];
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        uint32_t ov[32];
                        tmem_ld32(to + 32u * q, ov);
                        tmem_wait_ld();
                        float4* v = (q & 1) ? vb : va;
#pragma unroll
                        for (int qq = 0; qq < 8; ++qq) {
                            const float o0 = (__uint_as_float(ov[4 * qq]) * f_own + f * v[qq].x) * inv;
                            const float o1 = (__uint_as_float(ov[4 * qq + 1]) * f_own + f * v[qq].y) * inv;
                            const float o2 = (__uint_as_float(ov[4 * qq + 2]) * f_own + f * v[qq].z) * inv;
                            const float o3 = (__uint_as_float(ov[4 * qq + 3]) * f_own + f * v[qq].w) * inv;
                            pk[(q & 1) * 16 + 2 * qq] = pack_bf16x2(o0, o1);
                            pk[(q & 1) * 16 + 2 * qq + 1] = pack_bf16x2(o2, o3);
                        }
                        if (q + 2 < 4) {
#pragma unroll
                            for (int qq = 0; qq < 8; ++qq)
                                v[qq] = __ldcg(so + ((q + 2) * 8 + qq) * 128);
                        }
                        if (q & 1)
                            store_half(q >> 1, pk, out_warp, rows_ok);
                    }
                } else {
                    float mx = m_used;
                    for (int cc = c + 1; cc <= c_end; ++cc)
                        if (live(cc))
                            mx = fmaxf(mx, __ldcg(a.state_ml + (int64_t(cc) * 2 + head) * 128 + r).x);
                    const float f_own = m_used == -INFINITY ? 0.f : fast_exp2(m_used - mx);
                    float lt = l * f_own;
                    for (int cc = c + 1; cc <= c_end; ++cc) {
                        if (!live(cc))
                            continue;
                        const float2 ml = __ldcg(a.state_ml + (int64_t(cc) * 2 + head) * 128 + r);
                        lt += ml.x == -INFINITY ? 0.f : ml.y * fast_exp2(ml.x - mx);
                    }
                    const float inv = lt > 0.f ? a.out_scale / lt : 0.f;
#pragma unroll 1
                    for (int hf = 0; hf < 2; ++hf) {         // 64 columns per pass
                        uint32_t ov[64];
                        tmem_ld32(to + 64u * hf, ov);
                        tmem_ld32(to + 64u * hf + 32u, ov + 32);
                        tmem_wait_ld();
                        float* o = reinterpret_cast<float*>(ov);
#pragma unroll
                        for (int k = 0; k < 64; ++k)
                            o[k] *= f_own;
                        for (int cc = c + 1; cc <= c_end; ++cc) {
                            if (!live(cc))
                                continue;
                            const float2 ml = __ldcg(a.state_ml + (int64_t(cc) * 2 + head) * 128 + r);
                            const float f = ml.x == -INFINITY ? 0.f : fast_exp2(ml.x - mx);
                            const float4* so = reinterpret_cast<const float4*>(
                                                   a.state + (int64_t(cc) * 2 + head) * 128 * 128) +
                                               (hf * 16) * 128 + r;
                            float4 v[16];
#pragma unroll
                            for (int q = 0; q < 16; ++q)
                                v[q] = __ldcg(so + q * 128);
#pragma unroll
                            for (int q = 0; q < 16; ++q) {
                                o[4 * q] += f * v[q].x;
                                o[4 * q + 1] += f * v[q].y;
                                o[4 * q + 2] += f * v[q].z;
                                o[4 * q + 3] += f * v[q].w;
                            }
                        }
                        uint32_t pk[32];
#pragma unroll
                        for (int kq = 0; kq < 32; ++kq)
                            pk[kq] = pack_bf16x2(o[2 * kq] * inv, o[2 * kq + 1] * inv);
                        store_half(hf, pk, out_warp, rows_ok);
                    }
                }
            }
            tc_fence_before();
        }
        if (flag_pending)
            raise_flag();
    }

    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

}  // namespace

size_t prefill_split_smem_bytes() { return size_t(Layout::kBytes); }

size_t prefill_split_workspace_bytes(int grid)
{
    const size_t state = size_t(grid) * size_t(kStateFloats) * sizeof(float);
    const size_t ml = size_t(grid) * size_t(kMlEntries) * 2 * sizeof(float);
    const size_t flags = size_t(grid) * size_t(kFlags) * sizeof(unsigned long long);
    return state + ml + flags + 512;
}

cudaError_t launch_prefill_split(const CUtensorMap& q_map, const CUtensorMap& key_map,
                                 const CUtensorMap& value_map, SplitPrefillArgs a, int grid,
                                 void* workspace, int device, cudaStream_t stream)
{
    constexpr int kMaxDev = 64;
    static std::atomic<int> smem_set[kMaxDev][2];
    static std::atomic<int> regs_ok[kMaxDev][2];
    if (device < 0 || device >= kMaxDev)
        return cudaErrorInvalidDevice;
    const bool odd = a.G % 2 != 0;
    const void* fn = odd ? reinterpret_cast<const void*>(prefill_split_kernel<true>)
                         : reinterpret_cast<const void*>(prefill_split_kernel<false>);
    int rk = regs_ok[device][odd].load(std::memory_order_relaxed);
    if (rk == 0) {
        cudaFuncAttributes fa;
        cudaError_t e = cudaFuncGetAttributes(&fa, fn);
        if (e != cudaSuccess)
            return e;
        const bool fits = fa.numRegs >= kRegsProducer && fa.numRegs <= kRegsSoftmax &&
                          128 * kRegsProducer + 256 * kRegsSoftmax <= kThreads * fa.numRegs;
        rk = fits ? 1 : 2;
        regs_ok[device][odd].store(rk, std::memory_order_relaxed);
    }
    if (rk != 1)
        return cudaErrorNotSupported;
    const int smem = Layout::kBytes;
    if (smem_set[device][odd].load(std::memory_order_relaxed) < smem) {
        cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess)
            return e;
        smem_set[device][odd].store(smem, std::memory_order_relaxed);
    }
    const uint64_t st = next_launch_stamp();
    uint8_t* w = static_cast<uint8_t*>(workspace);
    const size_t state = size_t(grid) * size_t(kStateFloats) * sizeof(float);
    const size_t ml = size_t(grid) * size_t(kMlEntries) * 2 * sizeof(float);
    a.state = reinterpret_cast<float*>(w);
    a.state_ml = reinterpret_cast<float2*>(w + state);
    a.flags = reinterpret_cast<unsigned long long*>(w + state + ml);
    a.stamp = st;
    // A cooperative launch: every block is resident at once (or the launch
    // fails), so a first piece's wait for its later pieces always ends.
    cudaLaunchConfig_t cfg;
    memset(&cfg, 0, sizeof cfg);
    cfg.gridDim = dim3(unsigned(grid));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = size_t(smem);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return odd ? cudaLaunchKernelEx(&cfg, prefill_split_kernel<true>, q_map, key_map, value_map, a)
               : cudaLaunchKernelEx(&cfg, prefill_split_kernel<false>, q_map, key_map, value_map, a);
}

}  // namespace pa
