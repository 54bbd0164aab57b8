// Causal page-walking prefill attention on the 5th-generation tensor cores,
// two query heads of one KV group per block.
//
// Computes the same as the one-head prefill kernel: for request b, query
// head h_q and query rows i in [0, L) (absolute position n_b - L + i),
// softmax(scale * q . K^T + causal mask) . V over keys 0..position, K/V
// resolved page by page through block_table (Week 3 Day 4: Direct Paged
// Attention, "Task 2"; the heads of a KV group share every K/V tile, the
// grouped-query schedule of "Checkpoint 2").
//
// Why two heads: with one 128-row query tile per block, the tensor core
// waits for the softmax of every tile (one warp per SM sub-partition does
// the exponentials of a whole tile). Two heads see exactly the same keys, so
// one K/V tile serves two independent 128-row score tiles, and the MMAs of
// one head run while the other head's softmax works.
//
// Schedule: an item is (request, pair of query heads of one KV group, tile of
// 128 query rows). Items are ranked by the number of K/V tiles they visit,
// most first, and one block per SM takes them in that order as a snake
// (block c takes ranks c, 2G - 1 - c, 2G + c, ...; G blocks), the
// longest-first packing, keeping one pipeline running across its items: the
// next item's Q and K/V tiles load while the current item's last tiles are
// in flight, and its first scores are computed while the softmax warps write
// out the current item.
//   * warps 0, 2, 3 (loaders): per item, the K and V tiles of 128 keys page by
//     page (one box of min(page_size, 128) rows x 64 columns per page and
//     half, the boxes split over the three warps), two K and two V stages
//     released separately and shared by all items; warps 0 and 2 also load
//     head 0's and head 1's Q tile of each item, into a buffer per head that
//     is free once that head's last S of the item before has completed;
//   * warp 1 (one thread): tcgen05.mma kind::f16, M = 128, fp32 accumulate:
//     S_h = Q_h K^T (N = 128 keys; an N = 64 MMA takes as long as N = 128)
//     into head h's score buffer in TMEM, and O_h += P_h V (N = 128 =
//     head_dim) with P_h read from TMEM. An MMA issue returns only about as
//     fast as the tensor core executes it, so every wait of this thread is
//     time the tensor core idles; the order per tile j is P_0 V_j, S_0 for
//     tile j + 1, P_1 V_j, S_1 for tile j + 1, each S committed at once;
//   * warps 4-7 (head 0) and 8-11 (head 1): one thread per query row (TMEM
//     lane), the online-softmax fold with a lazily moved maximum (O and the
//     running sum are rescaled only when a tile's maximum exceeds the one in
//     use by more than 2^8; exponentials of a stale maximum stay below 2^8,
//     so the result is the same softmax). P (bf16, two per 32-bit column) is
//     written over the upper 64 columns of the head's score buffer. V rows
//     past the context are zeroed (by head 0's warps) before either P V. At
//     the end of an item O / l -> bf16, through a staging buffer per warp
//     and a TMA store of each 32-row x 64-column box.
//
// TMEM (512 columns): S_0 [0, 128), S_1 [128, 256), O_0 [256, 384),
// O_1 [384, 512). A score buffer holds P_h(j) until P_h(j) V_j completes;
// S_h(j + 1) is issued only after that completion has been observed, and
// its commit also covers P_h(j) V_j, so a softmax thread that sees S_h(j + 1)
// may rescale O_h without another wait. An item's first P_h V overwrites O_h;
// it is issued after the softmax warps of head h arrive for that tile, which
// they do after writing out the item before.
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

constexpr int kRows = 128;            // query rows per head and block
constexpr int kKeys = 128;            // keys per K/V tile
constexpr int kThreads = 384;
constexpr uint32_t kTmemCols = 512;
constexpr float kRescaleLog2 = 8.f;
constexpr int kRegsProducer = 128;     // per thread, warps 0-3 after the split
constexpr int kRegsSoftmax = 184;     // per thread, warps 4-11 after the split
static_assert(128 * kRegsProducer + 256 * kRegsSoftmax <= 65536, "register split");

__host__ __device__ constexpr uint32_t col_s(int head) { return uint32_t(head * 128); }
__host__ __device__ constexpr uint32_t col_o(int head) { return uint32_t(256 + head * 128); }
constexpr uint32_t kPCol = 64;        // P_h: columns [64, 128) of head h's score buffer

// Items a block can take; the host sizes the grid so that no block gets more.
constexpr int kMaxItems = 32;

// kD: head_dim, 128 or 64 (two or one 64-column halves per matrix row).
template <int kD>
struct Layout {
    static constexpr int kHalf = 128 * 128;        // 128 rows x 64 bf16 (128 B)
    static constexpr int kHalves = kD / 64;
    static constexpr int kMat = kHalves * kHalf;   // 128 x kD bf16, [half][row][128 B]
    static constexpr int kQ = 0;                   // [head] matrices
    static constexpr int kK = kQ + 2 * kMat;       // 2 stages
    static constexpr int kV = kK + 2 * kMat;       // 2 stages
    // output staging, 4 KiB per softmax warp (the item ranking uses it first)
    static constexpr int kStage = kV + 2 * kMat;
    static constexpr int kStageWarp = 4096;
    static constexpr int kItems = kStage + 8 * kStageWarp;   // [kMaxItems][12] int32
    static constexpr int kBar = kItems + kMaxItems * 12 * 4;
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
static_assert(kMmaDone < Layout<128>::kNumBars, "barrier count");

// Item table entry: request, query tile, the two query heads, the KV head,
// the (clamped) context length, K/V tiles run here, whether head 1 repeats
// head 0, the first K/V tile run here, the role (below), the tail piece's
// state slot (its donor block).
enum { kEB = 0, kET, kEH0, kEH1, kEHK, kEN, kENT, kEDup, kEK0, kERole, kESlot, kEntry = 12 };
// Item roles: the whole item here; the item's last tiles here, state left
// for its first block (run first on the receiving block); the item's first
// tiles here, merged at the end with the state its last tiles left.
enum { kWhole = 0, kPublish = 1, kMerge = 2 };

// Tail pieces, with at most two items per block (N items on G blocks, G < N
// <= 2G; the R = 2G - N blocks c < R hold one item): block c >= max(R, G - R)
// hands the last d tiles of its second item (position 2G - 1 - c) to block
// j = G - 1 - c, which runs them before its own item and leaves their state;
// block c merges that state into its own part of the item at the end. Loads in
// quarter tiles: 4 per K/V tile, kWItem per item (its Q, the pipeline restart,
// the epilogue), kWPiece more for a piece that leaves its state, kWMerge for the
// merge. d balances the two blocks: floor((L_c + kWMerge - L_j - kWItem -
// kWPiece) / 8), at most the item's tiles less one, none when below one. The
// weights are measured: on 4 requests of 512 rows after ragged prefixes (the
// busiest blocks at two items of 14 tiles, the idlest at one of 17) they give
// d = 6, 52.6 us per call back to back; d = 4 / 5 / 7 / 8 gave 55.0 / 53.8 /
// 54.5 / 56.5 (with an earlier hand-over that waited for a flag). A merge
// weight of 4 gives the same d there and measured 0.3 us faster than 8 on the
// whole batch (12 and 16: 0.7 and 1.7 us slower).
constexpr int kWItem = 4;
constexpr int kWPiece = 0;
constexpr int kWMerge = 4;

// Operand descriptors (128B swizzle). K-major [half][128 rows][128 B] (Q, K):
// k-step kk (16 elements along K) starts kmajor_off(kk) bytes in. MN-major
// [d half][128 keys][128 B] (V): k-step kk (16 keys) starts 16 rows in.
__host__ __device__ constexpr uint32_t kmajor_off(int kk)
{
    return uint32_t(kk >> 2) * Layout<128>::kHalf + uint32_t(kk & 3) * 32u;
}
__host__ __device__ constexpr uint32_t mnmajor_off(int kk) { return uint32_t(kk) * 16u * 128u; }
__device__ __forceinline__ uint64_t kmajor_base(uint32_t saddr) { return smem_desc_sw128(saddr, 16u, 1024u); }
__device__ __forceinline__ uint64_t mnmajor_base(uint32_t saddr)
{
    return smem_desc_sw128(saddr, uint32_t(Layout<128>::kHalf), 1024u);
}

// This block's part in the tail pieces (kWItem): (tiles it hands over, tiles
// it takes over). order / tiles_of: the ranking of the (request, query tile)
// pairs; item p (rank order) has tiles_of[order[p / pairs]] tiles.
__device__ __forceinline__ int2 plan_piece(const int* order, const int* tiles_of, int pairs, int n_all,
                                        int nblk, int c)
{
    auto size_at = [&](int p) { return tiles_of[order[p / pairs]]; };
    auto donated = [&](int dc) -> int {       // tiles block dc hands over
        const int s2 = size_at(2 * nblk - 1 - dc);
        const int lc = 4 * (size_at(dc) + s2) + 2 * kWItem;
        const int lj = 4 * size_at(nblk - 1 - dc) + kWItem;
        const int d = min((lc + kWMerge - lj - kWItem - kWPiece) / 8, s2 - 1);
        return d > 0 ? d : 0;
    };
    const int R = 2 * nblk - n_all;
    const int c_lo = max(R, nblk - R);
    if (c >= c_lo)
        return make_int2(donated(c), 0);
    if (c < R && nblk - 1 - c >= c_lo)
        return make_int2(0, donated(nblk - 1 - c));
    return make_int2(0, 0);
}

// Block t's load (quarter tiles) with whole items and with the pieces.
__device__ __forceinline__ int2 block_loads(const int* order, const int* tiles_of, int pairs, int n_all,
                                            int nblk, int t)
{
    auto size_at = [&](int p) { return tiles_of[order[p / pairs]]; };
    int before = 4 * size_at(t) + kWItem;
    if (2 * nblk - 1 - t < n_all)
        before += 4 * size_at(2 * nblk - 1 - t) + kWItem;
    const int2 cp = plan_piece(order, tiles_of, pairs, n_all, nblk, t);
    const int after = before - 4 * cp.x + (cp.x > 0 ? kWMerge : 0) +
                      (cp.y > 0 ? 4 * cp.y + kWItem + kWPiece : 0);
    return make_int2(before, after);
}

// This block's (tiles handed over, tiles taken over), the same in every thread
// and every block: only when the pieces lower the busiest block's load by a
// tile or more (with more overloaded blocks than blocks of one item, the ones
// left out keep the makespan and the pieces would only add their costs).
// red: 2 x kThreads / 32 ints of scratch. Called by every thread of the
// block (it synchronises them).
__device__ __forceinline__ int2 plan_tail_pieces(const int* order, const int* tiles_of, int* red, int pairs,
                                              int n_all, int nblk, int c)
{
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    int2 ld = make_int2(0, 0);
    if (int(threadIdx.x) < nblk)
        ld = block_loads(order, tiles_of, pairs, n_all, nblk, int(threadIdx.x));
    const int mb = __reduce_max_sync(0xffffffffu, ld.x), ma = __reduce_max_sync(0xffffffffu, ld.y);
    if (lane == 0) {
        red[warp] = mb;
        red[kThreads / 32 + warp] = ma;
    }
    __syncthreads();
    int max_before = 0, max_after = 0;
#pragma unroll
    for (int w = 0; w < kThreads / 32; ++w) {
        max_before = max(max_before, red[w]);
        max_after = max(max_after, red[kThreads / 32 + w]);
    }
    if (max_after + 4 > max_before)
        return make_int2(0, 0);
    return plan_piece(order, tiles_of, pairs, n_all, nblk, c);
}

// A piece's hand-over needs no wait. Each side of an item cut in two (its
// last tiles, run first by the receiving block; its first tiles, run by the
// donor at its end) arrives once per softmax warp at a word holding the
// launch's stamp and the arrivals so far. The donor normally finds the other
// side arrived and merges that side's state into its own O (in TMEM). If it
// comes first, it leaves its own state and arrives, and the receiving block,
// arriving second, merges the two states from memory. So no block ever waits
// for another, and no launch needs every block resident at once.

// Index of a piece's state: donor slot, part (0: last tiles, 1: first), head.
__device__ __forceinline__ int64_t piece_state(int slot, int part, int head)
{
    return (int64_t(slot) * 2 + part) * 2 + head;
}

// Arrival at a piece's word: the arrivals before this one in this launch (a
// word holding another launch's stamp counts as none). Two parties at most,
// so the loop retries at most a few times.
__device__ __forceinline__ unsigned arrive_piece(unsigned long long* w, uint32_t stamp32)
{
    unsigned long long old = *reinterpret_cast<volatile unsigned long long*>(w);
    for (;;) {
        const bool mine = uint32_t(old >> 32) == stamp32;
        const unsigned long long want =
            (uint64_t(stamp32) << 32) | (mine ? (old & 0xffffffffull) + 1 : 1ull);
        const unsigned long long got = atomicCAS(w, old, want);
        if (got == old)
            return mine ? unsigned(old) : 0u;
        old = got;
    }
}

// The merge of an item's two parts, each held as O / l (bf16) with its (m, l):
// out = w0 (O_0 / l_0) + w1 (O_1 / l_1), w_k = l_k 2^(m_k - M) out_scale / l,
// M = max(m_0, m_1), l = l_0 2^(m_0 - M) + l_1 2^(m_1 - M). Whichever block
// merges computes exactly this, in this order (no contraction), so the output
// bits do not depend on which one it was.
__device__ __forceinline__ float2 merge_weights(float2 ml0, float2 ml1, float out_scale)
{
    const float mx = fmaxf(ml0.x, ml1.x);
    const float f0 = ml0.x == -INFINITY ? 0.f : fast_exp2(ml0.x - mx);
    const float f1 = ml1.x == -INFINITY ? 0.f : fast_exp2(ml1.x - mx);
    const float p0 = __fmul_rn(ml0.y, f0), p1 = __fmul_rn(ml1.y, f1);
    const float lt = __fadd_rn(p0, p1);
    const float inv = lt > 0.f ? __fdiv_rn(out_scale, lt) : 0.f;
    return make_float2(__fmul_rn(p0, inv), __fmul_rn(p1, inv));
}
__device__ __forceinline__ float merge_one(float2 w, float a0, float a1)
{
    return __fmaf_rn(w.y, a1, __fmul_rn(w.x, a0));
}
// O / l as a piece's state holds it (the same rounding on both sides).
__device__ __forceinline__ float piece_inv(float l) { return l > 0.f ? __fdiv_rn(1.f, l) : 0.f; }

// This warp's 32 rows of a piece's O / l -> bf16 [16 chunks of 8 columns][128
// rows] at st (row r = lane already added), (m, l) at ml.
__device__ __forceinline__ void store_piece_state(uint4* st, float2* ml, uint32_t to, bool has_tiles,
                                                  float m_used, float l)
{
    const float inv = piece_inv(l);
#pragma unroll 1
    for (int q4 = 0; q4 < 4; ++q4) {
        uint32_t ov[32];
        if (has_tiles) {
            tmem_ld32(to + 32u * q4, ov);
            tmem_wait_ld();
        } else {
#pragma unroll
            for (int k = 0; k < 32; ++k)
                ov[k] = 0u;
        }
#pragma unroll
        for (int ch = 0; ch < 4; ++ch) {
            const uint32_t* o = ov + 8 * ch;
            __stcg(st + (q4 * 4 + ch) * 128,
                   make_uint4(pack_bf16x2(__uint_as_float(o[0]) * inv, __uint_as_float(o[1]) * inv),
                              pack_bf16x2(__uint_as_float(o[2]) * inv, __uint_as_float(o[3]) * inv),
                              pack_bf16x2(__uint_as_float(o[4]) * inv, __uint_as_float(o[5]) * inv),
                              pack_bf16x2(__uint_as_float(o[6]) * inv, __uint_as_float(o[7]) * inv)));
        }
    }
    __stcg(ml, make_float2(m_used, l));
}

// The receiving block's arrival, one tile after its piece's state was stored
// (the stores have drained by then). If the donor arrived first, this warp
// writes its 32 rows of the item from the two states (rare):
// M = max(m_0, m_1), l = l_0 2^(m_0 - M) + l_1 2^(m_1 - M),
// o = (O_0 / l_0 l_0 2^(m_0 - M) + O_1 / l_1 l_1 2^(m_1 - M)) / l.
__device__ __forceinline__ void piece_arrive_receiver(const uint4* state, const float2* state_ml,
                                                   unsigned long long* arrive, uint64_t stamp, int slot,
                                                   int head, int w4, int lane, uint16_t* out_row,
                                                   bool write, float out_scale)
{
    __threadfence();
    __syncwarp();
    unsigned old = 0;
    if (lane == 0)
        old = arrive_piece(arrive + (int64_t(slot) * 2 + head) * 4 + w4, uint32_t(stamp));
    old = __shfl_sync(0xffffffffu, old, 0);
    if (old == 0)
        return;                                // the donor merges
    __threadfence();                           // the donor's state, stored before its arrival
    __syncwarp();
    const int r = w4 * 32 + lane;
    const int64_t i0 = piece_state(slot, 0, head), i1 = piece_state(slot, 1, head);
    const float2 w = merge_weights(__ldcg(state_ml + i0 * 128 + r), __ldcg(state_ml + i1 * 128 + r),
                                   out_scale);
    const uint4* s0 = state + i0 * 16 * 128 + r;
    const uint4* s1 = state + i1 * 16 * 128 + r;
#pragma unroll 1
    for (int ch = 0; ch < 16; ++ch) {
        const uint4 v0 = __ldcg(s0 + ch * 128), v1 = __ldcg(s1 + ch * 128);
        const uint32_t a0[4] = {v0.x, v0.y, v0.z, v0.w}, a1[4] = {v1.x, v1.y, v1.z, v1.w};
        uint32_t o[4];
#pragma unroll
        for (int k = 0; k < 4; ++k)
            o[k] = pack_bf16x2(merge_one(w, __uint_as_float(a0[k] << 16), __uint_as_float(a1[k] << 16)),
                               merge_one(w, __uint_as_float(a0[k] & 0xffff0000u),
                                         __uint_as_float(a1[k] & 0xffff0000u)));
        if (write)
            *reinterpret_cast<uint4*>(out_row + ch * 8) = make_uint4(o[0], o[1], o[2], o[3]);
    }
}

// kOdd: the group size is odd and the last pair of each group repeats its
// last head (a separate instantiation, so that even groups keep their code).
// kD: head_dim (128, or 64: one 64-column half per Q, K and V row, four
// k-steps for S, N = 64 for P V and 64 of O's TMEM columns). kPieces: the
// tail pieces' planning and epilogues (head_dim 128; a separate instantiation,
// so that the whole-item kernel's code and registers stay as they are: with
// the piece code compiled in, whole items ran 2-3 us per call slower).
// kSmall: pages of fewer than 8 tokens. A TMA box of one page would start
// inside a 128-byte swizzle atom (8 rows), so the loaders copy the K/V rows
// one by one instead (cp.async into the swizzled layout, rows past the
// context zero-filled). Each loader warp waits for its own copies of a stage
// once it has issued the next stage's, fences them to the tensor cores'
// proxy and then arrives.
template <bool kOdd, int kD, bool kPieces, bool kSmall>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_pairs_kernel(const __grid_constant__ CUtensorMap q_map,
                         const __grid_constant__ CUtensorMap key_map,
                         const __grid_constant__ CUtensorMap value_map,
                         const __grid_constant__ CUtensorMap out_map, const PrefillArgs a)
{
    using Layout = pa::Layout<kD>;
    constexpr int kKSteps = kD / 16;                 // k-steps of S = Q K^T
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* bar = reinterpret_cast<uint64_t*>(smem + Layout::kBar);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + Layout::kTmemSlot);
    volatile int* misc = reinterpret_cast<volatile int*>(smem + Layout::kMisc);
    int32_t* items = reinterpret_cast<int32_t*>(smem + Layout::kItems);
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    grid_dependency_wait();  // the previous kernel's outputs are visible from here on

    // ---- this block's items ---------------------------------------------------
    // Items in rank order: the (request, query tile) pairs sorted by the number
    // of K/V tiles they visit, most first, then the head pairs of each. Every
    // block ranks all pairs itself (one thread per pair) when there are at most
    // kThreads of them; beyond that, query tiles are taken last to first.
    // Head pairs: ceil(G / 2) per KV group; with an odd group size the last
    // pair of each group holds its last head twice (computed by both softmax
    // warpgroups, written by the first only). Block c takes the items of rank
    // c, 2G - 1 - c, 2G + c, 4G - 1 - c, ... (G blocks).
    const int per_group = kOdd ? (a.G + 1) / 2 : a.G / 2;
    const int pairs = a.H_kv * per_group;
    const int cap = a.max_pages * a.ps;
    const int M = a.B * a.n_qtiles;
    const int64_t n_all = int64_t(M) * pairs;
    const int64_t nblk = gridDim.x, c = blockIdx.x;
    auto item_at = [&](int k) -> int64_t {   // k-th item of this block
        const int64_t w = k >> 1;
        return (k & 1) ? (2 * w + 2) * nblk - 1 - c : 2 * w * nblk + c;
    };
    int n_own = 0;
    while (n_own < kMaxItems - 1 && item_at(n_own) < n_all)
        ++n_own;
    // Context length of request bb (clamped; an entry out of range is
    // recorded) and the K/V tiles its query tile tt visits.
    auto tiles_for = [&](int bb, int tt, int* n_out) {
        int nn = a.context_lens[bb];
        if (nn < 0 || nn > cap)
            atomicOr(a.err, PA_DEVERR_CONTEXT_LEN_BIT);
        nn = nn < 0 ? 0 : (nn > cap ? cap : nn);
        const int r0 = tt * kRows;
        const int pl = nn - a.L + r0 + min(kRows, a.L - r0) - 1;
        int nk = a.causal ? min(nn, pl + 1) : nn;
        nk = nk < 0 ? 0 : nk;
        *n_out = nn;
        return (nk + kKeys - 1) / kKeys;
    };
    // scratch until the epilogues: the ranking, and the tiles and context
    // length of each (request, query tile) pair
    int* order = reinterpret_cast<int*>(smem + Layout::kStage);
    int* tiles_of = order + kThreads;
    int* n_of = tiles_of + kThreads;
    if (M <= kThreads) {
        const int m = threadIdx.x;
        if (m < M)
            tiles_of[m] = tiles_for(m / a.n_qtiles, m % a.n_qtiles, &n_of[m]);
        __syncthreads();
        if (m < M) {
            const int w = tiles_of[m];
            int rk = 0;
            for (int k = 0; k < M; ++k) {
                const int wk = tiles_of[k];
                rk += (wk > w || (wk == w && k < m)) ? 1 : 0;
            }
            order[rk] = m;
        }
        __syncthreads();
    }
    // Tail pieces (kWItem): with the state buffers, the ranking in shared
    // memory and between one and two items per block.
    const bool pieces =
        kPieces && kD == 128 && a.state != nullptr && M <= kThreads && n_all > nblk && n_all <= 2 * nblk;
    int my_cut = 0, my_piece = 0;             // tiles handed over / taken over
    if (pieces) {
        const int2 cp = plan_tail_pieces(order, tiles_of, n_of + kThreads, pairs, int(n_all), int(nblk),
                                         int(c));
        my_cut = cp.x;
        my_piece = cp.y;
    }
    const int n_items = n_own + (my_piece > 0 ? 1 : 0);
    if (int(threadIdx.x) < n_items) {
        // entry 0 of a receiving block is the piece (the donor's second item);
        // the last one under the test setting that makes the donors finish
        // first
        const int slot = my_piece > 0 ? int(nblk) - 1 - int(c) : int(c);
        const int pe = a.piece_last ? n_items - 1 : 0;    // the piece's entry
        const int own = my_piece > 0 ? (int(threadIdx.x) == pe ? -1 : int(threadIdx.x) - (pe == 0 ? 1 : 0))
                                     : int(threadIdx.x);
        const int64_t i = own < 0 ? nblk + c : item_at(own);
        const int rank = int(i / pairs);
        const int hp = int(i - int64_t(rank) * pairs);
        int b, t, n, nt;
        if (M <= kThreads) {
            const int combo = order[rank];
            b = combo / a.n_qtiles;
            t = combo - b * a.n_qtiles;
            n = n_of[combo];
            nt = tiles_of[combo];
        } else {
            t = a.n_qtiles - 1 - rank / a.B;
            b = rank - (rank / a.B) * a.B;
            nt = tiles_for(b, t, &n);
        }
        int hk, hq0;
        if constexpr (kOdd) {
            hk = hp / per_group;
            hq0 = hk * a.G + 2 * (hp - hk * per_group);
        } else {
            hq0 = 2 * hp;
            hk = hq0 / a.G;
        }
        const bool dup = kOdd && hq0 + 1 == (hk + 1) * a.G;   // odd group: one head, twice
        int32_t* e = items + threadIdx.x * kEntry;
        e[kEB] = b;
        e[kET] = t;
        e[kEH0] = hq0;
        e[kEH1] = dup ? hq0 : hq0 + 1;
        e[kEHK] = hk;
        e[kEN] = n;
        e[kEDup] = dup ? 1 : 0;
        e[kESlot] = slot;
        if (own < 0) {                        // the piece: the last my_piece tiles
            e[kEK0] = nt - my_piece;
            e[kENT] = my_piece;
            e[kERole] = kPublish;
        } else if (own == 1 && my_cut > 0) {  // the first tiles of the second item
            e[kEK0] = 0;
            e[kENT] = nt - my_cut;
            e[kERole] = kMerge;
        } else {
            e[kEK0] = 0;
            e[kENT] = nt;
            e[kERole] = kWhole;
        }
    }

    const uint32_t sQ = smem_u32(smem + Layout::kQ);
    const uint32_t sK = smem_u32(smem + Layout::kK);
    const uint32_t sV = smem_u32(smem + Layout::kV);

    if (threadIdx.x == 0) {
        misc[0] = 0;
        for (int h = 0; h < 2; ++h) {
            mbar_init(&bar[kQFull + h], 1);
            mbar_init(&bar[kQEmpty + h], 1);
        }
        for (int s = 0; s < 2; ++s) {
            mbar_init(&bar[kKFull + s], 3);   // one arrival per loader warp
            mbar_init(&bar[kKEmpty + s], 1);
            mbar_init(&bar[kVFull + s], 3);
            mbar_init(&bar[kVEmpty + s], 1);
        }
        for (int h = 0; h < 2; ++h) {
            mbar_init(&bar[kSFull + h], 1);
            mbar_init(&bar[kPFull + h], 4);   // one arrival per softmax warp
            mbar_init(&bar[kPVDone + h], 1);
        }
        mbar_init(&bar[kMmaDone], 1);
        fence_barrier_init();
        prefetch_tensormap(&q_map);
        prefetch_tensormap(&key_map);
        prefetch_tensormap(&value_map);
        prefetch_tensormap(&out_map);
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    // The Q tiles of the block's first item with K/V tiles go out now, while
    // the loaders still fetch its first page ids (the loaders load every later
    // item's Q).
    if (threadIdx.x == 0) {
        int it0 = 0;
        while (it0 < n_items && items[it0 * kEntry + kENT] == 0)
            ++it0;
        if (it0 < n_items) {
            const int32_t* e = items + it0 * kEntry;
            const uint64_t policy = l2_policy_evict_last();
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                mbar_arrive_expect_tx(&bar[kQFull + h], uint32_t(Layout::kMat));
                const int qrow = (e[kEB] * a.H_q + e[h == 0 ? kEH0 : kEH1]) * a.L + e[kET] * kRows;
                uint8_t* d = smem + Layout::kQ + h * Layout::kMat;
                tma_load_2d(d, &q_map, 0, qrow, &bar[kQFull + h], policy);
                if constexpr (kD == 128)
                    tma_load_2d(d + Layout::kHalf, &q_map, 64, qrow, &bar[kQFull + h], policy);
            }
        }
    }
    // Registers from the loader / MMA warpgroup (warps 0-3) to the two softmax
    // warpgroups: 128 x kRegsProducer + 256 x kRegsSoftmax <= 384 x the launch
    // count (checked on the host before every launch). Each change sits at the
    // top of its warpgroup's branch, so that the branch is compiled to it.
    if (warp < 4) {
        setmaxnreg_dec<kRegsProducer>();
        if (warp != 1) {
            // ===================== loaders =====================================
            // Box k of a tile goes to loader k mod 3; each loader arrives on the
            // stage barrier with its own byte count. Loader h < 2 also loads
            // head h's Q tile of each item.
            const int li = warp == 0 ? 0 : warp - 1;     // 0, 1, 2
            // K/V tiles are read again by the other query tiles and head pairs
            // of the same request and KV group: keep them in L2.
            const uint64_t policy = l2_policy_evict_last();
            const int box = a.box_rows;                  // min(ps, 128)
            const int my_box = li + 3 * lane;
            int g = 0;                                   // tiles of the block before this item
            int qk = 0;                                  // items with tiles before this one
            int pend_full = -1;                          // pages under 8 tokens: the stage whose
            bool pend_ok = false;                        // copies are pending (its full barrier)
            for (int it = 0; it < n_items; ++it) {
                const int32_t* e = items + it * kEntry;
                const int nt = e[kENT], k0 = e[kEK0];
                if (nt == 0)
                    continue;
                const int b = e[kEB], n = e[kEN], hk = e[kEHK];
                const int32_t* bt = a.block_table + int64_t(b) * a.max_pages;
                // tile j of the piece is the item's K/V tile k0 + j
                auto n_boxes = [&](int j) {
                    const int key0 = (k0 + j) * kKeys;
                    return (min(n, key0 + kKeys) - key0 + box - 1) / box;
                };
                // Raw block-table entry of this lane's box in tile j, loaded
                // ahead of use and checked at use (entry 0 when the box does
                // not exist, so that nothing waits for it before use).
                auto fetch_page = [&](int j) -> int {
                    const bool live = j < nt && my_box < n_boxes(j);
                    return bt[live ? ((k0 + j) * kKeys + my_box * box) / a.ps : 0];
                };
                auto pool_row = [&](int j, int phys) -> int {
                    if (unsigned(phys) >= unsigned(a.num_pages)) {
                        atomicOr(a.err, PA_DEVERR_PAGE_ID_BIT);
                        phys = 0;
                    }
                    const int tok = (k0 + j) * kKeys + my_box * box;
                    return (phys * a.H_kv + hk) * a.ps + (tok - (tok / a.ps) * a.ps);
                };
                // Pages of fewer than 8 tokens: row r of tile j (row r of
                // each 64-column half at r * 128 bytes, its 16-byte chunk c at
                // chunk c ^ (r mod 8), the 128-byte swizzle) from its page.
                // One stage's copies stay pending while the next stage's are
                // issued; then the pending stage is waited for, fenced and
                // arrived at. (Its consumer comes after the next stage's
                // empty barrier in the MMA order: K_j after the P V that frees
                // V_j, V_j after the S that frees K_j+1.)
                auto land_pending = [&](bool keep_one) {
                    if (keep_one)
                        cp_async_wait_group<1>();
                    else
                        cp_async_wait_group<0>();
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (pend_ok && lane == 0)
                        mbar_arrive_expect_tx(&bar[pend_full], 0u);
                    __syncwarp();
                    pend_full = -1;
                };
                auto load_rows = [&](int j, bool is_v) {
                    const int gj = g + j;
                    const int s = gj & 1;
                    const int full = (is_v ? kVFull : kKFull) + s;
                    const int empty = (is_v ? kVEmpty : kKEmpty) + s;
                    const bool ok = mbar_wait_warp(&bar[empty], ((gj >> 1) & 1) ^ 1u, misc, a.err);
                    if (ok) {
                        const int key0 = (k0 + j) * kKeys;
                        uint8_t* dst = smem + (is_v ? Layout::kV : Layout::kK) + s * Layout::kMat;
                        const uint16_t* pool = is_v ? a.value_pages : a.key_pages;
                        for (int r = li * 32 + lane; r < kKeys; r += 96) {
                            const int key = key0 + r;
                            const bool live = key < n;
                            int64_t row = 0;
                            if (live) {
                                int phys = bt[key / a.ps];
                                if (unsigned(phys) >= unsigned(a.num_pages)) {
                                    atomicOr(a.err, PA_DEVERR_PAGE_ID_BIT);
                                    phys = 0;
                                }
                                row = (int64_t(phys) * a.H_kv + hk) * a.ps + (key - (key / a.ps) * a.ps);
                            }
                            const uint8_t* src = reinterpret_cast<const uint8_t*>(pool + row * kD);
                            uint8_t* drow = dst + r * 128;
#pragma unroll
                            for (int h = 0; h < Layout::kHalves; ++h)
#pragma unroll
                                for (int c = 0; c < 8; ++c)
                                    cp_async_16(drow + h * Layout::kHalf + ((c ^ (r & 7)) << 4),
                                                src + h * 128 + c * 16, live ? 16u : 0u);
                        }
                    }
                    cp_async_commit();
                    if (pend_full >= 0)
                        land_pending(true);
                    pend_full = full;
                    pend_ok = ok;
                };
                auto load = [&](int j, bool is_v, int phys) {
                    const int nbox = n_boxes(j);
                    const int mine = nbox > li ? (nbox - li + 2) / 3 : 0;
                    const int gj = g + j;
                    const int s = gj & 1;
                    const int full = (is_v ? kVFull : kKFull) + s;
                    const int empty = (is_v ? kVEmpty : kKEmpty) + s;
                    const bool ok = mbar_wait_warp(&bar[empty], ((gj >> 1) & 1) ^ 1u, misc, a.err);
                    if (ok) {
                        if (lane == 0)
                            mbar_arrive_expect_tx(&bar[full], uint32_t(mine) * box * 128u * Layout::kHalves);
                        __syncwarp();
                        if (my_box < nbox) {
                            const int row = pool_row(j, phys);
                            uint8_t* d = smem + (is_v ? Layout::kV : Layout::kK) + s * Layout::kMat +
                                         my_box * box * 128;
                            const CUtensorMap* m = is_v ? &value_map : &key_map;
                            tma_load_2d(d, m, 0, row, &bar[full], policy);
                            if constexpr (kD == 128)
                                tma_load_2d(d + Layout::kHalf, m, 64, row, &bar[full], policy);
                        }
                    }
                    __syncwarp();
                };
                // Order of need: K_0 (its stage frees early), then this head's
                // Q (free once the item before has issued its last S), then
                // V_0, K_1, V_1, ... Page ids are fetched two tiles ahead in a
                // ring of three registers, the loop unrolled over the ring so
                // that no pending load result is ever copied.
                auto load_q = [&]() {
                    const bool ok = mbar_wait_warp(&bar[kQEmpty + li], (qk & 1) ^ 1u, misc, a.err);
                    if (ok && lane == 0) {
                        mbar_arrive_expect_tx(&bar[kQFull + li], uint32_t(Layout::kMat));
                        const int qrow = (b * a.H_q + e[li == 0 ? kEH0 : kEH1]) * a.L + e[kET] * kRows;
                        uint8_t* d = smem + Layout::kQ + li * Layout::kMat;
                        tma_load_2d(d, &q_map, 0, qrow, &bar[kQFull + li], policy);
                        if constexpr (kD == 128)
                            tma_load_2d(d + Layout::kHalf, &q_map, 64, qrow, &bar[kQFull + li], policy);
                    }
                    __syncwarp();
                };
                if constexpr (kSmall) {
                    load_rows(0, false);
                    if (li < 2 && qk > 0)    // the first item's Q went out at the start
                        load_q();
                    for (int j = 0; j < nt; ++j) {
                        load_rows(j, true);
                        if (j + 1 < nt)
                            load_rows(j + 1, false);
                    }
                    land_pending(false);
                } else {
                    int pg[3];
                    pg[0] = fetch_page(0);
                    pg[1] = fetch_page(1);
                    load(0, false, pg[0]);
                    if (li < 2 && qk > 0)    // the first item's Q went out at the start
                        load_q();
                    for (int j0 = 0; j0 < nt; j0 += 3) {
#pragma unroll
                        for (int u = 0; u < 3; ++u) {
                            const int j = j0 + u;
                            if (j < nt) {
                                pg[(u + 2) % 3] = fetch_page(j + 2);
                                load(j, true, pg[u]);
                                if (j + 1 < nt)
                                    load(j + 1, false, pg[(u + 1) % 3]);
                            }
                        }
                    }
                }
                g += nt;
                ++qk;
            }
            // No copy may still be landing when the block exits: wait (bounded)
            // for the last two stages of both streams and the last Q.
            for (int gj = max(0, g - 2); gj < g; ++gj) {
                mbar_wait_bounded(&bar[kKFull + (gj & 1)], (gj >> 1) & 1, misc, a.err);
                mbar_wait_bounded(&bar[kVFull + (gj & 1)], (gj >> 1) & 1, misc, a.err);
            }
            if (li < 2 && qk > 0)
                mbar_wait_bounded(&bar[kQFull + li], (qk - 1) & 1, misc, a.err);
        } else {
            // ===================== MMA issue (one elected thread) ==============
            // The whole warp runs the loop (waits are warp-uniform, which costs
            // less than branches in a lone lane); one elected lane issues. The
            // first wait after a tcgen05.commit costs about 0.1 us even on a
            // completed phase, so the waits that are normally already satisfied
            // (the next K and V tiles) are taken after the commits of a tile.
            const bool leader = elect_one();
            const uint32_t idesc_s = idesc_bf16_f32(kRows, kKeys, 0);
            const uint32_t idesc_pv = idesc_bf16_f32(kRows, kD, 1);
            // Base descriptors built once; every k-step is one add.
            const uint64_t dq0 = kmajor_base(sQ), dq1 = desc_advance(dq0, Layout::kMat);
            const uint64_t dk0 = kmajor_base(sK), dk1 = desc_advance(dk0, Layout::kMat);
            const uint64_t dv0 = mnmajor_base(sV), dv1 = desc_advance(dv0, Layout::kMat);
            auto s_mmas = [&](int h, int gj) {
                if (leader) {
                    const uint64_t da = h ? dq1 : dq0;
                    const uint64_t db = (gj & 1) ? dk1 : dk0;
                    const uint32_t d = tmem + col_s(h);
#pragma unroll
                    for (int kk = 0; kk < kKSteps; ++kk)
                        tc_mma_bf16(d, desc_advance(da, kmajor_off(kk)), desc_advance(db, kmajor_off(kk)),
                                    idesc_s, kk > 0);
                }
                __syncwarp();
            };
            auto pv_mmas = [&](int h, int gj, bool first) {
                if (leader) {
                    const uint64_t db = (gj & 1) ? dv1 : dv0;
                    const uint32_t d = tmem + col_o(h);
                    const uint32_t pa = tmem + col_s(h) + kPCol;
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk)
                        tc_mma_bf16_ts(d, pa + 8u * kk, desc_advance(db, mnmajor_off(kk)), idesc_pv,
                                       (!first || kk > 0) ? 1u : 0u);
                }
                __syncwarp();
            };
            auto commit = [&](int b) {
                if (leader)
                    tc_commit(&bar[b]);
                __syncwarp();
            };
            auto wait = [&](int b, uint32_t parity) {
                return __all_sync(0xffffffffu, mbar_wait_lean(&bar[b], parity, misc, a.err));
            };
            int g = 0, qk = 0;
            bool ok = true;
            for (int it = 0; it < n_items && ok; ++it) {
                const int nt = items[it * kEntry + kENT];
                if (nt == 0)
                    continue;
                // The item's first scores: both score buffers are free (the
                // last P_h V of the item before was waited for).
                ok = wait(kQFull, qk & 1) && wait(kKFull + (g & 1), (g >> 1) & 1);
                if (!ok)
                    break;
                tc_fence_after();
                s_mmas(0, g);
                if (nt == 1)
                    commit(kQEmpty);
                commit(kSFull);
                if (!(ok = wait(kQFull + 1, qk & 1)))
                    break;
                tc_fence_after();
                s_mmas(1, g);
                if (nt == 1)
                    commit(kQEmpty + 1);
                commit(kSFull + 1);
                commit(kKEmpty + (g & 1));
                ok = wait(kVFull + (g & 1), (g >> 1) & 1) &&
                     (nt < 2 || wait(kKFull + ((g + 1) & 1), ((g + 1) >> 1) & 1));
                for (int j = 0; j < nt && ok; ++j) {
                    const int gj = g + j;
                    const bool more = j + 1 < nt;
                    const bool last_s = j + 2 == nt;   // S for tile j + 1 is the item's last
                    // head 0: P_0 V_j, then S_0 for tile j + 1 once P_0 V_j is
                    // done (S_0 overwrites P_0)
                    if (!(ok = wait(kPFull, gj & 1)))
                        break;
                    tc_fence_after();
                    pv_mmas(0, gj, j == 0);
                    commit(kPVDone);
                    if (!(ok = wait(kPVDone, gj & 1)))
                        break;
                    tc_fence_after();
                    if (more) {
                        s_mmas(0, gj + 1);
                        if (last_s)
                            commit(kQEmpty);
                        commit(kSFull);
                    }
                    if (!(ok = wait(kPFull + 1, gj & 1)))
                        break;
                    // head 1: P_1 V_j, then S_1 for tile j + 1
                    tc_fence_after();
                    pv_mmas(1, gj, j == 0);
                    commit(kPVDone + 1);
                    commit(kVEmpty + (gj & 1));
                    if (!(ok = wait(kPVDone + 1, gj & 1)))
                        break;
                    if (more) {
                        tc_fence_after();
                        s_mmas(1, gj + 1);
                        if (last_s)
                            commit(kQEmpty + 1);
                        commit(kSFull + 1);
                        commit(kKEmpty + ((gj + 1) & 1));
                        // the next tile's V and the tile after's K
                        ok = wait(kVFull + ((gj + 1) & 1), ((gj + 1) >> 1) & 1) &&
                             (j + 2 >= nt || wait(kKFull + (gj & 1), ((gj + 2) >> 1) & 1));
                    }
                }
                g += nt;
                ++qk;
            }
            // Every MMA issued completes before the block ends.
            commit(kMmaDone);
            wait(kMmaDone, 0);
        }
    } else {
        setmaxnreg_inc<kRegsSoftmax>();
        // ===================== softmax: one warpgroup per head =============
        const int head = (warp - 4) >> 2;            // 0: warps 4-7, 1: warps 8-11
        const int w4 = warp & 3;                     // TMEM lane quarter of this warp
        const int r = w4 * 32 + lane;                // query row of the tile
        const uint32_t trow = tmem + (uint32_t(w4 * 32) << 16);
        const uint32_t ts = trow + col_s(head);
        const uint32_t to = trow + col_o(head);
        const float c = a.scale_log2;
        // Output rows go through a 4 KiB staging buffer per warp, 16-byte
        // chunks swizzled by row as the output map's 128-byte swizzle wants;
        // one lane then stores the warp's 32 rows x 64 columns by TMA.
        uint8_t* stage = smem + Layout::kStage + (warp - 4) * Layout::kStageWarp;
        int pend_it = -1;                            // a published piece whose arrival is due
        // the receiving block's arrival for the piece of item pend_it (rows
        // of this warp); writes them too if the donor came first
        auto arrive_pending = [&]() {
            const int32_t* pe = items + pend_it * kEntry;
            const int prow0 = pe[kET] * kRows;
            const bool pwrite = prow0 + r < a.L && misc[0] == 0 && !(head == 1 && pe[kEDup]);
            uint16_t* out_row =
                a.out + ((int64_t(pe[kEB]) * a.H_q + pe[head == 0 ? kEH0 : kEH1]) * a.L + prow0 + r) * 128;
            piece_arrive_receiver(a.state, a.state_ml, a.arrive, a.stamp, pe[kESlot], head, w4, lane,
                                  out_row, pwrite, a.out_scale);
            pend_it = -1;
        };
        int g = 0;                                   // tiles of the block before this item
        for (int it = 0; it < n_items; ++it) {
            const int32_t* e = items + it * kEntry;
            const int nt = e[kENT], n = e[kEN], k0 = e[kEK0], role = e[kERole];
            const int row0 = e[kET] * kRows;
            const int rows = min(kRows, a.L - row0);
            const int i = row0 + r;
            const int lim = a.causal ? min(n - a.L + i, n - 1) : n - 1;  // last visible key
            float m_used = -INFINITY;
            float l = 0.f;

            for (int j = 0; j < nt; ++j) {
                const int gj = g + j;
                mbar_wait_warp(&bar[kSFull + head], gj & 1, misc, a.err);
                tc_fence_after();
                // All 128 scores of the row in registers (four loads, one wait),
                // their maximum, then P of keys 64..127 over columns 96..127 and
                // of keys 0..63 over columns 64..95 (every score is read before
                // P overwrites any). Reading the two 64-column halves one after
                // the other, the lower half twice, was 0.9 us per call slower on
                // the 512-row batch.
                const int key0 = (k0 + j) * kKeys;
                const bool edge = key0 + kKeys - 1 > lim;
                uint32_t sv[128];
                float* s = reinterpret_cast<float*>(sv);
#pragma unroll
                for (int w = 0; w < 4; ++w)
                    tmem_ld32(ts + 32u * w, sv + 32 * w);
                tmem_wait_ld();
                if (edge) {
                    // Keys past this row's last visible key -> -inf (by select).
#pragma unroll
                    for (int w = 0; w < 4; ++w) {
                        const int nv = lim - (key0 + 32 * w) + 1;   // visible keys
                        const uint32_t vis = nv >= 32 ? 0xffffffffu : nv <= 0 ? 0u : (1u << nv) - 1u;
#pragma unroll
                        for (int k = 0; k < 32; ++k)
                            s[32 * w + k] = (vis >> k) & 1u ? s[32 * w + k] : -INFINITY;
                    }
                }
                float m8[8];
#pragma unroll
                for (int u = 0; u < 8; ++u)
                    m8[u] = -INFINITY;
#pragma unroll
                for (int k = 0; k < 128; k += 8)
#pragma unroll
                    for (int u = 0; u < 8; ++u)
                        m8[u] = fmaxf(m8[u], s[k + u]);
                const float mx = fmaxf(fmaxf(fmaxf(m8[0], m8[1]), fmaxf(m8[2], m8[3])),
                                       fmaxf(fmaxf(m8[4], m8[5]), fmaxf(m8[6], m8[7])));
                const float mxs = mx * c;
                const bool need =
                    mxs > m_used + kRescaleLog2 || (m_used == -INFINITY && mxs > -INFINITY);
                float factor = 1.f;
                if (need) {
                    factor = m_used == -INFINITY ? 0.f : fast_exp2(m_used - mxs);
                    m_used = mxs;
                    l *= factor;
                }
                const float mu = m_used == -INFINITY ? 0.f : m_used;
                // Exponent arguments and the running sum two at a time (packed
                // fp32x2 FMA and add): half the instructions of the scalar forms.
                const float2 c2 = make_float2(c, c), nmu2 = make_float2(-mu, -mu);
                float2 lsum[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f),
                                  make_float2(0.f, 0.f)};
                auto exp_store = [&](int hf) {
                    uint32_t pk[32];
#pragma unroll
                    for (int k = 0; k < 32; ++k) {
                        const float2 x = __ffma2_rn(make_float2(s[64 * hf + 2 * k], s[64 * hf + 2 * k + 1]), c2, nmu2);
                        const float2 pp = make_float2(fast_exp2(x.x), fast_exp2(x.y));
                        lsum[k & 3] = __fadd2_rn(lsum[k & 3], pp);
                        pk[k] = pack_bf16x2(pp.x, pp.y);
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
                // O_h holds P_h(j-1) V_{j-1} complete (the commit of S_h(j)
                // covers it): rescale it if the maximum moved (after P, when the
                // scores no longer occupy registers).
                if (j >= 1 && __any_sync(0xffffffffu, need)) {
#pragma unroll
                    for (int q4 = 0; q4 < kD / 32; ++q4) {
                        uint32_t ov[32];
                        tmem_ld32(to + 32u * q4, ov);
                        tmem_wait_ld();
#pragma unroll
                        for (int k = 0; k < 32; ++k)
                            ov[k] = __float_as_uint(__uint_as_float(ov[k]) * factor);
                        tmem_st32(to + 32u * q4, ov);
                    }
                }
                tmem_wait_st();
                // V rows past the context hold stale bytes: zero them (P is 0
                // there, but 0 * NaN is not) before either head's P V.
                if (head == 0 && n < key0 + kKeys) {
                    mbar_wait_bounded(&bar[kVFull + (gj & 1)], (gj >> 1) & 1, misc, a.err);
                    const int z0 = max(0, n - key0);
                    constexpr int kRowChunks = kD / 8;    // 16-byte chunks per V row
                    const int nz = (kKeys - z0) * kRowChunks;
                    uint8_t* vb = smem + Layout::kV + (gj & 1) * Layout::kMat;
                    for (int idx = r; idx < nz; idx += 128) {
                        const int zr = z0 + idx / kRowChunks, ch = idx % kRowChunks;
                        *reinterpret_cast<uint4*>(vb + (ch >> 3) * Layout::kHalf + zr * 128 +
                                                  (((ch & 7) ^ (zr & 7)) << 4)) = make_uint4(0, 0, 0, 0);
                    }
                    fence_proxy_async_smem();
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0)
                    mbar_arrive(&bar[kPFull + head]);
                if (kPieces && pend_it >= 0)
                    arrive_pending();
            }
            // ---- epilogue of the item ---------------------------------------------
            if (nt > 0) {
                mbar_wait_warp(&bar[kPVDone + head], (g + nt - 1) & 1, misc, a.err);
                tc_fence_after();
            }
            if constexpr (kPieces) {
                const int slot = e[kESlot];
                if (role == kPublish) {
                    // The item's last tiles: their state (part 0) for the block
                    // that holds the item's first tiles; this warp arrives one
                    // tile later, once the stores have drained.
                    const int64_t i0 = piece_state(slot, 0, head);
                    store_piece_state(a.state + i0 * 16 * 128 + r, a.state_ml + i0 * 128 + r, to, nt > 0,
                                      m_used, l);
                    pend_it = it;
                } else {
                    // O / l -> bf16; merged first with the state the item's last
                    // tiles left: M = max(m, m_t), l' = l 2^(m - M) + l_t 2^(m_t - M),
                    // o = (O 2^(m - M) + O_t / l_t l_t 2^(m_t - M)) / l'.
                    const float a_own = l > 0.f ? a.out_scale / l : 0.f;
                    float2 w_m = make_float2(0.f, 0.f);   // merge weights (last tiles, these)
                    const float inv_own = piece_inv(l);
                    const uint4* st_t = nullptr;
                    bool skip = false;                 // the receiving block writes these rows
                    if (role == kMerge) {
                        // Normally the last tiles' state is long there; if not,
                        // this part's state is left and the receiving block,
                        // arriving second, writes the rows (no wait either way).
                        unsigned long long* w = a.arrive + (int64_t(slot) * 2 + head) * 4 + w4;
                        bool got = false;
                        if (lane == 0) {
                            const unsigned long long v = ld_acquire_gpu(w);
                            got = uint32_t(v >> 32) == uint32_t(a.stamp) && uint32_t(v) >= 1u;
                        }
                        got = __shfl_sync(0xffffffffu, got, 0);
                        if (!got) {
                            const int64_t i1 = piece_state(slot, 1, head);
                            store_piece_state(a.state + i1 * 16 * 128 + r, a.state_ml + i1 * 128 + r, to,
                                              nt > 0, m_used, l);
                            __threadfence();
                            __syncwarp();
                            unsigned old = 0;
                            if (lane == 0)
                                old = arrive_piece(w, uint32_t(a.stamp));
                            old = __shfl_sync(0xffffffffu, old, 0);
                            skip = old == 0;
                            __threadfence();
                        }
                        __syncwarp();
                        const int64_t i0 = piece_state(slot, 0, head);
                        w_m = merge_weights(__ldcg(a.state_ml + i0 * 128 + r), make_float2(m_used, l),
                                            a.out_scale);
                        st_t = a.state + i0 * 16 * 128 + r;
                    }
                    // This warp's 32 rows: one TMA store of 32 rows x 64 columns per
                    // half from the staging buffer (rows past L are outside the output
                    // map's L extent and are not written).
                    const int oz = e[kEB] * a.H_q + e[head == 0 ? kEH0 : kEH1];
                    const bool write =
                        !skip && rows - w4 * 32 > 0 && misc[0] == 0 && !(head == 1 && e[kEDup]);
#pragma unroll 1
                    for (int hf = 0; hf < Layout::kHalves; ++hf) {
                        // the staging buffer's previous store has read it
                        if (lane == 0)
                            tma_store_wait_read();
                        __syncwarp();
#pragma unroll
                        for (int q = 0; q < 2; ++q) {     // columns 64 hf + 32 q .. + 31 of this row
                            uint32_t ov[32];
                            if (nt > 0) {
                                tmem_ld32(to + 32u * (2 * hf + q), ov);
                                tmem_wait_ld();
                            } else {
#pragma unroll
                                for (int k = 0; k < 32; ++k)
                                    ov[k] = 0u;
                            }
                            float* o = reinterpret_cast<float*>(ov);
                            if (st_t == nullptr) {
#pragma unroll
                                for (int k = 0; k < 32; ++k)
                                    o[k] *= a_own;
                            } else {
                                // this part's O / l rounded as its state would be, then
                                // the merge with the last tiles' state
#pragma unroll
                                for (int c4 = 0; c4 < 4; ++c4) {
                                    const uint4 v = __ldcg(st_t + (8 * hf + 4 * q + c4) * 128);
                                    const uint32_t vw[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                                    for (int k = 0; k < 4; ++k) {
                                        const uint32_t own = pack_bf16x2(o[8 * c4 + 2 * k] * inv_own,
                                                                         o[8 * c4 + 2 * k + 1] * inv_own);
                                        o[8 * c4 + 2 * k] = merge_one(w_m, __uint_as_float(vw[k] << 16),
                                                                      __uint_as_float(own << 16));
                                        o[8 * c4 + 2 * k + 1] =
                                            merge_one(w_m, __uint_as_float(vw[k] & 0xffff0000u),
                                                      __uint_as_float(own & 0xffff0000u));
                                    }
                                }
                            }
#pragma unroll
                            for (int c4 = 0; c4 < 4; ++c4) {
                                const int cq = 4 * q + c4;
                                const float* oc = o + 8 * c4;
                                *reinterpret_cast<uint4*>(stage + lane * 128 + ((cq ^ (lane & 7)) << 4)) =
                                    make_uint4(pack_bf16x2(oc[0], oc[1]), pack_bf16x2(oc[2], oc[3]),
                                               pack_bf16x2(oc[4], oc[5]), pack_bf16x2(oc[6], oc[7]));
                            }
                        }
                        fence_proxy_async_smem();
                        __syncwarp();
                        if (lane == 0 && write) {
                            tma_store_3d(&out_map, stage, hf * 64, row0 + w4 * 32, oz);
                            tma_store_commit();
                        }
                    }
                }
            } else {
                const int oz = e[kEB] * a.H_q + e[head == 0 ? kEH0 : kEH1];
                const bool write = rows - w4 * 32 > 0 && misc[0] == 0 && !(head == 1 && e[kEDup]);
                const float inv = l > 0.f ? a.out_scale / l : 0.f;
                // This warp's 32 rows: one TMA store of 32 rows x 64 columns per
                // half from the staging buffer (rows past L are outside the
                // output map's L extent and are not written).
#pragma unroll 1
                for (int hf = 0; hf < Layout::kHalves; ++hf) {
                    // the staging buffer's previous store has read it
                    if (lane == 0)
                        tma_store_wait_read();
                    __syncwarp();
#pragma unroll
                    for (int q = 0; q < 2; ++q) {     // columns 64 hf + 32 q .. + 31 of this row
                        uint32_t ov[32];
                        if (nt > 0) {
                            tmem_ld32(to + 32u * (2 * hf + q), ov);
                            tmem_wait_ld();
                        } else {
#pragma unroll
                            for (int k = 0; k < 32; ++k)
                                ov[k] = 0u;
                        }
#pragma unroll
                        for (int c4 = 0; c4 < 4; ++c4) {
                            const int cq = 4 * q + c4;
                            const uint32_t* o = ov + 8 * c4;
                            *reinterpret_cast<uint4*>(stage + lane * 128 + ((cq ^ (lane & 7)) << 4)) = make_uint4(
                                pack_bf16x2(__uint_as_float(o[0]) * inv, __uint_as_float(o[1]) * inv),
                                pack_bf16x2(__uint_as_float(o[2]) * inv, __uint_as_float(o[3]) * inv),
                                pack_bf16x2(__uint_as_float(o[4]) * inv, __uint_as_float(o[5]) * inv),
                                pack_bf16x2(__uint_as_float(o[6]) * inv, __uint_as_float(o[7]) * inv));
                        }
                    }
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0 && write) {
                        tma_store_3d(&out_map, stage, hf * 64, row0 + w4 * 32, oz);
                        tma_store_commit();
                    }
                }
            }
            // the O reads above are ordered before the next item's first P V
            // (issued once this warp arrives for that tile)
            tc_fence_before();
            g += nt;
        }
        if (kPieces && pend_it >= 0)
            arrive_pending();
        if (lane == 0)
            tma_store_wait_all();     // every output store has landed
        __syncwarp();
    }

    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

}  // namespace

size_t prefill_pairs_smem_bytes(int D)
{
    return D == 64 ? size_t(Layout<64>::kBytes) : size_t(Layout<128>::kBytes);
}

namespace {
// per block slot: O / l of both parts and heads, (m, l) per row, part and
// head, one arrival word per head and softmax warp
constexpr size_t kPieceState = 2 * 2 * 16 * 128 * sizeof(uint4);
constexpr size_t kPieceMl = 2 * 2 * 128 * sizeof(float2);
constexpr size_t kPieceArrive = 2 * 4 * sizeof(unsigned long long);
}  // namespace

size_t prefill_pairs_workspace_bytes(int grid)
{
    return size_t(grid) * (kPieceState + kPieceMl + kPieceArrive);
}

namespace {

// Register split and shared-memory limit checked once per device and
// instantiation, then the launch.
template <bool kOdd, int kD, bool kPieces, bool kSmall>
cudaError_t launch_pairs(const cudaLaunchConfig_t& cfg_in, const CUtensorMap& q_map,
                         const CUtensorMap& key_map, const CUtensorMap& value_map,
                         const CUtensorMap& out_map, const PrefillArgs& a, int device)
{
    constexpr int kMaxDev = 64;
    static std::atomic<int> smem_set[kMaxDev];
    static std::atomic<int> regs_ok[kMaxDev];
    if (device < 0 || device >= kMaxDev)
        return cudaErrorInvalidDevice;
    const void* fn = reinterpret_cast<const void*>(prefill_pairs_kernel<kOdd, kD, kPieces, kSmall>);
    const int smem = Layout<kD>::kBytes;
    // The register split needs 128 x kRegsProducer + 256 x kRegsSoftmax
    // registers out of the launch's own 384 x numRegs, a launch count no
    // higher than kRegsSoftmax (the increase must be one) and no lower than
    // kRegsProducer; otherwise the increase would wait forever.
    int rk = regs_ok[device].load(std::memory_order_relaxed);
    if (rk == 0) {
        cudaFuncAttributes fa;
        cudaError_t e = cudaFuncGetAttributes(&fa, fn);
        if (e != cudaSuccess)
            return e;
        const bool fits = fa.numRegs >= kRegsProducer && fa.numRegs <= kRegsSoftmax &&
                          128 * kRegsProducer + 256 * kRegsSoftmax <= kThreads * fa.numRegs;
        rk = fits ? 1 : 2;
        regs_ok[device].store(rk, std::memory_order_relaxed);
    }
    if (rk != 1)
        return cudaErrorNotSupported;
    if (smem_set[device].load(std::memory_order_relaxed) < smem) {
        cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess)
            return e;
        smem_set[device].store(smem, std::memory_order_relaxed);
    }
    cudaLaunchConfig_t cfg = cfg_in;
    cfg.dynamicSmemBytes = size_t(smem);
    return cudaLaunchKernelEx(&cfg, prefill_pairs_kernel<kOdd, kD, kPieces, kSmall>, q_map, key_map, value_map,
                              out_map, a);
}

}  // namespace

cudaError_t launch_prefill_pairs(const CUtensorMap& q_map, const CUtensorMap& key_map,
                                 const CUtensorMap& value_map, const CUtensorMap& out_map,
                                 const PrefillArgs& a_in, int device, int grid_cap, void* workspace,
                                 size_t workspace_bytes, cudaStream_t stream)
{
    PrefillArgs a = a_in;
    a.state = nullptr;
    a.state_ml = nullptr;
    a.arrive = nullptr;
    a.stamp = 0;
    if (a.D != 64 && a.D != 128)
        return cudaErrorInvalidValue;
    // One block per SM (grid_cap: the SM count; one block fits per SM); more
    // blocks only when one would get more than kMaxItems - 1 items (one entry
    // stays free for a piece).
    const int64_t n_items = int64_t(a.B) * a.H_kv * ((a.G + 1) / 2) * a.n_qtiles;
    int64_t grid = n_items < grid_cap ? n_items : grid_cap;
    const int64_t min_grid = (n_items + kMaxItems - 2) / (kMaxItems - 1);
    if (grid < min_grid)
        grid = min_grid;
    if (grid < 1 || grid >= (int64_t(1) << 31))
        return cudaErrorInvalidValue;
    // Programmatic stream serialization: the blocks may be scheduled while the
    // previous kernel in the stream finishes; each waits for it
    // (griddepcontrol.wait) before reading anything.
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(unsigned(grid));
    cfg.blockDim = dim3(kThreads);
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const bool odd = a.G % 2 != 0;
    const bool small = a.ps < 8;
    auto launch = [&]() {
        if (small) {
            if (a.D == 64)
                return odd ? launch_pairs<true, 64, false, true>(cfg, q_map, key_map, value_map, out_map, a, device)
                           : launch_pairs<false, 64, false, true>(cfg, q_map, key_map, value_map, out_map, a, device);
            return odd ? launch_pairs<true, 128, false, true>(cfg, q_map, key_map, value_map, out_map, a, device)
                       : launch_pairs<false, 128, false, true>(cfg, q_map, key_map, value_map, out_map, a, device);
        }
        if (a.D == 64)
            return odd ? launch_pairs<true, 64, false, false>(cfg, q_map, key_map, value_map, out_map, a, device)
                       : launch_pairs<false, 64, false, false>(cfg, q_map, key_map, value_map, out_map, a, device);
        if (a.state != nullptr)
            return odd ? launch_pairs<true, 128, true, false>(cfg, q_map, key_map, value_map, out_map, a, device)
                       : launch_pairs<false, 128, true, false>(cfg, q_map, key_map, value_map, out_map, a, device);
        return odd ? launch_pairs<true, 128, false, false>(cfg, q_map, key_map, value_map, out_map, a, device)
                   : launch_pairs<false, 128, false, false>(cfg, q_map, key_map, value_map, out_map, a, device);
    };
    // Tail pieces: with a workspace, one or two items per block and the
    // ranking in shared memory; otherwise whole items. No block waits for
    // another (the second to arrive merges), so the launch is an ordinary one.
    const int64_t M = int64_t(a.B) * a.n_qtiles;
    if (workspace && !small && a.D == 128 && M <= kThreads && n_items > grid && n_items <= 2 * grid &&
        workspace_bytes >= prefill_pairs_workspace_bytes(int(grid)) &&
        (reinterpret_cast<uintptr_t>(workspace) & 255u) == 0) {
        uint8_t* w = static_cast<uint8_t*>(workspace);
        a.state = reinterpret_cast<uint4*>(w);
        a.state_ml = reinterpret_cast<float2*>(w + size_t(grid) * kPieceState);
        a.arrive = reinterpret_cast<unsigned long long*>(w + size_t(grid) * (kPieceState + kPieceMl));
        a.stamp = next_launch_stamp();
    }
    return launch();
}

}  // namespace pa
