// Split-KV paged attention (the decode schedule).
//
// What it computes: for every request b, query head h_q and query row i,
// softmax(scale * q . K^T + causal mask) . V over the request's logical
// context, K/V read page by page through block_table (Week 3 Day 4: Direct
// Paged Attention, "Task 2"; Reading vLLM's PagedAttention Kernel, 3.3).
//
// Schedule (GB300-first, not the pages' Metal or vLLM threading):
//   * A segment is (request b, KV head h, tile of 16 query rows). The rows of
//     a tile are the G = H_q / H_kv query heads of the KV group times the L
//     query rows, so all heads of a group share every K/V byte that is loaded
//     (one grouped-query schedule for every ratio, Week 3 Day 4,
//     "Checkpoint 2").
//   * A segment's keys are cut into granules of 64 tokens; the granules of all
//     segments form one stream that the grid splits into equal contiguous
//     ranges (split-KV across blocks: the cached context is spread over the
//     whole GPU however ragged the lengths are).
//   * Per block: one producer warp finds each piece's segment, context
//     length and page-table row once, reads the row 64 page ids at a time into
//     registers (one window ahead), resolves each page id once per page by
//     shuffle (address translation hoisted per TMA box and issued behind the
//     previous granule's copies), and issues TMA tile loads of whole page
//     slices into a 3-stage shared-memory ring (128B swizzle; four half-size
//     stages for e4m3 pages). Four consumer warps split the
//     head dimension: each computes S = Q K^T for all 64 tokens of a granule
//     (the same values in every warp, so the softmax state needs no exchange)
//     and O += P V for its quarter of the output columns, on the tensor cores
//     (mma.sync m16n8k16, bf16 in, fp32 accumulate), with the online-softmax
//     recurrence in registers (running max, running sum, rescaled output;
//     Week 3 Day 4, "Task 2").
//   * A segment that one block finished alone is normalised and written at
//     once. A segment that straddles blocks leaves one partial (m, l, acc)
//     per block; a second, small kernel (one block per such segment, chained
//     by programmatic dependent launch so it is resident before this one
//     ends) merges them: M = max m_s, l = sum l_s 2^(m_s - M),
//     o = sum acc_s 2^(m_s - M) / l. No block ever waits for another block.
//   * Scores live in the log2 domain (scale * log2(e) folded into one FFMA)
//     so every exponential is one ex2.approx; the output is rescaled only
//     when a running maximum moves.
//   * Masked scores are selected to -inf (never multiplied by zero); V rows
//     past the context are zeroed in shared memory before P V, so stale or
//     NaN bytes in unused page slots never reach the result.
#include <cuda.h>
#include <cuda_bf16.h>
#include <math.h>
#include <stdint.h>

#include <atomic>

#include "pa_device.cuh"
#include "pa_internal.h"

namespace pa {
namespace {

constexpr int kConsumerWarps = 4;
constexpr int kConsumerThreads = 32 * kConsumerWarps;
constexpr int kThreads = kConsumerThreads + 32;

// F8: K/V pages of e4m3 codes (one byte per element; 128-byte rows at
// D = 128): half-size stages, four of them, and a tile for the merge of the
// four consumer warps' states at the end of a piece.
// TG: 16-row query tiles per segment; each stage holds the Q tiles of all of
// them. Three stages where they fit in about half the shared memory of an SM
// (two blocks per SM), otherwise two.
template <int D, bool F8 = false, int TG = 1>
struct Layout {
    static constexpr int kHalves = D / 64;                   // Q: 128-byte column blocks (bf16)
    static constexpr int kKVHalves = F8 ? D / 128 : D / 64;  // K/V: 128-byte column blocks
    static constexpr int kHalfBytes = kDecodeTokens * 128;   // 64 rows x 128 B
    static constexpr int kStageBytes = kKVHalves * kHalfBytes; // K (or V) of one granule
    // Q tiles of the segment whose piece starts at a stage's granule:
    // [stage][tile][half][16 rows][128 B], 128B swizzle (TMA box of 16 rows).
    static constexpr int kQHalfBytes = kDecodeRows * 128;
    static constexpr int kQStageBytes = TG * kHalves * kQHalfBytes;
    static constexpr int kStages =
        F8 ? 4 : (3 * (2 * kStageBytes + kQStageBytes) <= 110 * 1024 ? 3 : 2);
    static constexpr int kK = 0;
    static constexpr int kV = kK + kStages * kStageBytes;
    static constexpr int kQ = kV + kStages * kStageBytes;
    // F8: each consumer warp's normalised O (f16) at the end of a piece,
    // [warp][16 rows][D]
    static constexpr int kWork = kQ + kStages * kQStageBytes;
    static constexpr int kWorkBytes = F8 ? kConsumerWarps * kDecodeRows * D * 2 : 0;
    static constexpr int kBar = kWork + kWorkBytes;
    static constexpr int kMisc = kBar + 2 * kStages * 8;     // abort flag, test barrier
    // [B + 1] int32 granule prefix, then [B] int32 granules per segment
    static constexpr int kPrefix = kMisc + 32;
    static size_t bytes(int B) { return kPrefix + size_t(2 * B + 1) * 4 + 1024; }
};

__device__ __forceinline__ int clamp_context(int n, int cap, unsigned* err)
{
    if (n < 0 || n > cap) {
        atomicOr(err, PA_DEVERR_CONTEXT_LEN_BIT);
        n = n < 0 ? 0 : cap;
    }
    return n;
}

struct SegmentPos {
    int b, h, ms, seg;  // request, KV head, segment within the (b, h) rows
    int64_t seg_start;  // first granule of the segment in the stream
    int seg_len;        // granules in the segment
};

// The segment hm (0 <= hm < per_req) of request b. pre[b] = first granule of
// request b, gbr[b] = granules in each of its segments.
__device__ __forceinline__ SegmentPos segment_at(const int32_t* pre, const int32_t* gbr,
                                                 int per_req, int MS, int b, int hm)
{
    SegmentPos s;
    s.b = b;
    s.h = MS == 1 ? hm : hm / MS;
    s.ms = hm - s.h * MS;
    s.seg = b * per_req + hm;
    s.seg_len = gbr[b];
    s.seg_start = pre[b] + int64_t(hm) * s.seg_len;
    return s;
}

// The segment after s in the stream (segments are in (request, KV head, row
// tile group) order and none is empty).
__device__ __forceinline__ SegmentPos next_segment(const int32_t* pre, const int32_t* gbr,
                                                   int per_req, int MS, const SegmentPos& s)
{
    const int hm = s.seg - s.b * per_req + 1;
    return hm < per_req ? segment_at(pre, gbr, per_req, MS, s.b, hm)
                        : segment_at(pre, gbr, per_req, MS, s.b + 1, 0);
}

// The split over blocks weighs each segment as its granules plus pu units
// (DecodeArgs::piece_units): a piece costs a block more than its granules (the
// first granule's Q tile, the partial tail granule, the epilogue; for e4m3
// pages also the merge of the four warp states), and a block that gets many
// short segments would otherwise end last. Unit stream: segment s is pu units
// of overhead, then its granules, so granule x of segment s sits at unit
// x + pu * (s + 1); block i owns the units [floor(i*T/grid),
// floor((i+1)*T/grid)), T = granules + pu * nseg, i.e. the granules whose
// units fall there. The merge pass recomputes the split with the same pu.
// A piece costs about one granule beyond its own on bf16 pools and about
// three on e4m3 pools (measured on 128-token pages: 79.9 us with 1, 63.4
// with 3).
__host__ __device__ constexpr int piece_units(bool f8) { return f8 ? 3 : 1; }

// Block index that processes the granule at unit position u.
__device__ __forceinline__ int64_t block_of_unit(int64_t u, int64_t units, int64_t grid)
{
    return udiv64((u + 1) * grid - 1, units);
}

// First granule whose unit position is >= u (the granule count if none),
// and the request b and segment hm within it that hold that granule (b = B
// if none), for the two unit positions u0 <= u1 at once (the two searches
// and their divisions interleave). Called by whole warps.
struct StreamPoint {
    int64_t x;
    int b, hm;
};
__device__ __forceinline__ void granules_at_units(const int32_t* pre, const int32_t* gbr, int B,
                                                  int per_req, int64_t u0, int64_t u1,
                                                  int64_t units, int pu, StreamPoint& p0,
                                                  StreamPoint& p1)
{
    const int lane = threadIdx.x & 31;
    const int64_t per_b = int64_t(pu) * per_req;
    auto pre_u = [&](int b) { return int64_t(pre[b]) + per_b * b; };
    // largest b with pre_u(b) <= u, for both u (pre_u(0) = 0 <= u); each
    // round samples 32 evenly spaced candidates of the remaining range, so
    // B <= 32 takes one round of one shared-memory read per lane
    int lo0 = 0, n0 = B, lo1 = 0, n1 = B;
    while (n0 > 32 || n1 > 32) {
        const int s0 = (n0 + 31) >> 5, s1 = (n1 + 31) >> 5;
        const bool ok0 = lane * s0 < n0 && pre_u(lo0 + lane * s0) <= u0;
        const bool ok1 = lane * s1 < n1 && pre_u(lo1 + lane * s1) <= u1;
        const int l0 = 31 - __clz(__ballot_sync(0xffffffffu, ok0));
        const int l1 = 31 - __clz(__ballot_sync(0xffffffffu, ok1));
        lo0 += l0 * s0;
        n0 = min(s0, n0 - l0 * s0);
        lo1 += l1 * s1;
        n1 = min(s1, n1 - l1 * s1);
    }
    const bool ok0 = lane < n0 && pre_u(lo0 + lane) <= u0;
    const bool ok1 = lane < n1 && pre_u(lo1 + lane) <= u1;
    lo0 += 31 - __clz(__ballot_sync(0xffffffffu, ok0));
    lo1 += 31 - __clz(__ballot_sync(0xffffffffu, ok1));
    auto finish = [&](int lo, int64_t u, StreamPoint& p) {
        if (u >= units) {
            p = StreamPoint{pre[B], B, 0};
            return;
        }
        const int gb = gbr[lo];
        const int64_t r = u - pre_u(lo);
        const int64_t hm = udiv64(r, gb + pu);
        const int64_t in = r - hm * (gb + pu) - pu;
        p = StreamPoint{pre[lo] + hm * gb + (in > 0 ? in : 0), lo, int(hm)};
    };
    finish(lo0, u0, p0);
    finish(lo1, u1, p1);
}

template <int D, bool F8 = false, int TG = 1>
__global__ void __launch_bounds__(kThreads, 2)
    decode_kernel(const __grid_constant__ CUtensorMap key_map,
                  const __grid_constant__ CUtensorMap value_map,
                  const __grid_constant__ CUtensorMap q_map, const DecodeArgs a)
{
    using Lay = Layout<D, F8, TG>;
    constexpr int kStages = Lay::kStages;
    static_assert(!F8 || (D == 128 && TG == 1), "e4m3 pages: head_dim 128, one row tile");
    static_assert(TG == 1 || TG == 2 || TG == 4, "row tiles per segment");
    constexpr int kKS = D / 16;  // k-steps of 16 over the head dimension

    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    int32_t* pre = reinterpret_cast<int32_t*>(smem + Lay::kPrefix);
    int32_t* gbr = pre + a.B + 1;
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + Lay::kBar);
    uint64_t* empty = full + kStages;
    volatile int* misc = reinterpret_cast<volatile int*>(smem + Lay::kMisc);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int per_req = a.H_kv * a.MS;
    const int cap = a.max_pages * a.ps;

    // Set-up that reads no input runs before the wait below, overlapping the
    // tail of the previous kernel in the stream: the pipeline barriers and
    // the tensor-map prefetch.
    uint64_t* never = reinterpret_cast<uint64_t*>(smem + Lay::kMisc + 16);
    if (threadIdx.x == 0) {
        misc[0] = 0;
        misc[1] = 0;
        misc[2] = 0;
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], kConsumerWarps);
        }
        mbar_init(never, 1);
        fence_barrier_init();
    }
    if (warp == kConsumerWarps && lane == 0) {
        prefetch_tensormap(&key_map);
        prefetch_tensormap(&value_map);
        prefetch_tensormap(&q_map);
    }

    // The prologue below (granule prefix, this block's range and first
    // segment) runs twice: first on made-up context lengths (64 granules
    // each), before the wait for the previous kernel, so that its code
    // is fetched into the instruction caches while that kernel drains; then,
    // after the wait, on the real inputs. Only the second pass's results are
    // used.
    constexpr int kPU = piece_units(F8);
    int64_t total = 0, units = 0, grid = 0;
    const int64_t cta = blockIdx.x;
    // The block's granules [x_begin, x_end) and the segment of x_begin.
    int64_t x_begin = 0, x_end = 0;
    SegmentPos first;
#pragma unroll 1
    for (int pass = 0; pass < 2; ++pass) {
        const bool real = pass == 1;
        if (real) {
            // Inputs may come from the previous kernel in the stream (e.g. the
            // append of this step): wait for it before reading any of them,
            // and let the merge pass that follows this kernel be scheduled
            // right away.
            grid_dependency_wait();
            grid_launch_dependents();
        }
        // ---- granule prefix over requests (one warp) -----------------------
        if (warp == 0) {
            int carry = 0;
            if (lane == 0)
                pre[0] = 0;
            for (int base = 0; base < a.B; base += 32) {
                const int b = base + lane;
                int g = 0;
                if (b < a.B) {
                    const int n =
                        real ? clamp_context(a.context_lens[b], cap, a.err) : 64 * kDecodeTokens;
                    const int gs = max(1, (n + kDecodeTokens - 1) / kDecodeTokens);
                    gbr[b] = gs;
                    g = gs * per_req;
                }
                int incl = g;
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) {
                    const int v = __shfl_up_sync(0xffffffffu, incl, o);
                    if (lane >= o)
                        incl += v;
                }
                if (b < a.B)
                    pre[b + 1] = carry + incl;
                carry += __shfl_sync(0xffffffffu, incl, 31);
            }
        }
        if (real && threadIdx.x == 0 && a.debug_unset_wait && blockIdx.x == 0) {
            // Test support: a wait on a barrier nothing arrives at must run
            // out, record the timeout bit and let the kernel finish normally.
            // The whole block waits for it below, before any copy is issued.
            const uint64_t t0 = global_timer_ns();
            while (!mbar_try_wait(never, 0)) {
                if (global_timer_ns() - t0 > kWaitLimitNs) {
                    atomicOr(a.err, PA_DEVERR_TIMEOUT_BIT);
                    break;
                }
            }
        }
        __syncthreads();

        total = pre[a.B];
        units = total + int64_t(kPU) * a.B * per_req;
        // The unit stream is split over min(gridDim.x, units) blocks so that
        // every block in use owns at least one unit; a segment whose granules
        // span blocks first..last then has exactly last - first + 1 pieces
        // (every block in between owns units inside the segment's granules).
        grid = a.whole_segments ? int64_t(gridDim.x)
                                : (int64_t(gridDim.x) < units ? int64_t(gridDim.x) : units);
        x_begin = x_end = 0;
        if (cta < grid) {
            if (a.whole_segments) {
                // Whole segments per block: segments [s0, s1) of nseg.
                const int64_t nseg = int64_t(a.B) * per_req;
                const int64_t s0 = udiv64(cta * nseg, grid), s1 = udiv64((cta + 1) * nseg, grid);
                if (s0 < s1) {
                    const int b0 = int(udiv64(s0, per_req));
                    first = segment_at(pre, gbr, per_req, a.MS, b0, int(s0 - int64_t(b0) * per_req));
                    x_begin = first.seg_start;
                    if (s1 >= nseg) {
                        x_end = total;
                    } else {
                        const int b1 = int(udiv64(s1, per_req));
                        x_end = pre[b1] + (s1 - int64_t(b1) * per_req) * gbr[b1];
                    }
                }
            } else {
                StreamPoint p0, p1;
                granules_at_units(pre, gbr, a.B, per_req, udiv64(cta * units, grid),
                                  udiv64((cta + 1) * units, grid), units, kPU, p0, p1);
                x_begin = p0.x;
                x_end = p1.x;
                if (x_begin < x_end)
                    first = segment_at(pre, gbr, per_req, a.MS, p0.b, p0.hm);
            }
        }
        if (!real)
            __syncthreads();   // pass 0's tables are read by every warp before pass 1 rewrites them
    }
    if (x_begin >= x_end)
        return;

    auto k_half = [&](int stage, int half) -> uint8_t* {
        return smem + Lay::kK + stage * Lay::kStageBytes + half * Lay::kHalfBytes;
    };
    auto v_half = [&](int stage, int half) -> uint8_t* {
        return smem + Lay::kV + stage * Lay::kStageBytes + half * Lay::kHalfBytes;
    };

    if (warp == kConsumerWarps) {
        // ===================== producer warp: page walk + TMA =================
        const uint64_t policy = l2_policy_evict_first();
        const int box = a.box_rows;
        int stage = 0;
        uint32_t phase = 0;
        // Per piece (the granules of one segment inside this block's range):
        // the segment, its context length, page-table row and Q rows, found
        // once. Per granule only the address translation of its boxes remains,
        // and the next granule's is issued as soon as this one's copies are
        // out, so its loads overlap the wait for a free stage.
        int64_t x = x_begin;
        for (SegmentPos sp = first; x < x_end;
             sp = next_segment(pre, gbr, per_req, a.MS, sp)) {
            const int64_t piece_start = x;
            const int64_t piece_end =
                x_end < sp.seg_start + sp.seg_len ? x_end : sp.seg_start + sp.seg_len;
            const int n = clamp_context(__ldg(a.context_lens + sp.b), cap, a.err);
            const int32_t* bt = a.block_table + int64_t(sp.b) * a.max_pages;
            // The piece's page ids, 64 at a time: a window of pages [wb, wb + 64)
            // with page wb + lane in c0 and wb + 32 + lane in c1, and the next
            // window already on its way (n0, n1), so a granule finds its ids by
            // shuffle instead of waiting on a load. Pool page and box sizes are
            // powers of two; a granule's pages never straddle two windows. The
            // dense layout (request b is page b, of any length) reads no table.
            const int ps_shift = __ffs(a.ps) - 1;
            const int box_shift = __ffs(box) - 1;
            auto load_window = [&](int w, int& e0, int& e1) {
                e0 = e1 = 0;
                if (a.dense)
                    return;
                if (w + lane < a.max_pages)
                    e0 = __ldg(bt + w + lane);
                if (w + 32 + lane < a.max_pages)
                    e1 = __ldg(bt + w + 32 + lane);
            };
            int wb = a.dense ? 0 : (int((x - sp.seg_start) * kDecodeTokens) >> ps_shift) & ~63;
            int c0, c1, n0, n1;
            load_window(wb, c0, c1);
            load_window(wb + 64, n0, n1);
            // The TMA row of each box of granule xx (boxes lane and lane + 32).
            auto translate = [&](int64_t xx, int& nbox, int& ra, int& rb) {
                const int t0 = int(xx - sp.seg_start) * kDecodeTokens;
                const int nvalid = min(kDecodeTokens, n - t0);
                ra = rb = 0;
                if (a.dense) {
                    // one page per request holding the whole context (t < n <= ps)
                    nbox = nvalid > 0 ? (nvalid + box - 1) / box : 0;
                    const int base = (sp.b * a.H_kv + sp.h) * a.ps + t0;
                    if (lane < nbox)
                        ra = base + lane * box;
                    if (lane + 32 < nbox)
                        rb = base + (lane + 32) * box;
                    return;
                }
                nbox = nvalid > 0 ? (nvalid + box - 1) >> box_shift : 0;
                const int lp0 = t0 >> ps_shift;
                while (lp0 >= wb + 64) {     // warp-uniform: move to the next window
                    wb += 64;
                    c0 = n0;
                    c1 = n1;
                    load_window(wb + 64, n0, n1);
                }
#pragma unroll
                for (int k = 0; k < 2; ++k) {
                    const int j = lane + 32 * k;
                    const int tok = t0 + (j << box_shift);
                    const int lp = tok >> ps_shift;
                    const int idx = (lp - wb) & 63;
                    const int p0 = __shfl_sync(0xffffffffu, c0, idx & 31);
                    const int p1 = __shfl_sync(0xffffffffu, c1, idx & 31);
                    if (j < nbox) {
                        int phys = idx < 32 ? p0 : p1;
                        if (unsigned(phys) >= unsigned(a.num_pages)) {
                            atomicOr(a.err, PA_DEVERR_PAGE_ID_BIT);
                            phys = 0;
                        }
                        const int row = (phys * a.H_kv + sp.h) * a.ps + (tok - (lp << ps_shift));
                        if (k == 0)
                            ra = row;
                        else
                            rb = row;
                    }
                }
            };
            int nbox, row_a, row_b;
            translate(x, nbox, row_a, row_b);
            // Row tiles of this segment that hold query rows (the others are
            // padding: no Q load, no compute).
            const int q_tiles = min(TG, (a.R - sp.ms * TG * kDecodeRows + kDecodeRows - 1) / kDecodeRows);
            for (; x < piece_end; ++x) {
                // The first granule of a piece also brings the segment's Q tiles
                // (the G heads x L rows of a KV group are consecutive rows of q).
                const bool first = x == piece_start;
                const bool ok = mbar_wait_warp(&empty[stage], phase ^ 1u, misc, a.err);
                if (ok && (nbox > 0 || first)) {
                    const uint32_t bytes =
                        uint32_t(nbox) * box * 128u * Lay::kKVHalves * 2u +
                        (first ? uint32_t(q_tiles * Lay::kHalves * Lay::kQHalfBytes) : 0u);
                    if (lane == 0) {
                        mbar_arrive_expect_tx(&full[stage], bytes);
                        if (first) {
                            for (int t = 0; t < q_tiles; ++t) {
                                const int qrow = (sp.b * a.H_q + sp.h * a.G) * a.L +
                                                 (sp.ms * TG + t) * kDecodeRows;
#pragma unroll
                                for (int hf = 0; hf < Lay::kHalves; ++hf)
                                    tma_load_2d(smem + Lay::kQ + stage * Lay::kQStageBytes +
                                                    (t * Lay::kHalves + hf) * Lay::kQHalfBytes,
                                                &q_map, hf * 64, qrow, &full[stage], policy);
                            }
                        }
                    }
                    __syncwarp();
#pragma unroll
                    for (int k = 0; k < 2; ++k) {
                        const int j = lane + 32 * k;
                        if (j < nbox) {
                            const int row = k == 0 ? row_a : row_b;
                            const int dst = j * box * 128;
#pragma unroll
                            for (int hf = 0; hf < Lay::kKVHalves; ++hf) {
                                // a box row is 128 bytes: 64 bf16 or 128 e4m3 elements
                                tma_load_2d(k_half(stage, hf) + dst, &key_map, hf * (F8 ? 128 : 64),
                                            row, &full[stage], policy);
                                tma_load_2d(v_half(stage, hf) + dst, &value_map,
                                            hf * (F8 ? 128 : 64), row, &full[stage], policy);
                            }
                        }
                    }
                } else if (ok && lane == 0) {
                    mbar_arrive(&full[stage]);  // empty granule: nothing to load
                }
                __syncwarp();
                if (++stage == kStages) {
                    stage = 0;
                    phase ^= 1u;
                }
                if (x + 1 < piece_end)
                    translate(x + 1, nbox, row_a, row_b);
            }
        }
        return;
    }

    // ===================== consumer warps ===================================
    // The TG row tiles of a segment are spread over the four consumer warps:
    // kWPT = 4 / TG warps per tile, each owning D / kWPT output columns. Every
    // warp computes the scores of all 64 tokens of a granule for its tile's
    // rows (identical in the kWPT warps of a tile, so the softmax state needs
    // no exchange) and P V for its own columns; a segment's result never has
    // to be merged across warps. (e4m3 pages: TG = 1, see below.)
    constexpr int kWPT = kConsumerWarps / TG;  // warps per row tile
    constexpr int kCols = D / kWPT;            // output columns per warp
    constexpr int kON = kCols / 8;             // output n-tiles per warp
    constexpr int kSN = kDecodeTokens / 8;     // score n-tiles per granule
    const int swz = a.swz;        // stage layout: chunk ^ (row & 7) when swizzled
    const int row0 = lane >> 2;   // fragment rows row0 and row0 + 8
    const int quad = lane & 3;
    const int tw = warp / kWPT;   // this warp's row tile within a segment
    const int col0 = (warp % kWPT) * kCols;
    int stage = 0;
    uint32_t phase = 0;
    constexpr int kTileFloats = kDecodeRows * (D + 2);   // m[16], l[16], acc[16][D]
    constexpr int kSlotFloats = TG * kTileFloats;

    // Row of this warp's tile of a segment, in the (request, KV head) rows
    auto tile_row = [&](const SegmentPos& p, int rw) -> int {
        return (p.ms * TG + tw) * kDecodeRows + rw;
    };
    // Output row index of fragment row rw of a segment, or -1 for padding.
    auto out_row = [&](const SegmentPos& p, int rw) -> int64_t {
        const int rg = tile_row(p, rw);
        if (rg >= a.R)
            return -1;
        const int g = rg / a.L, i = rg - g * a.L;
        return (int64_t(p.b) * a.H_q + p.h * a.G + g) * a.L + i;
    };

    if constexpr (F8) {
        // ---- e4m3 pages: warp w owns tokens [16 w, 16 w + 16) of every granule.
        // It reads their codes straight from the stage (ldmatrix on the byte
        // rows), converts them in registers to f16 (exact), computes their
        // scores and P V over all D columns on the tensor cores (f16 in, fp32
        // accumulate) and keeps its own online-softmax state; at the end of a
        // piece the four states merge through the work tile (each warp's O / l_w
        // in f16, relative error 2^-11), M = max m_w, l = sum l_w 2^(m_w - M),
        // o = sum l_w 2^(m_w - M) (O_w / l_w). Every warp then
        // holds its D/4 columns, as in the bf16 schedule, and the same
        // epilogue follows.
        //   * Codes become f16 (exact) two at a time with one conversion
        //     instruction; k_scale and v_scale stay in the softmax scale and
        //     the output.
        //   * K: ldmatrix (no transpose) of 8 byte rows gives lane (row0,
        //     quad) the codes of token row0 at d = 16 kk + 4 quad .. + 3; their
        //     two halves are the two f16 B registers when the head dimension
        //     is permuted inside each 16-wide k-step the same way in Q (a0 / a1
        //     hold d = 16 kk + 4 quad + {0, 1}, a2 / a3 + {2, 3}).
        //   * V: ldmatrix.trans of byte rows gives codes (t, d), (t, d + 1),
        //     (t + 1, d), (t + 1, d + 1), t = 2 quad (+ 8), d = 16 c + 2 (lane
        //     / 4); bytes 0, 2 feed the P V of the even d, bytes 1, 3 that of
        //     the odd d: o[2 c] holds columns 16 c + 4 quad + {0, 2},
        //     o[2 c + 1] columns 16 c + 4 quad + {1, 3}.
        constexpr int kWT = kDecodeTokens / kConsumerWarps;   // tokens per warp
        constexpr int kONF = D / 8;                           // output n-tiles per warp
        __shared__ float wstate[kConsumerWarps][2][kDecodeRows];   // (m, l) per warp and row
        uint16_t* wtile = reinterpret_cast<uint16_t*>(smem + Lay::kWork);  // [warp][16 rows][D] f16
        const int r_lo = warp * kWT;
        int64_t x = x_begin;
        for (SegmentPos sp = first; x < x_end;
             sp = next_segment(pre, gbr, per_req, a.MS, sp)) {
            const int64_t piece_end = min(x_end, sp.seg_start + sp.seg_len);
            const int n = clamp_context(a.context_lens[sp.b], cap, a.err);
            uint32_t qa[kKS][4];
            bool need_q = true;
            int lim[2];
#pragma unroll
            for (int rr = 0; rr < 2; ++rr) {
                const int rg = tile_row(sp, row0 + rr * 8);
                const int i = rg < a.R ? rg % a.L : a.L - 1;
                lim[rr] = a.causal ? min(n - a.L + i, n - 1) : n - 1;
            }
            const int lim_min = __reduce_min_sync(0xffffffffu, min(lim[0], lim[1]));
            float m_run[2] = {-INFINITY, -INFINITY};
            float l_run[2] = {0.f, 0.f};
            float o[kONF][4];
#pragma unroll
            for (int nt = 0; nt < kONF; ++nt)
                o[nt][0] = o[nt][1] = o[nt][2] = o[nt][3] = 0.f;

            for (; x < piece_end; ++x) {
                const int t0 = int(x - sp.seg_start) * kDecodeTokens;
                const int nvalid = min(kDecodeTokens, n - t0);
                const bool ok = mbar_wait_warp(&full[stage], phase, misc, a.err);
                if (need_q) {
                    const uint8_t* qs = smem + Lay::kQ + stage * Lay::kQStageBytes;
#pragma unroll
                    for (int kk = 0; kk < kKS; ++kk) {
                        const int d = 16 * kk + 4 * quad;
                        const int hf = d >> 6, ch = (d & 63) >> 3;
#pragma unroll
                        for (int rr = 0; rr < 2; ++rr) {
                            const int r = row0 + 8 * rr;
                            const uint2 v = *reinterpret_cast<const uint2*>(
                                qs + hf * Lay::kQHalfBytes + r * 128 + ((ch ^ (r & 7)) << 4) +
                                (quad & 1) * 8);
                            qa[kk][rr] = bf16x2_to_f16x2(v.x);
                            qa[kk][2 + rr] = bf16x2_to_f16x2(v.y);
                        }
                    }
                    need_q = false;
                }
                const bool live = ok && nvalid > r_lo;
                if (live && nvalid < r_lo + kWT) {
                    // V rows of this warp past the context hold stale codes
                    // (NaN among them): zero them (P is 0 there, 0 * NaN is not)
                    const int nz = (r_lo + kWT - nvalid) * 8;          // 16-byte chunks
                    for (int idx = lane; idx < nz; idx += 32) {
                        const int r = nvalid + idx / 8, c = idx % 8;
                        *reinterpret_cast<uint4*>(v_half(stage, 0) + r * 128 + ((c ^ (r & swz)) << 4)) =
                            make_uint4(0, 0, 0, 0);
                    }
                    // ordered before the TMA that refills the stage later
                    fence_proxy_async_smem();
                    __syncwarp();
                }
                if (live) {
                    // S = Q K^T for the warp's 16 tokens (2 n-tiles)
                    float sc[2][4];
#pragma unroll
                    for (int nt = 0; nt < 2; ++nt)
                        sc[nt][0] = sc[nt][1] = sc[nt][2] = sc[nt][3] = 0.f;
                    {
                        // matrices: (tokens 0-7, chunk kk), (8-15, kk), (0-7, kk + 1), (8-15, kk + 1)
                        const int tr = r_lo + (lane & 7) + (((lane >> 3) & 1) << 3);
                        const int chsel = lane >> 4;
#pragma unroll
                        for (int kp = 0; kp < kKS; kp += 2) {
                            const int ch = kp + chsel;
                            uint32_t r4[4];
                            ldsm_x4(smem_u32(k_half(stage, 0) + tr * 128 + ((ch ^ (tr & swz)) << 4)),
                                    r4[0], r4[1], r4[2], r4[3]);
#pragma unroll
                            for (int u = 0; u < 4; ++u)
                                mma_f16_16816(sc[u & 1], qa[kp + (u >> 1)],
                                              e4m3x2_to_f16x2(r4[u]),
                                              e4m3x2_hi_to_f16x2(r4[u]));
                        }
                    }
                    if (t0 + r_lo + kWT - 1 > lim_min) {
#pragma unroll
                        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                            for (int j = 0; j < 4; ++j) {
                                const int tok = t0 + r_lo + nt * 8 + 2 * quad + (j & 1);
                                if (tok > lim[j >> 1])
                                    sc[nt][j] = -INFINITY;
                            }
                    }
                    float mx[2], mu[2], mn[2];
                    bool changed = false;
#pragma unroll
                    for (int rr = 0; rr < 2; ++rr) {
                        mx[rr] = fmaxf(fmaxf(sc[0][2 * rr], sc[0][2 * rr + 1]),
                                       fmaxf(sc[1][2 * rr], sc[1][2 * rr + 1]));
                        mx[rr] = fmaxf(mx[rr], __shfl_xor_sync(0xffffffffu, mx[rr], 1));
                        mx[rr] = fmaxf(mx[rr], __shfl_xor_sync(0xffffffffu, mx[rr], 2));
                        mn[rr] = fmaxf(m_run[rr], mx[rr] * a.scale_log2);
                        changed |= mn[rr] != m_run[rr];
                        mu[rr] = mn[rr] == -INFINITY ? 0.f : mn[rr];
                    }
                    if (__any_sync(0xffffffffu, changed)) {
                        float corr[2];
#pragma unroll
                        for (int rr = 0; rr < 2; ++rr) {
                            corr[rr] = mn[rr] == m_run[rr] ? 1.f : fast_exp2(m_run[rr] - mu[rr]);
                            m_run[rr] = mn[rr];
                            l_run[rr] *= corr[rr];
                        }
#pragma unroll
                        for (int nt = 0; nt < kONF; ++nt) {
                            o[nt][0] *= corr[0];
                            o[nt][1] *= corr[0];
                            o[nt][2] *= corr[1];
                            o[nt][3] *= corr[1];
                        }
                    }
                    uint32_t pa[4];
#pragma unroll
                    for (int nt = 0; nt < 2; ++nt) {
                        float p[4];
#pragma unroll
                        for (int j = 0; j < 4; ++j) {
                            p[j] = fast_exp2(fmaf(sc[nt][j], a.scale_log2, -mu[j >> 1]));
                            l_run[j >> 1] += p[j];
                        }
                        pa[nt * 2 + 0] = pack_f16x2(p[0], p[1]);
                        pa[nt * 2 + 1] = pack_f16x2(p[2], p[3]);
                    }
                    // O[:, all D] += P V over the warp's 16 tokens
                    {
                        // matrices: (tokens 0-7, chunk c), (8-15, c), (0-7, c + 1), (8-15, c + 1)
                        const int tr = r_lo + (lane & 7) + (((lane >> 3) & 1) << 3);
                        const int chsel = lane >> 4;
#pragma unroll
                        for (int cp = 0; cp < D / 16; cp += 2) {
                            const int ch = cp + chsel;
                            uint32_t r4[4];
                            ldsm_x4_trans(smem_u32(v_half(stage, 0) + tr * 128 + ((ch ^ (tr & swz)) << 4)),
                                          r4[0], r4[1], r4[2], r4[3]);
#pragma unroll
                            for (int u = 0; u < 2; ++u) {
                                const int c = cp + u;
                                const uint32_t lo = r4[2 * u], hi = r4[2 * u + 1];
                                mma_f16_16816(o[2 * c], pa,
                                              e4m3x2_to_f16x2(__byte_perm(lo, 0u, 0x0020u)),
                                              e4m3x2_to_f16x2(__byte_perm(hi, 0u, 0x0020u)));
                                mma_f16_16816(o[2 * c + 1], pa,
                                              e4m3x2_to_f16x2(__byte_perm(lo, 0u, 0x0031u)),
                                              e4m3x2_to_f16x2(__byte_perm(hi, 0u, 0x0031u)));
                            }
                        }
                    }
                }
                __syncwarp();
                if (lane == 0)
                    mbar_arrive(&empty[stage]);       // the stage is no longer read
                if (++stage == kStages) {
                    stage = 0;
                    phase ^= 1u;
                }
            }

            // ---- end of a piece: merge the four warp states ----------------
#pragma unroll
            for (int rr = 0; rr < 2; ++rr) {
                l_run[rr] += __shfl_xor_sync(0xffffffffu, l_run[rr], 1);
                l_run[rr] += __shfl_xor_sync(0xffffffffu, l_run[rr], 2);
            }
            named_barrier_sync(1, kConsumerThreads);   // the work tile's K/V are no longer read
#pragma unroll
            for (int rr = 0; rr < 2; ++rr) {
                const int rw = row0 + rr * 8;
                const float il = l_run[rr] > 0.f ? 1.f / l_run[rr] : 0.f;
                uint16_t* dst = wtile + (warp * kDecodeRows + rw) * D + 4 * quad;
#pragma unroll
                for (int c = 0; c < D / 16; ++c)
                    *reinterpret_cast<uint2*>(dst + 16 * c) =
                        make_uint2(pack_f16x2(o[2 * c][2 * rr] * il, o[2 * c + 1][2 * rr] * il),
                                   pack_f16x2(o[2 * c][2 * rr + 1] * il, o[2 * c + 1][2 * rr + 1] * il));
                if (quad == 0) {
                    wstate[warp][0][rw] = m_run[rr];
                    wstate[warp][1][rw] = l_run[rr];
                }
            }
            named_barrier_sync(1, kConsumerThreads);
            float om[kON][4];
            float Mr[2], Lr[2];
#pragma unroll
            for (int rr = 0; rr < 2; ++rr) {
                const int rw = row0 + rr * 8;
                float M = -INFINITY;
#pragma unroll
                for (int w = 0; w < kConsumerWarps; ++w)
                    M = fmaxf(M, wstate[w][0][rw]);
                float g[kConsumerWarps];                 // l_w 2^(m_w - M)
                float L = 0.f;
#pragma unroll
                for (int w = 0; w < kConsumerWarps; ++w) {
                    const float mw = wstate[w][0][rw];
                    g[w] = mw == -INFINITY ? 0.f : wstate[w][1][rw] * fast_exp2(mw - M);
                    L += g[w];
                }
                Mr[rr] = M;
                Lr[rr] = L;
#pragma unroll
                for (int nt = 0; nt < kON; ++nt) {
                    float s0 = 0.f, s1 = 0.f;
#pragma unroll
                    for (int w = 0; w < kConsumerWarps; ++w) {
                        const __half2 h = *reinterpret_cast<const __half2*>(
                            wtile + (w * kDecodeRows + rw) * D + col0 + nt * 8 + 2 * quad);
                        const float2 v = __half22float2(h);
                        s0 += g[w] * v.x;
                        s1 += g[w] * v.y;
                    }
                    om[nt][2 * rr] = s0;
                    om[nt][2 * rr + 1] = s1;
                }
            }
            named_barrier_sync(1, kConsumerThreads);   // the tile may be refilled

            // The segment lies inside this block's range: no other block
            // holds a piece of it.
            const bool single = a.whole_segments ||
                                (sp.seg_start >= x_begin && sp.seg_start + sp.seg_len <= x_end);
            const bool aborted = misc[0] != 0;
            if (!aborted && single) {
#pragma unroll
                for (int rr = 0; rr < 2; ++rr) {
                    const int64_t orow = out_row(sp, row0 + rr * 8);
                    if (orow < 0)
                        continue;
                    const float inv = Lr[rr] > 0.f ? a.v_scale / Lr[rr] : 0.f;
                    uint16_t* dst = a.out + orow * D + col0 + 2 * quad;
#pragma unroll
                    for (int nt = 0; nt < kON; ++nt)
                        *reinterpret_cast<uint32_t*>(dst + nt * 8) =
                            pack_bf16x2(om[nt][2 * rr] * inv, om[nt][2 * rr + 1] * inv);
                }
            } else if (!aborted) {
                // the state carries v_scale, so the merge pass needs no change
                float* slot = a.partials + (int64_t(sp.seg) + cta) * kSlotFloats;
#pragma unroll
                for (int rr = 0; rr < 2; ++rr) {
                    const int rw = row0 + rr * 8;
                    if (out_row(sp, rw) < 0)
                        continue;
                    if (warp == 0 && quad == 0) {
                        slot[rw] = Mr[rr];
                        slot[kDecodeRows + rw] = Lr[rr];
                    }
                    float* dst = slot + 2 * kDecodeRows + rw * D + col0 + 2 * quad;
#pragma unroll
                    for (int nt = 0; nt < kON; ++nt)
                        *reinterpret_cast<float2*>(dst + nt * 8) =
                            make_float2(om[nt][2 * rr] * a.v_scale, om[nt][2 * rr + 1] * a.v_scale);
                }
            }
        }
    } else {
    int64_t x = x_begin;
    for (SegmentPos sp = first; x < x_end; sp = next_segment(pre, gbr, per_req, a.MS, sp)) {
        const int64_t piece_end = min(x_end, sp.seg_start + sp.seg_len);
        const int n = clamp_context(a.context_lens[sp.b], cap, a.err);

        // Q fragments of the piece: from the stage of its first granule,
        // loaded (ldmatrix) once that stage has landed. A tile past the
        // segment's rows (a group of 3 tiles in a slot of 4) computes nothing.
        uint32_t qa[kKS][4];
        const bool live_tile = tile_row(sp, 0) < a.R;
        bool need_q = live_tile;

        // Last visible position of this thread's two fragment rows.
        int lim[2];
#pragma unroll
        for (int rr = 0; rr < 2; ++rr) {
            const int rg = tile_row(sp, row0 + rr * 8);
            const int i = rg < a.R ? rg % a.L : a.L - 1;
            lim[rr] = a.causal ? min(n - a.L + i, n - 1) : n - 1;
        }
        const int lim_min = __reduce_min_sync(0xffffffffu, min(lim[0], lim[1]));

        float m_run[2] = {-INFINITY, -INFINITY};
        float l_run[2] = {0.f, 0.f};
        float o[kON][4];
#pragma unroll
        for (int nt = 0; nt < kON; ++nt)
            o[nt][0] = o[nt][1] = o[nt][2] = o[nt][3] = 0.f;

        for (; x < piece_end; ++x) {
            const int t0 = int(x - sp.seg_start) * kDecodeTokens;
            const int nvalid = min(kDecodeTokens, n - t0);
            const bool ok = mbar_wait_warp(&full[stage], phase, misc, a.err);
            if (need_q) {
                const uint8_t* qs = smem + Lay::kQ + stage * Lay::kQStageBytes +
                                    tw * Lay::kHalves * Lay::kQHalfBytes;
#pragma unroll
                for (int kk = 0; kk < kKS; ++kk) {
                    const int r = lane & 15;
                    const int ch = 2 * kk + (lane >> 4);   // 16-byte chunk along D
                    ldsm_x4(smem_u32(qs + (ch >> 3) * Lay::kQHalfBytes + r * 128 +
                                     (((ch & 7) ^ (r & 7)) << 4)),
                            qa[kk][0], qa[kk][1], qa[kk][2], qa[kk][3]);
                }
                need_q = false;
            }
            bool wrote = false;
            if (nvalid > 0 && nvalid < kDecodeTokens) {
                // Zero the V rows past the context: P is 0 there, but 0 * NaN
                // is not. One row tile per segment: each warp zeroes its own
                // columns. Several: the warps of different tiles read the same
                // columns, so the four warps zero disjoint chunks and meet at a
                // barrier (reached by all of them, whatever their waits gave).
                if constexpr (TG == 1) {
                    if (ok) {
                        constexpr int kChunks = kCols / 8;  // 16-byte chunks per row
                        const int nz = (kDecodeTokens - nvalid) * kChunks;
                        for (int idx = lane; idx < nz; idx += 32) {
                            const int r = nvalid + idx / kChunks;
                            const int ch = col0 / 8 + idx % kChunks;
                            *reinterpret_cast<uint4*>(v_half(stage, ch >> 3) + r * 128 +
                                                      (((ch & 7) ^ (r & swz)) << 4)) =
                                make_uint4(0, 0, 0, 0);
                        }
                        wrote = true;
                    }
                    __syncwarp();
                } else {
                    if (ok) {
                        constexpr int kChunks = D / 8;
                        const int nz = (kDecodeTokens - nvalid) * kChunks;
                        for (int idx = threadIdx.x; idx < nz; idx += kConsumerThreads) {
                            const int r = nvalid + idx / kChunks;
                            const int ch = idx % kChunks;
                            *reinterpret_cast<uint4*>(v_half(stage, ch >> 3) + r * 128 +
                                                      (((ch & 7) ^ (r & swz)) << 4)) =
                                make_uint4(0, 0, 0, 0);
                        }
                        wrote = true;
                    }
                    named_barrier_sync(1, kConsumerThreads);
                }
            }
            if (ok && nvalid > 0 && live_tile) {
                // S = Q K^T for all 64 tokens (8 n-tiles of 8 tokens).
                float sc[kSN][4];
#pragma unroll
                for (int nt = 0; nt < kSN; ++nt)
                    sc[nt][0] = sc[nt][1] = sc[nt][2] = sc[nt][3] = 0.f;
                {
                    const int trl = (lane & 7) + ((lane >> 4) << 3);
                    const int chsel = (lane >> 3) & 1;
#pragma unroll
                    for (int kk = 0; kk < kKS; ++kk) {
                        const int ch = 2 * kk + chsel;
#pragma unroll
                        for (int tq = 0; tq < kSN / 2; ++tq) {
                            const int tr = tq * 16 + trl;
                            uint32_t b0, b1, b2, b3;
                            ldsm_x4(smem_u32(k_half(stage, ch >> 3) + tr * 128 +
                                             (((ch & 7) ^ (tr & swz)) << 4)),
                                    b0, b1, b2, b3);
                            mma_bf16_16816(sc[2 * tq], qa[kk], b0, b1);
                            mma_bf16_16816(sc[2 * tq + 1], qa[kk], b2, b3);
                        }
                    }
                }
                // Mask (select to -inf, never multiply) only where some row's
                // last visible position falls inside this granule.
                if (t0 + kDecodeTokens - 1 > lim_min) {
#pragma unroll
                    for (int nt = 0; nt < kSN; ++nt)
#pragma unroll
                        for (int j = 0; j < 4; ++j) {
                            const int tok = t0 + nt * 8 + 2 * quad + (j & 1);
                            if (tok > lim[j >> 1])
                                sc[nt][j] = -INFINITY;
                        }
                }
                // Online softmax in the log2 domain: m_run is kept scaled
                // (scale * log2 e > 0 preserves the order); p = 2^(c s - m) is
                // one FFMA and one ex2.
                float mx[2] = {-INFINITY, -INFINITY};
#pragma unroll
                for (int nt = 0; nt < kSN; ++nt) {
                    mx[0] = fmaxf(mx[0], fmaxf(sc[nt][0], sc[nt][1]));
                    mx[1] = fmaxf(mx[1], fmaxf(sc[nt][2], sc[nt][3]));
                }
                float mu[2], mn[2];
                bool changed = false;
#pragma unroll
                for (int rr = 0; rr < 2; ++rr) {
                    mx[rr] = fmaxf(mx[rr], __shfl_xor_sync(0xffffffffu, mx[rr], 1));
                    mx[rr] = fmaxf(mx[rr], __shfl_xor_sync(0xffffffffu, mx[rr], 2));
                    mn[rr] = fmaxf(m_run[rr], mx[rr] * a.scale_log2);
                    changed |= mn[rr] != m_run[rr];
                    mu[rr] = mn[rr] == -INFINITY ? 0.f : mn[rr];
                }
                if (__any_sync(0xffffffffu, changed)) {
                    // Rescale only when a running max moved: corr = 2^(m_old -
                    // m_new), exactly 1 for rows whose max did not move.
                    float corr[2];
#pragma unroll
                    for (int rr = 0; rr < 2; ++rr) {
                        corr[rr] = mn[rr] == m_run[rr] ? 1.f : fast_exp2(m_run[rr] - mu[rr]);
                        m_run[rr] = mn[rr];
                        l_run[rr] *= corr[rr];
                    }
#pragma unroll
                    for (int nt = 0; nt < kON; ++nt) {
                        o[nt][0] *= corr[0];
                        o[nt][1] *= corr[0];
                        o[nt][2] *= corr[1];
                        o[nt][3] *= corr[1];
                    }
                }
                uint32_t pa[kSN / 2][4];
#pragma unroll
                for (int nt = 0; nt < kSN; ++nt) {
                    float p[4];
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        p[j] = fast_exp2(fmaf(sc[nt][j], a.scale_log2, -mu[j >> 1]));
                        l_run[j >> 1] += p[j];
                    }
                    pa[nt >> 1][(nt & 1) * 2 + 0] = pack_bf16x2(p[0], p[1]);
                    pa[nt >> 1][(nt & 1) * 2 + 1] = pack_bf16x2(p[2], p[3]);
                }
                // O[:, col0 .. col0 + kCols) += P V; ldmatrix.trans gives the
                // k-major V fragments.
                {
                    const int trl = (lane & 7) + (((lane >> 3) & 1) << 3);
                    const int chsel = lane >> 4;
#pragma unroll
                    for (int kt = 0; kt < kSN / 2; ++kt) {
                        const int tr = kt * 16 + trl;
#pragma unroll
                        for (int jj = 0; jj < kON / 2; ++jj) {
                            const int ch = col0 / 8 + 2 * jj + chsel;
                            uint32_t b0, b1, b2, b3;
                            ldsm_x4_trans(smem_u32(v_half(stage, ch >> 3) + tr * 128 +
                                                   (((ch & 7) ^ (tr & swz)) << 4)),
                                          b0, b1, b2, b3);
                            mma_bf16_16816(o[2 * jj], pa[kt], b0, b1);
                            mma_bf16_16816(o[2 * jj + 1], pa[kt], b2, b3);
                        }
                    }
                }
            }
            if (wrote)
                fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0)
                mbar_arrive(&empty[stage]);
            if (++stage == kStages) {
                stage = 0;
                phase ^= 1u;
            }
        }

        // ---- end of a piece: every warp holds identical (m, l) and its own
        // output columns.
#pragma unroll
        for (int rr = 0; rr < 2; ++rr) {
            l_run[rr] += __shfl_xor_sync(0xffffffffu, l_run[rr], 1);
            l_run[rr] += __shfl_xor_sync(0xffffffffu, l_run[rr], 2);
        }
        // The segment lies inside this block's range: no other block holds a
        // piece of it.
        const bool single = a.whole_segments ||
                            (sp.seg_start >= x_begin && sp.seg_start + sp.seg_len <= x_end);
        const bool aborted = misc[0] != 0;

        if (!aborted && single) {
#pragma unroll
            for (int rr = 0; rr < 2; ++rr) {
                const int64_t orow = out_row(sp, row0 + rr * 8);
                if (orow < 0)
                    continue;
                const float inv = l_run[rr] > 0.f ? 1.f / l_run[rr] : 0.f;
                uint16_t* dst = a.out + orow * D + col0 + 2 * quad;
#pragma unroll
                for (int nt = 0; nt < kON; ++nt)
                    *reinterpret_cast<uint32_t*>(dst + nt * 8) =
                        pack_bf16x2(o[nt][2 * rr] * inv, o[nt][2 * rr + 1] * inv);
            }
        } else if (!aborted) {
            // A segment that straddles blocks: leave this block's partial
            // (m, l, acc) of every row tile for the merge pass.
            float* slot = a.partials + (int64_t(sp.seg) + cta) * kSlotFloats + tw * kTileFloats;
#pragma unroll
            for (int rr = 0; rr < 2; ++rr) {
                const int rw = row0 + rr * 8;
                if (out_row(sp, rw) < 0)
                    continue;  // padding rows of the tile carry nothing
                if (warp % kWPT == 0 && quad == 0) {
                    slot[rw] = m_run[rr];
                    slot[kDecodeRows + rw] = l_run[rr];
                }
                float* dst = slot + 2 * kDecodeRows + rw * D + col0 + 2 * quad;
#pragma unroll
                for (int nt = 0; nt < kON; ++nt)
                    *reinterpret_cast<float2*>(dst + nt * 8) =
                        make_float2(o[nt][2 * rr], o[nt][2 * rr + 1]);
            }
        }

    }
    }
}

// Merge pass over the segments that straddle decode blocks: one block per
// segment (blocks of the other segments return at once). Its per-segment
// arithmetic repeats the decode kernel's partition, on the inputs only; the
// partial states are read after the decode grid has completed.
// Thread -> (row tid / 16, columns c0 .. c0 + D/16) of each of the segment's
// row tiles in turn: M = max m_k, l = sum l_k 2^(m_k - M),
// o = sum acc_k 2^(m_k - M) / l, as one running pass over the pieces with
// up to eight of them in flight.
constexpr int kMergeThreads = 256;
template <int D>
__global__ void __launch_bounds__(kMergeThreads) decode_merge_kernel(const DecodeArgs a, int decode_grid)
{
    constexpr int kTileFloats = kDecodeRows * (D + 2);
    constexpr int kCols = D / 16;              // output columns per thread (4 or 8)
    constexpr int kVec = kCols / 4;            // float4 per piece and thread
    constexpr int kFly = 8;                    // pieces in flight
    const int64_t slot_floats = int64_t(a.TG) * kTileFloats;
    __shared__ long long red[2][kMergeThreads / 32];
    // The next kernel in the stream may be scheduled now; it still waits for
    // this one to complete before it reads or writes anything.
    grid_launch_dependents();
    const int tid = threadIdx.x;
    const int seg = blockIdx.x;
    const int per_req = a.H_kv * a.MS;
    const int b = seg / per_req, hm = seg - b * per_req;
    const int cap = a.max_pages * a.ps;
    auto granules = [&](int q) {
        int n = a.context_lens[q];
        n = n < 0 ? 0 : (n > cap ? cap : n);
        return max(1, (n + kDecodeTokens - 1) / kDecodeTokens);
    };
    long long before = 0, total = 0;
    for (int q = tid; q < a.B; q += blockDim.x) {
        const long long g = (long long)granules(q) * per_req;
        total += g;
        if (q < b)
            before += g;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        total += __shfl_xor_sync(0xffffffffu, total, o);
        before += __shfl_xor_sync(0xffffffffu, before, o);
    }
    if ((tid & 31) == 0) {
        red[0][tid >> 5] = total;
        red[1][tid >> 5] = before;
    }
    __syncthreads();
    total = before = 0;
#pragma unroll
    for (int w = 0; w < kMergeThreads / 32; ++w) {
        total += red[0][w];
        before += red[1][w];
    }
    const int gb = granules(b);
    const int64_t seg_start = before + int64_t(hm) * gb;
    const int64_t units = total + int64_t(a.piece_units) * a.B * per_req;
    const int64_t grid = int64_t(decode_grid) < units ? int64_t(decode_grid) : units;
    const int64_t u0 = seg_start + int64_t(a.piece_units) * (seg + 1);
    const int64_t first = block_of_unit(u0, units, grid);
    const int64_t last = block_of_unit(u0 + gb - 1, units, grid);
    if (first == last)
        return;  // finished and written by one decode block
    grid_dependency_wait();  // the decode grid has completed: its partials are visible

    const int r = tid >> 4;
    const int c0 = (tid & 15) * kCols;
    const int ms = hm % a.MS, h = hm / a.MS;
    const int np = int(last - first) + 1;
    for (int t = 0; t < a.TG; ++t) {
        const int rg = (ms * a.TG + t) * kDecodeRows + r;
        if (rg >= a.R)
            break;   // this and every later tile row are padding
        const int g = rg / a.L, i = rg - g * a.L;
        const int64_t orow = (int64_t(b) * a.H_q + h * a.G + g) * a.L + i;
        const float* base = a.partials + (int64_t(seg) + first) * slot_floats + t * kTileFloats;
        // M' = max(M, m_k), l = l 2^(M - M') + l_k 2^(m_k - M'), likewise o
        // (the pieces in order, so repeated calls give the same bits).
        float Mx = -INFINITY, L2 = 0.f;
        float fin[kCols];
#pragma unroll
        for (int c = 0; c < kCols; ++c)
            fin[c] = 0.f;
        for (int k0 = 0; k0 < np; k0 += kFly) {
            float mk[kFly], lk[kFly];
            float4 v[kFly][kVec];
#pragma unroll
            for (int u = 0; u < kFly; ++u) {
                const bool live = k0 + u < np;
                const float* sk = base + int64_t(live ? k0 + u : 0) * slot_floats;
                mk[u] = live ? __ldcg(sk + r) : -INFINITY;
                lk[u] = live ? __ldcg(sk + kDecodeRows + r) : 0.f;
                const float4* src =
                    reinterpret_cast<const float4*>(sk + 2 * kDecodeRows + r * D + c0);
#pragma unroll
                for (int c = 0; c < kVec; ++c)
                    v[u][c] = live ? __ldcg(src + c) : make_float4(0.f, 0.f, 0.f, 0.f);
            }
#pragma unroll
            for (int u = 0; u < kFly; ++u) {
                if (mk[u] == -INFINITY)
                    continue;  // absent piece, or no visible key in it
                const float Mn = fmaxf(Mx, mk[u]);
                const float co = Mx == -INFINITY ? 0.f : fast_exp2(Mx - Mn);
                const float cn = fast_exp2(mk[u] - Mn);
                Mx = Mn;
                L2 = L2 * co + lk[u] * cn;
#pragma unroll
                for (int c = 0; c < kVec; ++c) {
                    fin[4 * c] = fin[4 * c] * co + cn * v[u][c].x;
                    fin[4 * c + 1] = fin[4 * c + 1] * co + cn * v[u][c].y;
                    fin[4 * c + 2] = fin[4 * c + 2] * co + cn * v[u][c].z;
                    fin[4 * c + 3] = fin[4 * c + 3] * co + cn * v[u][c].w;
                }
            }
        }
        const float inv = L2 > 0.f ? 1.f / L2 : 0.f;
        uint16_t* dst = a.out + orow * D + c0;
#pragma unroll
        for (int c = 0; c < kCols; c += 4)   // 4 bf16 (8 bytes) at a time
            *reinterpret_cast<uint2*>(dst + c) =
                make_uint2(pack_bf16x2(fin[c + 0] * inv, fin[c + 1] * inv),
                           pack_bf16x2(fin[c + 2] * inv, fin[c + 3] * inv));
    }
}

}  // namespace

size_t decode_smem_bytes(int D, int B, bool fp8, int TG)
{
    if (fp8)
        return Layout<128, true>::bytes(B);
    if (D == 64)
        return TG == 4 ? Layout<64, false, 4>::bytes(B)
             : TG == 2 ? Layout<64, false, 2>::bytes(B) : Layout<64>::bytes(B);
    return TG == 4 ? Layout<128, false, 4>::bytes(B)
         : TG == 2 ? Layout<128, false, 2>::bytes(B) : Layout<128>::bytes(B);
}

int decode_max_grid(int sm_count) { return 2 * sm_count; }

size_t decode_workspace_bytes(int64_t nseg, int grid_max, int D, int TG)
{
    const size_t slots = size_t(nseg) + size_t(grid_max);
    return slots * size_t(TG) * kDecodeRows * (D + 2) * 4;
}

namespace {

using DecodeKernel = void (*)(CUtensorMap, CUtensorMap, CUtensorMap, DecodeArgs);

// The instantiation for (head_dim, e4m3 pages, row tiles per segment), with
// its index in the table of raised shared-memory limits.
DecodeKernel decode_kernel_for(int D, bool fp8, int TG, int* index)
{
    if (fp8) {
        *index = 0;
        return decode_kernel<128, true>;
    }
    const int t = TG == 4 ? 2 : TG == 2 ? 1 : 0;
    *index = 1 + (D == 64 ? 0 : 3) + t;
    if (D == 64)
        return t == 2 ? decode_kernel<64, false, 4> : t == 1 ? decode_kernel<64, false, 2>
                                                              : decode_kernel<64>;
    return t == 2 ? decode_kernel<128, false, 4> : t == 1 ? decode_kernel<128, false, 2>
                                                           : decode_kernel<128>;
}

}  // namespace

cudaError_t launch_decode(const CUtensorMap& key_map, const CUtensorMap& value_map,
                          const CUtensorMap& q_map, const DecodeArgs& a, int grid, int device,
                          cudaStream_t stream)
{
    // The dynamic shared-memory limit is raised once per (device, kernel)
    // and only grows.
    constexpr int kMaxDev = 64;
    static std::atomic<int> smem_set[kMaxDev][7];
    const bool fp8 = a.fp8 != 0;
    if ((fp8 && (a.D != 128 || a.TG != 1)) || (a.TG != 1 && a.TG != 2 && a.TG != 4))
        return cudaErrorInvalidValue;
    const int smem = int(decode_smem_bytes(a.D, a.B, fp8, a.TG));
    int di = 0;
    const DecodeKernel kern = decode_kernel_for(a.D, fp8, a.TG, &di);
    if (device < 0 || device >= kMaxDev)
        return cudaErrorInvalidDevice;
    if (smem_set[device][di].load(std::memory_order_relaxed) < smem) {
        cudaError_t e = cudaFuncSetAttribute(reinterpret_cast<const void*>(kern),
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess)
            return e;
        smem_set[device][di].store(smem, std::memory_order_relaxed);
    }
    // Both kernels are launched with programmatic stream serialization: each
    // may be scheduled before its predecessor in the stream has finished and
    // waits for it (griddepcontrol.wait) before touching its data.
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
    cudaError_t e = cudaLaunchKernelEx(&cfg, kern, key_map, value_map, q_map, a);
    if (e != cudaSuccess || a.whole_segments)
        return e;
    DecodeArgs ma = a;
    ma.piece_units = piece_units(fp8);
    cudaLaunchConfig_t mcfg = cfg;
    mcfg.gridDim = dim3(unsigned(int64_t(a.B) * a.H_kv * a.MS));
    mcfg.blockDim = dim3(kMergeThreads);
    mcfg.dynamicSmemBytes = 0;
    return a.D == 64 ? cudaLaunchKernelEx(&mcfg, decode_merge_kernel<64>, ma, grid)
                     : cudaLaunchKernelEx(&mcfg, decode_merge_kernel<128>, ma, grid);
}

}  // namespace pa
