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
//   * Per block: one producer warp resolves each page id once per page
//     (address translation hoisted per TMA box) and issues TMA tile loads of
//     whole page slices into a 3-stage shared-memory ring (128B swizzle);
//     four consumer warps each take 16 tokens of a granule and run
//     S = Q K^T and O += P V on the tensor cores (mma.sync m16n8k16, bf16 in,
//     fp32 accumulate) with the online-softmax recurrence in registers
//     (running max, running sum, rescaled output; Week 3 Day 4, "Task 2").
//   * At the end of a segment piece the four warps merge their (m, l, O)
//     through shared memory. A segment that one block finished alone is
//     normalised and written; otherwise the block writes its partial state,
//     and the last block to finish the segment (an atomic ticket, no waiting
//     on other blocks) merges all partials: M = max m_s,
//     l = sum l_s 2^(m_s - M), o = sum acc_s 2^(m_s - M) / l.
//   * Scores live in the log2 domain (scale * log2(e) folded into one
//     multiply) so every exponential is one exp2f.
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

constexpr int kStages = 3;
constexpr int kConsumerWarps = 4;
constexpr int kConsumerThreads = 32 * kConsumerWarps;
constexpr int kThreads = kConsumerThreads + 32;
constexpr int kConsumerBarrier = 1;  // named barrier id for the consumer warps

template <int D>
struct Layout {
    static constexpr int kHalves = D / 64;                   // 128-byte column blocks
    static constexpr int kHalfBytes = kDecodeTokens * 128;   // 64 rows x 128 B
    static constexpr int kStageBytes = kHalves * kHalfBytes; // K (or V) of one granule
    static constexpr int kK = 0;
    static constexpr int kV = kK + kStages * kStageBytes;
    static constexpr int kQ = kV + kStages * kStageBytes;    // [16][D] bf16, swizzled
    static constexpr int kML = kQ + kDecodeRows * D * 2;     // [warps][2][16] float
    static constexpr int kBar = kML + kConsumerWarps * 2 * kDecodeRows * 4;
    static constexpr int kMisc = kBar + 2 * kStages * 8;     // abort flag, ticket, test barrier
    static constexpr int kPrefix = kMisc + 16;               // [B + 1] int32
    static size_t bytes(int B) { return kPrefix + size_t(B + 1) * 4 + 1024; }
    static_assert(kStageBytes * 2 >= 4 * kDecodeRows * D * 4,
                  "merge scratch must fit in one stage");
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
    int b, h, mt, seg;
    int64_t seg_start;  // first granule of the segment in the stream
    int seg_len;        // granules in the segment
};

// Locates granule x of the stream. pre[b] = first granule of request b.
__device__ __forceinline__ SegmentPos locate(const int32_t* pre, int B, int per_req, int MT,
                                             int64_t x)
{
    int lo = 0, hi = B - 1;
    while (lo < hi) {  // largest b with pre[b] <= x
        int mid = (lo + hi + 1) >> 1;
        if (pre[mid] <= x)
            lo = mid;
        else
            hi = mid - 1;
    }
    SegmentPos s;
    s.b = lo;
    const int gb = (pre[lo + 1] - pre[lo]) / per_req;
    const int r = int(x - pre[lo]);
    const int hm = r / gb;
    s.h = hm / MT;
    s.mt = hm - s.h * MT;
    s.seg = lo * per_req + hm;
    s.seg_start = pre[lo] + int64_t(hm) * gb;
    s.seg_len = gb;
    return s;
}

// Block index that processes granule x when `total` granules are split over
// `grid` blocks as [floor(i*total/grid), floor((i+1)*total/grid)).
__device__ __forceinline__ int64_t block_of(int64_t x, int64_t total, int64_t grid)
{
    return ((x + 1) * grid - 1) / total;
}

template <int D>
__global__ void __launch_bounds__(kThreads, 2)
    decode_kernel(const __grid_constant__ CUtensorMap key_map,
                  const __grid_constant__ CUtensorMap value_map, const DecodeArgs a)
{
    using Lay = Layout<D>;
    constexpr int kNT = D / 8;   // n-tiles of 8 output columns
    constexpr int kKS = D / 16;  // k-steps of 16 over the head dimension

    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    int32_t* pre = reinterpret_cast<int32_t*>(smem + Lay::kPrefix);
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + Lay::kBar);
    uint64_t* empty = full + kStages;
    volatile int* misc = reinterpret_cast<volatile int*>(smem + Lay::kMisc);
    float* ml = reinterpret_cast<float*>(smem + Lay::kML);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int per_req = a.H_kv * a.MT;
    const int cap = a.max_pages * a.ps;

    // ---- granule prefix over requests (one warp) ---------------------------
    if (warp == 0) {
        int carry = 0;
        if (lane == 0)
            pre[0] = 0;
        for (int base = 0; base < a.B; base += 32) {
            const int b = base + lane;
            int g = 0;
            if (b < a.B) {
                const int n = clamp_context(a.context_lens[b], cap, a.err);
                g = max(1, (n + kDecodeTokens - 1) / kDecodeTokens) * per_req;
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
    uint64_t* never = reinterpret_cast<uint64_t*>(smem + Lay::kMisc + 8);
    if (threadIdx.x == 0) {
        misc[0] = 0;
        misc[1] = 0;
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], kConsumerWarps);
        }
        mbar_init(never, 1);
        fence_barrier_init();
        if (a.debug_unset_wait && blockIdx.x == 0) {
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
    }
    __syncthreads();

    const int64_t total = pre[a.B];
    const int64_t cta = blockIdx.x;
    // The stream is split over min(gridDim.x, total) blocks so that every
    // block in use owns at least one granule; a segment spanning blocks
    // first..last then has exactly last - first + 1 pieces.
    const int64_t grid = a.whole_segments ? int64_t(gridDim.x)
                                          : (int64_t(gridDim.x) < total ? int64_t(gridDim.x) : total);
    if (cta >= grid)
        return;
    int64_t x_begin, x_end;
    if (a.whole_segments) {
        // Whole segments per block: segments [s0, s1) of nseg.
        const int64_t nseg = int64_t(a.B) * per_req;
        const int64_t s0 = cta * nseg / grid, s1 = (cta + 1) * nseg / grid;
        if (s0 >= s1)
            return;
        auto seg_first = [&](int64_t s) -> int64_t {
            if (s >= nseg)
                return total;
            const int b = int(s / per_req), hm = int(s % per_req);
            const int gb = (pre[b + 1] - pre[b]) / per_req;
            return pre[b] + int64_t(hm) * gb;
        };
        x_begin = seg_first(s0);
        x_end = seg_first(s1);
    } else {
        x_begin = cta * total / grid;
        x_end = (cta + 1) * total / grid;
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
        if (lane == 0) {
            prefetch_tensormap(&key_map);
            prefetch_tensormap(&value_map);
        }
        const uint64_t policy = l2_policy_evict_first();
        int stage = 0;
        uint32_t phase = 0;
        for (int64_t x = x_begin; x < x_end; ++x) {
            const SegmentPos sp = locate(pre, a.B, per_req, a.MT, x);
            const int n = clamp_context(a.context_lens[sp.b], cap, a.err);
            const int t0 = int(x - sp.seg_start) * kDecodeTokens;
            const int nvalid = min(kDecodeTokens, n - t0);
            const bool ok = mbar_wait_bounded(&empty[stage], phase ^ 1u, misc, a.err);
            if (ok && nvalid > 0) {
                const int box = a.box_rows;
                const int nbox = (nvalid + box - 1) / box;
                const uint32_t bytes = uint32_t(nbox) * box * 128u * Lay::kHalves * 2u;
                if (lane == 0)
                    mbar_arrive_expect_tx(&full[stage], bytes);
                __syncwarp();
                const int32_t* bt = a.block_table + int64_t(sp.b) * a.max_pages;
                for (int j = lane; j < nbox; j += 32) {
                    const int tok = t0 + j * box;
                    const int lp = tok / a.ps;
                    const int slot0 = tok - lp * a.ps;
                    int phys = bt[lp];
                    if (unsigned(phys) >= unsigned(a.num_pages)) {
                        atomicOr(a.err, PA_DEVERR_PAGE_ID_BIT);
                        phys = 0;
                    }
                    const int row = (phys * a.H_kv + sp.h) * a.ps + slot0;
                    const int dst = j * box * 128;
#pragma unroll
                    for (int hf = 0; hf < Lay::kHalves; ++hf) {
                        tma_load_2d(k_half(stage, hf) + dst, &key_map, hf * 64, row, &full[stage],
                                    policy);
                        tma_load_2d(v_half(stage, hf) + dst, &value_map, hf * 64, row,
                                    &full[stage], policy);
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
        }
        return;
    }

    // ===================== consumer warps ===================================
    const int tid = threadIdx.x;  // 0..127
    const int swz = a.swz;        // stage layout: chunk ^ (row & 7) when swizzled
    const int row0 = lane >> 2;   // fragment rows row0 and row0 + 8
    const int quad = lane & 3;
    uint8_t* q_smem = smem + Lay::kQ;
    int stage = 0;
    uint32_t phase = 0;

    int64_t x = x_begin;
    while (x < x_end) {
        const SegmentPos sp = locate(pre, a.B, per_req, a.MT, x);
        const int64_t piece_end = min(x_end, sp.seg_start + sp.seg_len);
        const int n = clamp_context(a.context_lens[sp.b], cap, a.err);

        // ---- Q tile (16 rows x D) into shared memory, 16-byte chunks swizzled
        for (int c = tid; c < kDecodeRows * kNT; c += kConsumerThreads) {
            const int r = c / kNT, ch = c - r * kNT;
            const int rg = sp.mt * kDecodeRows + r;
            uint4 v = make_uint4(0, 0, 0, 0);
            if (rg < a.R) {
                const int g = rg / a.L, i = rg - g * a.L;
                const int hq = sp.h * a.G + g;
                const uint16_t* src =
                    a.q + ((int64_t(sp.b) * a.H_q + hq) * a.L + i) * D + ch * 8;
                v = *reinterpret_cast<const uint4*>(src);
            }
            *reinterpret_cast<uint4*>(q_smem + r * D * 2 + ((ch ^ (r & 7)) << 4)) = v;
        }
        named_barrier_sync(kConsumerBarrier, kConsumerThreads);
        uint32_t qa[kKS][4];
#pragma unroll
        for (int kk = 0; kk < kKS; ++kk) {
            const int r = lane & 15;
            const int ch = 2 * kk + (lane >> 4);
            ldsm_x4(smem_u32(q_smem + r * D * 2 + ((ch ^ (r & 7)) << 4)), qa[kk][0], qa[kk][1],
                    qa[kk][2], qa[kk][3]);
        }

        // Last visible position of this thread's two fragment rows.
        int lim[2];
#pragma unroll
        for (int rr = 0; rr < 2; ++rr) {
            const int rg = sp.mt * kDecodeRows + row0 + rr * 8;
            const int i = rg < a.R ? rg % a.L : a.L - 1;
            lim[rr] = a.causal ? min(n - a.L + i, n - 1) : n - 1;
        }

        float m_run[2] = {-INFINITY, -INFINITY};
        float l_run[2] = {0.f, 0.f};
        float o[kNT][4];
#pragma unroll
        for (int nt = 0; nt < kNT; ++nt)
            o[nt][0] = o[nt][1] = o[nt][2] = o[nt][3] = 0.f;

        int hold = 0;
        bool wrote_hold = false;
        for (; x < piece_end; ++x) {
            const int t0 = int(x - sp.seg_start) * kDecodeTokens;
            const int nvalid = min(kDecodeTokens, n - t0);
            const bool ok = mbar_wait_bounded(&full[stage], phase, misc, a.err);
            const int my0 = warp * 16;
            bool wrote = false;
            if (ok && my0 < nvalid) {
                if (nvalid < my0 + 16) {
                    // Zero V rows past the context: P is 0 there, but 0 * NaN is not.
                    const int z0 = nvalid;
                    const int nz = (my0 + 16 - z0) * kNT;
                    for (int idx = lane; idx < nz; idx += 32) {
                        const int r = z0 + idx / kNT, ch = idx % kNT;
                        *reinterpret_cast<uint4*>(v_half(stage, ch >> 3) + r * 128 +
                                                  ((ch & 7) << 4)) = make_uint4(0, 0, 0, 0);
                    }
                    wrote = true;
                    __syncwarp();
                }
                // S = Q K^T for tokens my0..my0+15 (two n-tiles of 8 tokens).
                float s[2][4];
#pragma unroll
                for (int nt = 0; nt < 2; ++nt)
                    s[nt][0] = s[nt][1] = s[nt][2] = s[nt][3] = 0.f;
                {
                    const int tr = my0 + (lane & 7) + ((lane >> 4) << 3);
                    const int chsel = (lane >> 3) & 1;
#pragma unroll
                    for (int kk = 0; kk < kKS; ++kk) {
                        const int ch = 2 * kk + chsel;
                        uint32_t b0, b1, b2, b3;
                        ldsm_x4(smem_u32(k_half(stage, ch >> 3) + tr * 128 +
                                         (((ch & 7) ^ (tr & swz)) << 4)),
                                b0, b1, b2, b3);
                        mma_bf16_16816(s[0], qa[kk], b0, b1);
                        mma_bf16_16816(s[1], qa[kk], b2, b3);
                    }
                }
                // Scale into the log2 domain and mask (select, never multiply).
                float mx[2] = {-INFINITY, -INFINITY};
#pragma unroll
                for (int nt = 0; nt < 2; ++nt) {
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        const int tok = t0 + my0 + nt * 8 + 2 * quad + (j & 1);
                        const int rr = j >> 1;
                        const float v = s[nt][j] * a.scale_log2;
                        s[nt][j] = tok <= lim[rr] ? v : -INFINITY;
                        mx[rr] = fmaxf(mx[rr], s[nt][j]);
                    }
                }
                float corr[2], mu[2];
#pragma unroll
                for (int rr = 0; rr < 2; ++rr) {
                    mx[rr] = fmaxf(mx[rr], __shfl_xor_sync(0xffffffffu, mx[rr], 1));
                    mx[rr] = fmaxf(mx[rr], __shfl_xor_sync(0xffffffffu, mx[rr], 2));
                    const float mn = fmaxf(m_run[rr], mx[rr]);
                    mu[rr] = mn == -INFINITY ? 0.f : mn;
                    corr[rr] = exp2f(m_run[rr] - mu[rr]);
                    m_run[rr] = mn;
                }
                float psum[2] = {0.f, 0.f};
#pragma unroll
                for (int nt = 0; nt < 2; ++nt) {
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        const float p = exp2f(s[nt][j] - mu[j >> 1]);
                        s[nt][j] = p;
                        psum[j >> 1] += p;
                    }
                }
#pragma unroll
                for (int rr = 0; rr < 2; ++rr)
                    l_run[rr] = l_run[rr] * corr[rr] + psum[rr];
#pragma unroll
                for (int nt = 0; nt < kNT; ++nt) {
                    o[nt][0] *= corr[0];
                    o[nt][1] *= corr[0];
                    o[nt][2] *= corr[1];
                    o[nt][3] *= corr[1];
                }
                uint32_t pa[4];
                pa[0] = pack_bf16x2(s[0][0], s[0][1]);
                pa[1] = pack_bf16x2(s[0][2], s[0][3]);
                pa[2] = pack_bf16x2(s[1][0], s[1][1]);
                pa[3] = pack_bf16x2(s[1][2], s[1][3]);
                // O += P V: ldmatrix.trans gives the k-major V fragments.
                {
                    const int tr = my0 + (lane & 7) + (((lane >> 3) & 1) << 3);
                    const int chsel = lane >> 4;
#pragma unroll
                    for (int jj = 0; jj < kNT / 2; ++jj) {
                        const int ch = 2 * jj + chsel;
                        uint32_t b0, b1, b2, b3;
                        ldsm_x4_trans(smem_u32(v_half(stage, ch >> 3) + tr * 128 +
                                               (((ch & 7) ^ (tr & swz)) << 4)),
                                      b0, b1, b2, b3);
                        mma_bf16_16816(o[2 * jj], pa, b0, b1);
                        mma_bf16_16816(o[2 * jj + 1], pa, b2, b3);
                    }
                }
            }
            if (x + 1 < piece_end) {
                if (wrote)
                    fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0)
                    mbar_arrive(&empty[stage]);
            } else {
                hold = stage;  // kept as merge scratch, released after the merge
                wrote_hold = wrote;
            }
            if (++stage == kStages) {
                stage = 0;
                phase ^= 1u;
            }
        }
        (void)wrote_hold;

        // ---- merge the four warps' states through the held stage -----------
#pragma unroll
        for (int rr = 0; rr < 2; ++rr) {
            l_run[rr] += __shfl_xor_sync(0xffffffffu, l_run[rr], 1);
            l_run[rr] += __shfl_xor_sync(0xffffffffu, l_run[rr], 2);
        }
        named_barrier_sync(kConsumerBarrier, kConsumerThreads);  // all done reading `hold`
        float* scratch = reinterpret_cast<float*>(warp < 2 ? k_half(hold, 0) : v_half(hold, 0)) +
                         (warp & 1) * kDecodeRows * D;
#pragma unroll
        for (int nt = 0; nt < kNT; ++nt) {
#pragma unroll
            for (int rr = 0; rr < 2; ++rr) {
                const int r = row0 + rr * 8;
                const int k2 = ((nt ^ (r & 7)) << 2) | quad;  // float2 index in the row
                *reinterpret_cast<float2*>(scratch + r * D + 2 * k2) =
                    make_float2(o[nt][2 * rr], o[nt][2 * rr + 1]);
            }
        }
        if (quad == 0) {
#pragma unroll
            for (int rr = 0; rr < 2; ++rr) {
                ml[(warp * 2 + 0) * kDecodeRows + row0 + rr * 8] = m_run[rr];
                ml[(warp * 2 + 1) * kDecodeRows + row0 + rr * 8] = l_run[rr];
            }
        }
        named_barrier_sync(kConsumerBarrier, kConsumerThreads);

        // Combine: thread -> (row, D/8 columns).
        const int r = tid >> 3;
        const int c0 = (tid & 7) * (D / 8);
        const int rg = sp.mt * kDecodeRows + r;
        float acc[D / 8];
        float Lsum = 0.f, M = -INFINITY;
        {
            float mw[kConsumerWarps], lw[kConsumerWarps];
#pragma unroll
            for (int w = 0; w < kConsumerWarps; ++w) {
                mw[w] = ml[(w * 2 + 0) * kDecodeRows + r];
                lw[w] = ml[(w * 2 + 1) * kDecodeRows + r];
                M = fmaxf(M, mw[w]);
            }
            const float Mu = M == -INFINITY ? 0.f : M;
#pragma unroll
            for (int c = 0; c < D / 8; ++c)
                acc[c] = 0.f;
#pragma unroll
            for (int w = 0; w < kConsumerWarps; ++w) {
                const float f = exp2f(mw[w] - Mu);
                Lsum += f * lw[w];
                const float* sw =
                    reinterpret_cast<const float*>(w < 2 ? k_half(hold, 0) : v_half(hold, 0)) +
                    (w & 1) * kDecodeRows * D + r * D;
#pragma unroll
                for (int c = 0; c < D / 8; c += 2) {
                    const int col = c0 + c;
                    const int nt = col >> 3, qd = (col & 7) >> 1;
                    const int k2 = ((nt ^ (r & 7)) << 2) | qd;
                    const float2 v = *reinterpret_cast<const float2*>(sw + 2 * k2);
                    acc[c] += f * v.x;
                    acc[c + 1] += f * v.y;
                }
            }
        }

        const int64_t nseg_blocks_first = a.whole_segments ? cta : block_of(sp.seg_start, total, grid);
        const int64_t nseg_blocks_last =
            a.whole_segments ? cta : block_of(sp.seg_start + sp.seg_len - 1, total, grid);
        const int npieces = int(nseg_blocks_last - nseg_blocks_first) + 1;
        const bool aborted = misc[0] != 0;

        auto store_out = [&](const float* v, float l) {
            if (rg >= a.R)
                return;
            const int g = rg / a.L, i = rg - g * a.L;
            const int hq = sp.h * a.G + g;
            uint16_t* dst = a.out + ((int64_t(sp.b) * a.H_q + hq) * a.L + i) * D + c0;
            const float inv = l > 0.f ? 1.f / l : 0.f;
#pragma unroll
            for (int c = 0; c < D / 8; c += 8) {
                uint4 w;
                w.x = pack_bf16x2(v[c + 0] * inv, v[c + 1] * inv);
                w.y = pack_bf16x2(v[c + 2] * inv, v[c + 3] * inv);
                w.z = pack_bf16x2(v[c + 4] * inv, v[c + 5] * inv);
                w.w = pack_bf16x2(v[c + 6] * inv, v[c + 7] * inv);
                *reinterpret_cast<uint4*>(dst + c) = w;
            }
        };

        if (npieces == 1) {
            if (!aborted)
                store_out(acc, Lsum);
        } else if (!aborted) {
            constexpr int kSlotFloats = kDecodeRows * (D + 2);
            float* slot = a.partials + (int64_t(sp.seg) + cta) * kSlotFloats;
            if ((tid & 7) == 0) {
                slot[r] = M;
                slot[kDecodeRows + r] = Lsum;
            }
            float* dst = slot + 2 * kDecodeRows + r * D + c0;
#pragma unroll
            for (int c = 0; c < D / 8; c += 4)
                *reinterpret_cast<float4*>(dst + c) =
                    make_float4(acc[c], acc[c + 1], acc[c + 2], acc[c + 3]);
            __threadfence();
            named_barrier_sync(kConsumerBarrier, kConsumerThreads);
            if (tid == 0) {
                const int t = atomicAdd(&a.counters[sp.seg], 1);
                misc[1] = (t == npieces - 1) ? 1 : 0;
            }
            named_barrier_sync(kConsumerBarrier, kConsumerThreads);
            if (misc[1]) {
                __threadfence();
                const float* base = a.partials + (int64_t(sp.seg) + nseg_blocks_first) * kSlotFloats;
                float Mx = -INFINITY;
                for (int k = 0; k < npieces; ++k)
                    Mx = fmaxf(Mx, __ldcg(base + int64_t(k) * kSlotFloats + r));
                const float Mu = Mx == -INFINITY ? 0.f : Mx;
                float L2 = 0.f;
                float fin[D / 8];
#pragma unroll
                for (int c = 0; c < D / 8; ++c)
                    fin[c] = 0.f;
                for (int k = 0; k < npieces; ++k) {
                    const float* sk = base + int64_t(k) * kSlotFloats;
                    const float f = exp2f(__ldcg(sk + r) - Mu);
                    L2 += f * __ldcg(sk + kDecodeRows + r);
                    const float4* src =
                        reinterpret_cast<const float4*>(sk + 2 * kDecodeRows + r * D + c0);
#pragma unroll
                    for (int c = 0; c < D / 8; c += 4) {
                        const float4 v = __ldcg(src + c / 4);
                        fin[c] += f * v.x;
                        fin[c + 1] += f * v.y;
                        fin[c + 2] += f * v.z;
                        fin[c + 3] += f * v.w;
                    }
                }
                store_out(fin, L2);
                if (tid == 0)
                    a.counters[sp.seg] = 0;
            }
        }
        named_barrier_sync(kConsumerBarrier, kConsumerThreads);  // scratch, Q and misc reuse
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0)
            mbar_arrive(&empty[hold]);
    }
}

}  // namespace

size_t decode_smem_bytes(int D, int B)
{
    return D == 64 ? Layout<64>::bytes(B) : Layout<128>::bytes(B);
}

int decode_max_grid(int sm_count) { return 2 * sm_count; }

size_t decode_workspace_bytes(int64_t nseg, int grid_max, int D)
{
    const size_t slots = size_t(nseg) + size_t(grid_max);
    return kCounterRegionBytes + slots * kDecodeRows * (D + 2) * 4;
}

cudaError_t launch_decode(const CUtensorMap& key_map, const CUtensorMap& value_map,
                          const DecodeArgs& a, int grid, int device, cudaStream_t stream)
{
    // The dynamic shared-memory limit is raised once per (device, head_dim)
    // and only grows.
    constexpr int kMaxDev = 64;
    static std::atomic<int> smem_set[kMaxDev][2];
    const int smem = int(decode_smem_bytes(a.D, a.B));
    const int di = a.D == 64 ? 0 : 1;
    if (device < 0 || device >= kMaxDev)
        return cudaErrorInvalidDevice;
    if (smem_set[device][di].load(std::memory_order_relaxed) < smem) {
        const void* fn = a.D == 64 ? reinterpret_cast<const void*>(decode_kernel<64>)
                                   : reinterpret_cast<const void*>(decode_kernel<128>);
        cudaError_t e =
            cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess)
            return e;
        smem_set[device][di].store(smem, std::memory_order_relaxed);
    }
    if (a.D == 64)
        decode_kernel<64><<<grid, kThreads, smem, stream>>>(key_map, value_map, a);
    else
        decode_kernel<128><<<grid, kThreads, smem, stream>>>(key_map, value_map, a);
    return cudaGetLastError();
}

}  // namespace pa
