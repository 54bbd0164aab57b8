// Device-side helpers: inline PTX for mbarriers, TMA tile loads, ldmatrix and
// warp-level bf16 MMA, plus bounded waits. sm_103a only.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <stdint.h>

#include "pa_internal.h"

namespace pa {

__device__ __forceinline__ uint32_t smem_u32(const void* p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t global_timer_ns()
{
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// a / b for 0 <= a, 0 < b. When both are below 2^24 (the usual case) the
// quotient comes from one fp32 division (a and b are exact in fp32, the
// estimate is within a few units of a / b) and is then corrected to the exact
// floor; an integer division is a long dependent instruction sequence (about
// 230 cycles for 32 bits, measured), and the block prologue and the piece
// ends lie on the call's critical path.
__device__ __forceinline__ int64_t udiv64(int64_t a, int64_t b)
{
    if (uint64_t(a) < (1ull << 24) && uint64_t(b) < (1ull << 24)) {
        int32_t q = int32_t(__fdividef(float(a), float(b)));
        int32_t r = int32_t(a) - q * int32_t(b);
        while (r < 0) {
            --q;
            r += int32_t(b);
        }
        while (r >= int32_t(b)) {
            ++q;
            r -= int32_t(b);
        }
        return q;
    }
    if (uint64_t(a) <= 0xffffffffull && uint64_t(b) <= 0xffffffffull)
        return int64_t(uint32_t(a) / uint32_t(b));
    return a / b;
}

// ---------------------------------------------------------------------------
// mbarrier

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
                 : "memory");
}

__device__ __forceinline__ void fence_barrier_init()
{
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(
                     smem_u32(bar)),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar)
{
    asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar))
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Waits for the phase of `bar` with the given parity to complete. The first
// wait of a block that runs out (kWaitLimitNs) records PA_DEVERR_TIMEOUT and
// sets `abort_flag` (shared memory); from then on the block's waits give up
// after kShortWaitLimitNs instead, which still lets copies that are really in
// flight land, and the block skips its output writes. Returns true when the
// phase completed.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity,
                                                  volatile int* abort_flag, unsigned* err)
{
    if (mbar_try_wait(bar, parity))
        return true;
    const uint64_t limit = *abort_flag ? kShortWaitLimitNs : kWaitLimitNs;
    const uint64_t t0 = global_timer_ns();
    for (uint32_t i = 1;; ++i) {
        if (mbar_try_wait(bar, parity))
            return true;
        if ((i & 15u) == 0 && global_timer_ns() - t0 > limit) {
            if (!*abort_flag) {
                *abort_flag = 1;
                atomicOr(err, PA_DEVERR_TIMEOUT_BIT);
            }
            return false;
        }
    }
}

// mbar_wait_bounded with the waiting loop marked unlikely, so that the
// common case of a thread whose every wait delays the tensor core (the MMA
// issuer), a phase that has already completed, stays one try_wait and a
// branch (the loop's set-up otherwise costs several times that per call).
__device__ __forceinline__ bool mbar_wait_lean(uint64_t* bar, uint32_t parity,
                                               volatile int* abort_flag, unsigned* err)
{
    if (__builtin_expect(mbar_try_wait(bar, parity), 1))
        return true;
    const uint64_t limit = *abort_flag ? kShortWaitLimitNs : kWaitLimitNs;
    const uint64_t t0 = global_timer_ns();
    for (uint32_t i = 1;; ++i) {
        if (mbar_try_wait(bar, parity))
            return true;
        if ((i & 15u) == 0 && global_timer_ns() - t0 > limit) {
            if (!*abort_flag) {
                *abort_flag = 1;
                atomicOr(err, PA_DEVERR_TIMEOUT_BIT);
            }
            return false;
        }
    }
}

// The same wait for a whole warp; the result is the same in every lane, so
// it can gate warp-collective code.
__device__ __forceinline__ bool mbar_wait_warp(uint64_t* bar, uint32_t parity,
                                               volatile int* abort_flag, unsigned* err)
{
    const bool ok = mbar_wait_bounded(bar, parity, abort_flag, err);
    return __all_sync(0xffffffffu, ok);
}

// 16 bytes global -> shared without a register round trip (cp.async, L2
// only); src_bytes < 16 fills the rest with zeros (0: no read at all).
__device__ __forceinline__ void cp_async_16(void* smem_dst, const void* gmem_src, uint32_t src_bytes)
{
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(smem_u32(smem_dst)),
                 "l"(gmem_src), "r"(src_bytes)
                 : "memory");
}
// Closes the group of this thread's cp.async issued since the last commit.
__device__ __forceinline__ void cp_async_commit()
{
    asm volatile("cp.async.commit_group;" ::: "memory");
}
// Waits until at most kPending of this thread's committed groups (the most
// recent ones) are still landing.
template <int kPending>
__device__ __forceinline__ void cp_async_wait_group()
{
    asm volatile("cp.async.wait_group %0;" ::"n"(kPending) : "memory");
}

// Orders this thread's generic-proxy shared-memory writes before later
// async-proxy (TMA) accesses of the same bytes.
__device__ __forceinline__ void fence_proxy_async_smem()
{
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ---------------------------------------------------------------------------
// TMA: 2-D tiled load global -> shared, completion counted on an mbarrier.

__device__ __forceinline__ void tma_load_2d(void* smem_dst, const CUtensorMap* map, int32_t x,
                                            int32_t y, uint64_t* bar, uint64_t policy)
{
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        ".L2::cache_hint [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(smem_u32(smem_dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar)), "l"(policy)
        : "memory");
}

// TMA: stores a 3-D box of `map` from shared memory (128B-swizzled like the
// map), in the thread's bulk group; elements outside the tensor are not
// written. The shared memory must not be rewritten before tma_store_wait_read.
__device__ __forceinline__ void tma_store_3d(const CUtensorMap* map, const void* smem_src, int32_t x,
                                             int32_t y, int32_t z)
{
    asm volatile(
        "cp.async.bulk.tensor.3d.global.shared::cta.tile.bulk_group [%0, {%2, %3, %4}], [%1];" ::"l"(
            reinterpret_cast<uint64_t>(map)),
        "r"(smem_u32(smem_src)), "r"(x), "r"(y), "r"(z)
        : "memory");
}
__device__ __forceinline__ void tma_store_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// The thread's committed stores have read their shared memory.
__device__ __forceinline__ void tma_store_wait_read()
{
    asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}
// The thread's committed stores are complete.
__device__ __forceinline__ void tma_store_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

// TMA: brings a 2-D tile of `map` into L2 (no shared memory, no completion).
__device__ __forceinline__ void tma_prefetch_l2_2d(const CUtensorMap* map, int32_t x, int32_t y)
{
    asm volatile("cp.async.bulk.prefetch.tensor.2d.L2.global.tile [%0, {%1, %2}];" ::"l"(
                     reinterpret_cast<uint64_t>(map)),
                 "r"(x), "r"(y)
                 : "memory");
}

// Release store / acquire load of a 64-bit flag at GPU scope.
__device__ __forceinline__ void st_release_gpu(unsigned long long* p, unsigned long long v)
{
    asm volatile("st.release.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}

__device__ __forceinline__ unsigned long long ld_relaxed_gpu(const unsigned long long* p)
{
    unsigned long long v;
    asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ unsigned long long ld_acquire_gpu(const unsigned long long* p)
{
    unsigned long long v;
    asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ uint64_t l2_policy_evict_first()
{
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}

__device__ __forceinline__ uint64_t l2_policy_evict_last()
{
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
    return p;
}

__device__ __forceinline__ void prefetch_tensormap(const CUtensorMap* map)
{
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// ---------------------------------------------------------------------------
// ldmatrix / mma.sync (bf16 in, fp32 accumulate)

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                        uint32_t& r3)
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}

__device__ __forceinline__ void ldsm_x4_trans(uint32_t addr, uint32_t& r0, uint32_t& r1,
                                              uint32_t& r2, uint32_t& r3)
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}

// D += A * B for one m16n8k16 tile. a: 4 regs (bf16x2), b: 2 regs, d: 4 floats.
__device__ __forceinline__ void mma_bf16_16816(float* d, const uint32_t* a, uint32_t b0,
                                               uint32_t b1)
{
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
        "{%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// 2^x with the hardware approximation (ex2.approx.ftz.f32: relative error
// about 2^-22, 2^-inf = +0).
__device__ __forceinline__ float fast_exp2(float x)
{
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// mma.sync m16n8k16, f16 x f16 -> fp32 (the FP8-page decode path: e4m3
// values are exact in f16).
__device__ __forceinline__ void mma_f16_16816(float* d, const uint32_t* a, uint32_t b0,
                                              uint32_t b1)
{
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Two e4m3 codes (bits 0-7 and 8-15 of w) -> two f16, the first in the lower
// half: one conversion instruction, exact for every code (every e4m3 value,
// subnormals included, is an f16 value; a NaN code gives NaN).
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint32_t w)
{
    uint32_t r;
    asm("{\n .reg .b16 lo, hi;\n mov.b32 {lo, hi}, %1;\n cvt.rn.f16x2.e4m3x2 %0, lo;\n}"
        : "=r"(r) : "r"(w));
    return r;
}
// The same for the codes in bits 16-31 of w.
__device__ __forceinline__ uint32_t e4m3x2_hi_to_f16x2(uint32_t w)
{
    uint32_t r;
    asm("{\n .reg .b16 lo, hi;\n mov.b32 {lo, hi}, %1;\n cvt.rn.f16x2.e4m3x2 %0, hi;\n}"
        : "=r"(r) : "r"(w));
    return r;
}

// Two fp32 -> two e4m3 codes (round to nearest even, saturated to +-448),
// the first in the lower byte.
__device__ __forceinline__ uint32_t f32x2_to_e4m3x2(float lo, float hi)
{
    return uint32_t(__nv_cvt_float2_to_fp8x2(make_float2(lo, hi), __NV_SATFINITE, __NV_E4M3));
}

// bf16 pair -> f16 pair (rounded to nearest; exact for magnitudes in f16's
// normal range).
__device__ __forceinline__ uint32_t bf16x2_to_f16x2(uint32_t v)
{
    const __half2 h = __floats2half2_rn(__uint_as_float(v << 16), __uint_as_float(v & 0xffff0000u));
    return *reinterpret_cast<const uint32_t*>(&h);
}

__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi)
{
    const __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<const uint32_t*>(&h);
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi)
{
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
}

// Programmatic dependent launch. wait: blocks until the grid this launch
// depends on (the previous kernel in the stream) has completed and its
// memory is visible; a kernel launched without the attribute returns at
// once. launch_dependents: lets the next kernel in the stream be scheduled.
__device__ __forceinline__ void grid_dependency_wait()
{
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

__device__ __forceinline__ void grid_launch_dependents()
{
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Named barrier among the first `threads` threads of the block.
__device__ __forceinline__ void named_barrier_sync(int id, int threads)
{
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

}  // namespace pa
