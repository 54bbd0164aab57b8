// Prefill over e4m3 page pools, first step: every K/V token a request can see
// is copied out of the e4m3 pool into bf16 pages of 128 tokens (the value of
// each code, exactly: e4m3 values are a subset of bf16's), which the
// tensor-core prefill kernels then read through a table of their own. The
// per-tensor scales are not applied here: k_scale goes into the softmax
// scale and v_scale into the output normalisation, so the scaled values are
// never rounded (Reading vLLM's PagedAttention Kernel, 3.2: the cache write
// path takes kv_cache_dtype, k_scale and v_scale).
//
// Why a copy and not a conversion inside the prefill pipeline: a prefill
// chunk reuses each K/V element G * L times on the tensor cores, so the copy
// (one e4m3 read and one bf16 write per visible element) is small next to the
// attention, and the prefill kernels keep their bf16 operand path unchanged.
//
// One block per (request, KV head, 128-token page of the copy); a thread
// converts 16-byte vectors of codes (16 elements of one token row) into two
// 16-byte bf16 vectors, so the reads of the pool's page slices and the writes
// of the copy are coalesced. Pages wholly past a request's context are not
// written (the prefill never reads them); rows past it in the last page are
// written as zeros.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <stdint.h>

#include "pa_device.cuh"
#include "pa_internal.h"

namespace pa {
namespace {

constexpr int kCopyRows = 128;   // tokens per page of the copy
constexpr int kRowCodes = 128;   // head_dim: bytes per e4m3 row

// Four e4m3 codes (one 32-bit word, lowest byte first) -> four bf16 (exact).
__device__ __forceinline__ uint2 e4m3x4_to_bf16x4(uint32_t w)
{
    uint32_t r[2];
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        const __half2_raw h = __nv_cvt_fp8x2_to_halfraw2(
            static_cast<__nv_fp8x2_storage_t>((w >> (16 * i)) & 0xFFFFu), __NV_E4M3);
        const float2 f = __half22float2(__half2(h));
        const __nv_bfloat162 b = __float22bfloat162_rn(f);
        r[i] = *reinterpret_cast<const uint32_t*>(&b);
    }
    return make_uint2(r[0], r[1]);
}

__global__ void __launch_bounds__(256) fp8_pages_to_bf16_kernel(const Fp8PagesArgs a)
{
    // Launched with programmatic stream serialization: wait for the previous
    // kernel in the stream (which may still write the pool or the tables).
    grid_dependency_wait();
    grid_launch_dependents();
    int64_t blk = blockIdx.x;
    const int p2 = int(blk % a.P2);
    blk /= a.P2;
    const int h = int(blk % a.H_kv);
    const int b = int(blk / a.H_kv);
    const int64_t page = int64_t(b) * a.P2 + p2;            // page of the copy
    if (h == 0 && threadIdx.x == 0)
        a.table_out[page] = int32_t(page);
    const int cap = min(a.max_pages * a.ps, a.P2 * kCopyRows);
    int n = a.context_lens[b];
    if (n < 0 || n > cap) {
        if (h == 0 && p2 == 0 && threadIdx.x == 0)
            atomicOr(a.err, PA_DEVERR_CONTEXT_LEN_BIT);
        n = n < 0 ? 0 : cap;
    }
    const int t0 = p2 * kCopyRows;
    if (t0 >= n)
        return;
    const int64_t out0 = (page * a.H_kv + h) * int64_t(kCopyRows) * kRowCodes;  // element offset
    const int32_t* bt = a.block_table + int64_t(b) * a.max_pages;
    constexpr int kVecs = kCopyRows * (kRowCodes / 16);       // 16-byte code vectors per tensor
    for (int idx = threadIdx.x; idx < kVecs; idx += blockDim.x) {
        const int r = idx >> 3, c = idx & 7;
        const int t = t0 + r;
        uint4 kc = make_uint4(0, 0, 0, 0), vc = make_uint4(0, 0, 0, 0);
        if (t < n) {
            const int lp = t / a.ps;
            int phys = bt[lp];
            if (unsigned(phys) >= unsigned(a.num_pages)) {
                atomicOr(a.err, PA_DEVERR_PAGE_ID_BIT);
                phys = 0;
            }
            const int64_t row = (int64_t(phys) * a.H_kv + h) * a.ps + (t - lp * a.ps);
            kc = *reinterpret_cast<const uint4*>(a.key_pages + row * kRowCodes + c * 16);
            vc = *reinterpret_cast<const uint4*>(a.value_pages + row * kRowCodes + c * 16);
        }
        const int64_t o = out0 + int64_t(r) * kRowCodes + c * 16;
        const uint2 k0 = e4m3x4_to_bf16x4(kc.x), k1 = e4m3x4_to_bf16x4(kc.y);
        const uint2 k2 = e4m3x4_to_bf16x4(kc.z), k3 = e4m3x4_to_bf16x4(kc.w);
        const uint2 v0 = e4m3x4_to_bf16x4(vc.x), v1 = e4m3x4_to_bf16x4(vc.y);
        const uint2 v2 = e4m3x4_to_bf16x4(vc.z), v3 = e4m3x4_to_bf16x4(vc.w);
        *reinterpret_cast<uint4*>(a.key_out + o) = make_uint4(k0.x, k0.y, k1.x, k1.y);
        *reinterpret_cast<uint4*>(a.key_out + o + 8) = make_uint4(k2.x, k2.y, k3.x, k3.y);
        *reinterpret_cast<uint4*>(a.value_out + o) = make_uint4(v0.x, v0.y, v1.x, v1.y);
        *reinterpret_cast<uint4*>(a.value_out + o + 8) = make_uint4(v2.x, v2.y, v3.x, v3.y);
    }
}

}  // namespace

int64_t fp8_copy_pages(int64_t max_context_len)
{
    const int64_t p = (max_context_len + kCopyRows - 1) / kCopyRows;
    return p > 0 ? p : 1;
}

cudaError_t launch_fp8_pages_to_bf16(const Fp8PagesArgs& a, cudaStream_t stream)
{
    const int64_t blocks = int64_t(a.B) * a.H_kv * a.P2;
    if (blocks <= 0 || blocks >= (int64_t(1) << 31))
        return cudaErrorInvalidValue;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(unsigned(blocks));
    cfg.blockDim = dim3(256);
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const cudaError_t e = cudaLaunchKernelEx(&cfg, fp8_pages_to_bf16_kernel, a);
    return e;
}

}  // namespace pa
