// Write path: scatter new K/V rows into the page pool by slot_mapping
// (Reading vLLM's PagedAttention Kernel, 3.2 "Writing into the cache").
//
// One thread moves one 16-byte vector (8 bf16) of one token's K or V row for
// one KV head: consecutive threads cover consecutive 16-byte pieces of a row,
// so both the read of the new rows and the write into the page slice are
// fully coalesced. The copy is bit-exact (no conversion); pages of e4m3 codes
// get the quantised rows instead.
#include <stdint.h>

#include "pa_device.cuh"
#include "pa_internal.h"

namespace pa {
namespace {

__global__ void __launch_bounds__(256) append_kernel(const AppendArgs a)
{
    // Launched with programmatic stream serialization: wait for the previous
    // kernel in the stream (which may still read the pool) before writing,
    // and let the attention kernel that follows be scheduled.
    grid_dependency_wait();
    grid_launch_dependents();
    const int vec_per_row = a.D / 8;
    const int64_t per_tensor = int64_t(a.B) * a.L_new * a.H_kv * vec_per_row;
    const int64_t total = 2 * per_tensor;
    for (int64_t t = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; t < total;
         t += int64_t(gridDim.x) * blockDim.x) {
        const bool is_v = t >= per_tensor;
        int64_t u = is_v ? t - per_tensor : t;
        const int c = int(u % vec_per_row);
        u /= vec_per_row;
        const int h = int(u % a.H_kv);
        u /= a.H_kv;
        const int i = int(u % a.L_new);
        const int b = int(u / a.L_new);
        const int64_t slot = a.slot_mapping[int64_t(b) * a.L_new + i];
        if (slot < 0)
            continue;  // padding token
        const int64_t page = slot / a.ps;
        const int64_t off = slot - page * a.ps;
        if (page >= a.num_pages) {
            if (c == 0 && h == 0 && !is_v)
                atomicOr(a.err, PA_DEVERR_SLOT_BIT);
            continue;
        }
        const int64_t src = ((int64_t(b) * a.H_kv + h) * a.L_new + i) * a.D + c * 8;
        const int64_t dst = ((page * a.H_kv + h) * a.ps + off) * a.D + c * 8;
        const uint16_t* s = is_v ? a.value : a.key;
        uint16_t* d = is_v ? a.value_pages : a.key_pages;
        *reinterpret_cast<uint4*>(d + dst) = *reinterpret_cast<const uint4*>(s + src);
    }
}

// The same scatter into pages of e4m3 codes: every element is stored as the
// code nearest to fp32(x) / scale (ties to even, saturated to +-448), one
// thread per 8 elements (16 bytes in, 8 bytes out).
__global__ void __launch_bounds__(256) append_fp8_kernel(const AppendArgs a)
{
    grid_dependency_wait();
    grid_launch_dependents();
    const int vec_per_row = a.D / 8;
    const int64_t per_tensor = int64_t(a.B) * a.L_new * a.H_kv * vec_per_row;
    const int64_t total = 2 * per_tensor;
    uint8_t* const kp = reinterpret_cast<uint8_t*>(a.key_pages);
    uint8_t* const vp = reinterpret_cast<uint8_t*>(a.value_pages);
    for (int64_t t = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; t < total;
         t += int64_t(gridDim.x) * blockDim.x) {
        const bool is_v = t >= per_tensor;
        int64_t u = is_v ? t - per_tensor : t;
        const int c = int(u % vec_per_row);
        u /= vec_per_row;
        const int h = int(u % a.H_kv);
        u /= a.H_kv;
        const int i = int(u % a.L_new);
        const int b = int(u / a.L_new);
        const int64_t slot = a.slot_mapping[int64_t(b) * a.L_new + i];
        if (slot < 0)
            continue;
        const int64_t page = slot / a.ps;
        const int64_t off = slot - page * a.ps;
        if (page >= a.num_pages) {
            if (c == 0 && h == 0 && !is_v)
                atomicOr(a.err, PA_DEVERR_SLOT_BIT);
            continue;
        }
        const int64_t src = ((int64_t(b) * a.H_kv + h) * a.L_new + i) * a.D + c * 8;
        const int64_t dst = ((page * a.H_kv + h) * a.ps + off) * a.D + c * 8;
        const uint4 x = *reinterpret_cast<const uint4*>((is_v ? a.value : a.key) + src);
        const float sc = is_v ? a.v_scale : a.k_scale;
        auto q2 = [&](uint32_t w) {   // two bf16 -> two e4m3 codes (16 bits)
            return f32x2_to_e4m3x2(__fdiv_rn(__uint_as_float(w << 16), sc),
                                   __fdiv_rn(__uint_as_float(w & 0xffff0000u), sc));
        };
        const uint2 y = make_uint2(q2(x.x) | (q2(x.y) << 16), q2(x.z) | (q2(x.w) << 16));
        *reinterpret_cast<uint2*>((is_v ? vp : kp) + dst) = y;
    }
}

}  // namespace

cudaError_t launch_append(const AppendArgs& a, cudaStream_t stream)
{
    const int64_t total = 2 * int64_t(a.B) * a.L_new * a.H_kv * (a.D / 8);
    if (total == 0)
        return cudaSuccess;
    int64_t blocks = (total + 255) / 256;
    if (blocks > 65535)
        blocks = 65535;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(unsigned(blocks));
    cfg.blockDim = dim3(256);
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return a.fp8 ? cudaLaunchKernelEx(&cfg, append_fp8_kernel, a)
                 : cudaLaunchKernelEx(&cfg, append_kernel, a);
}

}  // namespace pa
