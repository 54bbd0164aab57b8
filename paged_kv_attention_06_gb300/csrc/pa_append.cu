// Write path: scatter new K/V rows into the page pool by slot_mapping
// (Reading vLLM's PagedAttention Kernel, 3.2 "Writing into the cache").
//
// One thread moves one 16-byte vector (8 bf16) of one token's K row and the
// same vector of its V row for one KV head. The flat thread index runs over
// [B, H_kv, L_new, D / 8], the layout of the new rows, so the source offset
// is the index itself and both the reads and the writes of consecutive
// threads are consecutive 16-byte pieces of rows (a token's page row, and
// the next token's when it sits in the next slot). The copy is bit-exact (no
// conversion); pages of e4m3 codes get the quantised rows instead.
#include <stdint.h>

#include "pa_device.cuh"
#include "pa_internal.h"

namespace pa {
namespace {

// Thread t of the flat index (t below the thread count): vector c of row
// (b, h, i) (i fastest among the rows); its source is element t * 8 of key /
// value.
struct AppendPos {
    int64_t dst;      // element offset in the page pool, or -1: skip
};

__device__ __forceinline__ void append_pos(const AppendArgs& a, int64_t t, int vshift,
                                           AppendPos& p)
{
    const int64_t r = t >> vshift;
    const int c = int(t & ((1 << vshift) - 1));
    const int64_t bh = udiv64(r, a.L_new);
    const int i = int(r - bh * a.L_new);
    const int b = int(udiv64(bh, a.H_kv));
    const int h = int(bh - int64_t(b) * a.H_kv);
    p.dst = -1;
    const int64_t slot = a.slot_mapping[int64_t(b) * a.L_new + i];
    if (slot < 0)
        return;  // padding token
    const int64_t page = udiv64(slot, a.ps);
    const int64_t off = slot - page * a.ps;
    if (page >= a.num_pages) {
        if (c == 0 && h == 0)
            atomicOr(a.err, PA_DEVERR_SLOT_BIT);
        return;
    }
    p.dst = ((page * a.H_kv + h) * a.ps + off) * a.D + c * 8;
}

__global__ void __launch_bounds__(256) append_kernel(const AppendArgs a)
{
    // Launched with programmatic stream serialization: wait for the previous
    // kernel in the stream (which may still read the pool) before writing,
    // and let the attention kernel that follows be scheduled.
    grid_dependency_wait();
    grid_launch_dependents();
    const int vshift = a.D == 128 ? 4 : 3;   // 16-byte vectors per row: 16 or 8
    const int64_t total = (int64_t(a.B) * a.H_kv * a.L_new) << vshift;
    for (int64_t t = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; t < total;
         t += int64_t(gridDim.x) * blockDim.x) {
        // The source rows do not depend on the slot: their loads are in
        // flight together with the slot_mapping load.
        const uint4 k = *reinterpret_cast<const uint4*>(a.key + t * 8);
        const uint4 v = *reinterpret_cast<const uint4*>(a.value + t * 8);
        AppendPos p;
        append_pos(a, t, vshift, p);
        if (p.dst < 0)
            continue;
        *reinterpret_cast<uint4*>(a.key_pages + p.dst) = k;
        *reinterpret_cast<uint4*>(a.value_pages + p.dst) = v;
    }
}

// The same scatter into pages of e4m3 codes: every element is stored as the
// code nearest to fp32(x) / scale (ties to even, saturated to +-448), 8
// elements of K and of V per thread (16 bytes in, 8 bytes out each).
__global__ void __launch_bounds__(256) append_fp8_kernel(const AppendArgs a)
{
    grid_dependency_wait();
    grid_launch_dependents();
    const int vshift = a.D == 128 ? 4 : 3;
    uint8_t* const kp = reinterpret_cast<uint8_t*>(a.key_pages);
    uint8_t* const vp = reinterpret_cast<uint8_t*>(a.value_pages);
    const int64_t total = (int64_t(a.B) * a.H_kv * a.L_new) << vshift;
    for (int64_t t = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; t < total;
         t += int64_t(gridDim.x) * blockDim.x) {
        const uint4 k = *reinterpret_cast<const uint4*>(a.key + t * 8);
        const uint4 v = *reinterpret_cast<const uint4*>(a.value + t * 8);
        AppendPos p;
        append_pos(a, t, vshift, p);
        if (p.dst < 0)
            continue;
        auto q2 = [&](uint32_t w, float sc) {   // two bf16 -> two e4m3 codes (16 bits)
            return f32x2_to_e4m3x2(__fdiv_rn(__uint_as_float(w << 16), sc),
                                   __fdiv_rn(__uint_as_float(w & 0xffff0000u), sc));
        };
        auto q8 = [&](uint4 x, float sc) {
            return make_uint2(q2(x.x, sc) | (q2(x.y, sc) << 16), q2(x.z, sc) | (q2(x.w, sc) << 16));
        };
        *reinterpret_cast<uint2*>(kp + p.dst) = q8(k, a.k_scale);
        *reinterpret_cast<uint2*>(vp + p.dst) = q8(v, a.v_scale);
    }
}

}  // namespace

cudaError_t launch_append(const AppendArgs& a, cudaStream_t stream)
{
    const int64_t total = int64_t(a.B) * a.L_new * a.H_kv * (a.D / 8);   // threads
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
