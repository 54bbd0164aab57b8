// Dense baseline, first step: gather every request's visible K and V rows
// out of the page pool into dense [B, H_kv, dense_len, D] buffers (the dense
// path of Week 3 Day 4 materialises each request's cached K/V contiguously
// before attending; Direct Paged Attention avoids exactly this copy).
//
// One thread moves one 16-byte vector (8 bf16) of one token's K or V row for
// one KV head: consecutive threads cover consecutive 16-byte pieces of a
// row and consecutive rows of a page, so both the read of the page slice and
// the write of the dense row are coalesced. Bit copy; rows at or past a
// request's context are not written.
#include <stdint.h>

#include "pa_device.cuh"
#include "pa_internal.h"

namespace pa {
namespace {

__global__ void __launch_bounds__(256) gather_kernel(const GatherArgs a)
{
    // Launched with programmatic stream serialization: wait for the previous
    // kernel in the stream (which may still write the pool or the tables).
    grid_dependency_wait();
    grid_launch_dependents();
    const int vec_per_row = a.D / 8;
    const int64_t per_tensor = int64_t(a.B) * a.H_kv * a.dense_len * vec_per_row;
    const int64_t total = 2 * per_tensor;
    const int cap = a.max_pages * a.ps;
    for (int64_t t = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; t < total;
         t += int64_t(gridDim.x) * blockDim.x) {
        const bool is_v = t >= per_tensor;
        int64_t u = is_v ? t - per_tensor : t;
        const int c = int(u % vec_per_row);
        u /= vec_per_row;
        const int tok = int(u % a.dense_len);
        u /= a.dense_len;
        const int h = int(u % a.H_kv);
        const int b = int(u / a.H_kv);
        int n = a.context_lens[b];
        if (n < 0 || n > cap || n > a.dense_len) {
            if (tok == 0 && c == 0 && h == 0 && !is_v)
                atomicOr(a.err, PA_DEVERR_CONTEXT_LEN_BIT);
            n = n < 0 ? 0 : min(min(n, cap), a.dense_len);
        }
        if (tok >= n)
            continue;
        const int lp = tok / a.ps;
        const int phys = a.block_table[int64_t(b) * a.max_pages + lp];
        if (unsigned(phys) >= unsigned(a.num_pages)) {
            if (c == 0 && h == 0 && !is_v)
                atomicOr(a.err, PA_DEVERR_PAGE_ID_BIT);
            continue;
        }
        const int64_t src = ((int64_t(phys) * a.H_kv + h) * a.ps + (tok - lp * a.ps)) * a.D + c * 8;
        const int64_t dst = ((int64_t(b) * a.H_kv + h) * a.dense_len + tok) * a.D + c * 8;
        const uint16_t* s = is_v ? a.value_pages : a.key_pages;
        uint16_t* d = is_v ? a.value_dense : a.key_dense;
        *reinterpret_cast<uint4*>(d + dst) = *reinterpret_cast<const uint4*>(s + src);
    }
}

}  // namespace

cudaError_t launch_gather(const GatherArgs& a, cudaStream_t stream)
{
    const int64_t total = 2 * int64_t(a.B) * a.H_kv * a.dense_len * (a.D / 8);
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
    return cudaLaunchKernelEx(&cfg, gather_kernel, a);
}

}  // namespace pa
