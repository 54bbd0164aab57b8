// pa_decode_noalloc: the split-KV decode with its scratch held inside the
// library, for callers that cannot allocate device memory.
//
// Some callers of this library have no way to obtain device memory of their
// own: a host program embedded in another runtime that owns every device
// allocation and only hands out the input and output pointers, or a serving
// loop in which cudaMalloc and cudaFree are off limits because they can
// synchronise the device and stall the requests in flight. pa_decode needs a
// caller-provided workspace; this entry point takes the same inputs and
// output but uses a fixed scratch array that lives in the library's device
// image instead.
//
// The array (kNoAllocScratchBytes) belongs to every GPU that loads this part
// of the library and stays allocated until the process exits. Its device
// address is looked up once per device, with that device current; the host
// symbol itself is only a stand-in and is never passed to a kernel.
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "../../include/pagedattn.h"
#include "pa_internal.h"

// Upper bound of the built-in scratch: 32 MiB.
constexpr size_t kNoAllocScratchBytes = size_t(32) << 20;

static __device__ __align__(256) unsigned char g_pa_noalloc_scratch[kNoAllocScratchBytes];

namespace {

constexpr int kMaxNoAllocDevices = 64;
std::mutex g_noalloc_mutex;
void* g_noalloc_scratch_ptr[kMaxNoAllocDevices] = {};

// Device address of the scratch array on the current device (looked up on the
// first call for each device).
pa_status noalloc_scratch(void** out)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxNoAllocDevices)
        return PA_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_noalloc_mutex);
    if (!g_noalloc_scratch_ptr[dev]) {
        void* ptr = nullptr;
        if (cudaGetSymbolAddress((void**)&ptr, g_pa_noalloc_scratch) != cudaSuccess || !ptr)
            return PA_ERR_CUDA;
        g_noalloc_scratch_ptr[dev] = ptr;
    }
    *out = g_noalloc_scratch_ptr[dev];
    return PA_OK;
}

}  // namespace

extern "C" pa_status pa_decode_noalloc(const void* query, const void* key_pages,
                                       const void* value_pages, const int32_t* block_table,
                                       const int32_t* context_lens, int32_t page_size,
                                       float scale, int causal, void* out, pa_shape shape,
                                       int32_t max_context_len, void* stream)
{
    // Same checks as pa_decode, before anything is queued on the stream.
    pa_status st = pa::validate_decode(query, key_pages, value_pages, block_table, context_lens,
                                       page_size, scale, out, shape);
    if (st != PA_OK)
        return st;
    const size_t need = pa_decode_workspace_bytes(shape);
    if (need == 0)
        return PA_ERR_CUDA;
    if (need > kNoAllocScratchBytes)
        return PA_ERR_WORKSPACE;  // the shape needs more scratch than the built-in array
    void* scratch = nullptr;
    if ((st = noalloc_scratch(&scratch)) != PA_OK)
        return st;
    // The array keeps whatever the previous call left; the decode reads only
    // what it writes first, so nothing needs clearing.
    return pa_decode(query, key_pages, value_pages, block_table, context_lens, page_size, scale,
                     causal, out, shape, max_context_len, scratch, kNoAllocScratchBytes, stream);
}
