// Native timed loops for bench.py: the benchmark's steps issued from C
// through the public C ABI of libpagedattn.so, so that no interpreter runs
// between launches inside a timed region. Not part of the library.
//
// One step = pa_append_kv (new K/V rows by slot_mapping) + pa_attention on
// page-pool copy k % n_copies. CUDA events bracket the whole loop, and
// optionally the attention call of every `sample_every`-th step: an event
// between two kernels stops the second from being scheduled early
// (programmatic dependent launch), so the benchmark takes the time of one
// call from blocks of back-to-back calls instead (pa_bench_attention_calls).
#include <cuda_runtime.h>
#include <stdint.h>

#include <vector>

#include "include/pagedattn.h"

namespace {

struct EventPool {
    std::vector<cudaEvent_t> ev;
    explicit EventPool(size_t n) : ev(n, nullptr)
    {
        for (auto& e : ev)
            if (cudaEventCreate(&e) != cudaSuccess)
                e = nullptr;
    }
    ~EventPool()
    {
        for (auto e : ev)
            if (e)
                cudaEventDestroy(e);
    }
    bool ok() const
    {
        for (auto e : ev)
            if (!e)
                return false;
        return true;
    }
};

}  // namespace

extern "C" {

// Returns 0 on success, a pa_status (> 0) if a call failed, -1 on a CUDA
// error. step_ms[j]: device time of the attention call of step
// j * sample_every (no such events when sample_every < 1); *total_ms: the
// whole loop (first append to last attention).
int pa_bench_steps(int n_steps, int sample_every, int n_copies, const void* key_new, const void* value_new,
                   void* const* key_pages, void* const* value_pages,
                   const int32_t* slot_mapping, int32_t page_size, pa_shape append_shape,
                   const void* query, const int32_t* block_table, const int32_t* context_lens,
                   float scale, int causal, void* out, pa_shape shape, int32_t max_context_len,
                   void* workspace, size_t workspace_bytes, void* stream, float* step_ms,
                   float* total_ms)
{
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    // sample_every < 1: no event inside the loop
    const int n_samples = sample_every < 1 ? 0 : (n_steps + sample_every - 1) / sample_every;
    EventPool pool(2 * size_t(n_samples) + 2);
    if (!pool.ok())
        return -1;
    cudaEvent_t t0 = pool.ev[2 * n_samples], t1 = pool.ev[2 * n_samples + 1];
    if (cudaEventRecord(t0, s) != cudaSuccess)
        return -1;
    for (int k = 0; k < n_steps; ++k) {
        const int c = k % n_copies;
        const bool sampled = n_samples > 0 && k % sample_every == 0;
        const int j = n_samples > 0 ? k / sample_every : 0;
        pa_status st = pa_append_kv(key_new, value_new, key_pages[c], value_pages[c],
                                    slot_mapping, page_size, append_shape, stream);
        if (st != PA_OK)
            return int(st);
        if (sampled)
            cudaEventRecord(pool.ev[2 * j], s);
        st = pa_attention(query, key_pages[c], value_pages[c], block_table, context_lens,
                          page_size, scale, causal, out, shape, max_context_len, workspace,
                          workspace_bytes, stream);
        if (st != PA_OK)
            return int(st);
        if (sampled)
            cudaEventRecord(pool.ev[2 * j + 1], s);
    }
    if (cudaEventRecord(t1, s) != cudaSuccess || cudaEventSynchronize(t1) != cudaSuccess)
        return -1;
    for (int j = 0; j < n_samples; ++j)
        if (cudaEventElapsedTime(&step_ms[j], pool.ev[2 * j], pool.ev[2 * j + 1]) != cudaSuccess)
            return -1;
    return cudaEventElapsedTime(total_ms, t0, t1) == cudaSuccess ? 0 : -1;
}

// pa_bench_steps for e4m3 page pools: pa_append_kv_fp8 + pa_decode_fp8 per
// step, the same events.
int pa_bench_steps_fp8(int n_steps, int sample_every, int n_copies, const void* key_new,
                       const void* value_new, void* const* key_pages, void* const* value_pages,
                       const int32_t* slot_mapping, int32_t page_size, pa_shape append_shape,
                       const void* query, const int32_t* block_table, const int32_t* context_lens,
                       float scale, float k_scale, float v_scale, int causal, void* out,
                       pa_shape shape, int32_t max_context_len, void* workspace,
                       size_t workspace_bytes, void* stream, float* step_ms, float* total_ms)
{
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const int n_samples = sample_every < 1 ? 0 : (n_steps + sample_every - 1) / sample_every;
    EventPool pool(2 * size_t(n_samples) + 2);
    if (!pool.ok())
        return -1;
    cudaEvent_t t0 = pool.ev[2 * n_samples], t1 = pool.ev[2 * n_samples + 1];
    if (cudaEventRecord(t0, s) != cudaSuccess)
        return -1;
    for (int k = 0; k < n_steps; ++k) {
        const int c = k % n_copies;
        const bool sampled = n_samples > 0 && k % sample_every == 0;
        const int j = n_samples > 0 ? k / sample_every : 0;
        pa_status st = pa_append_kv_fp8(key_new, value_new, key_pages[c], value_pages[c],
                                        slot_mapping, page_size, k_scale, v_scale, append_shape,
                                        stream);
        if (st != PA_OK)
            return int(st);
        if (sampled)
            cudaEventRecord(pool.ev[2 * j], s);
        st = pa_decode_fp8(query, key_pages[c], value_pages[c], block_table, context_lens,
                           page_size, scale, k_scale, v_scale, causal, out, shape,
                           max_context_len, workspace, workspace_bytes, stream);
        if (st != PA_OK)
            return int(st);
        if (sampled)
            cudaEventRecord(pool.ev[2 * j + 1], s);
    }
    if (cudaEventRecord(t1, s) != cudaSuccess || cudaEventSynchronize(t1) != cudaSuccess)
        return -1;
    for (int j = 0; j < n_samples; ++j)
        if (cudaEventElapsedTime(&step_ms[j], pool.ev[2 * j], pool.ev[2 * j + 1]) != cudaSuccess)
            return -1;
    return cudaEventElapsedTime(total_ms, t0, t1) == cudaSuccess ? 0 : -1;
}

// End-to-end steps from pinned host buffers: every step copies the step's
// inputs host -> device (query, new K/V, slot_mapping, block_table,
// context_lens), runs the step, and copies the output back.
int pa_bench_e2e_steps(int n_steps, int n_copies, const void* const* host_src,
                       void* const* dev_dst, const size_t* bytes, int n_inputs,
                       const void* dev_out, void* host_out, size_t out_bytes,
                       const void* key_new, const void* value_new, void* const* key_pages,
                       void* const* value_pages, const int32_t* slot_mapping, int32_t page_size,
                       pa_shape append_shape, const void* query, const int32_t* block_table,
                       const int32_t* context_lens, float scale, int causal, void* out,
                       pa_shape shape, int32_t max_context_len, void* workspace,
                       size_t workspace_bytes, void* stream, float* total_ms)
{
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    EventPool pool(2);
    if (!pool.ok())
        return -1;
    if (cudaEventRecord(pool.ev[0], s) != cudaSuccess)
        return -1;
    for (int k = 0; k < n_steps; ++k) {
        const int c = k % n_copies;
        for (int i = 0; i < n_inputs; ++i)
            if (cudaMemcpyAsync(dev_dst[i], host_src[i], bytes[i], cudaMemcpyHostToDevice, s) !=
                cudaSuccess)
                return -1;
        pa_status st = pa_append_kv(key_new, value_new, key_pages[c], value_pages[c],
                                    slot_mapping, page_size, append_shape, stream);
        if (st != PA_OK)
            return int(st);
        st = pa_attention(query, key_pages[c], value_pages[c], block_table, context_lens,
                          page_size, scale, causal, out, shape, max_context_len, workspace,
                          workspace_bytes, stream);
        if (st != PA_OK)
            return int(st);
        if (cudaMemcpyAsync(host_out, dev_out, out_bytes, cudaMemcpyDeviceToHost, s) !=
            cudaSuccess)
            return -1;
    }
    if (cudaEventRecord(pool.ev[1], s) != cudaSuccess || cudaEventSynchronize(pool.ev[1]) != cudaSuccess)
        return -1;
    return cudaEventElapsedTime(total_ms, pool.ev[0], pool.ev[1]) == cudaSuccess ? 0 : -1;
}

// The end-to-end step with its copies overlapped with the kernels of the
// neighbouring steps, as a serving loop runs it. Step k's inputs (one packed
// pinned region, `in_bytes`) are copied on copy_stream into device region
// k % 2 while step k - 1 computes on `stream`. Step k's output (device buffer
// k % 2) comes back on out_stream while step k + 1 computes (a stream of its
// own, so that the next input copy does not queue behind it). Every step still
// moves its own inputs and its own output inside the timed region. The
// inputs sit at byte offsets off[0..5] (query, new K, new V, slot_mapping,
// block_table, context_lens) of each device region.
int pa_bench_e2e_pipelined(int n_steps, int n_copies, const void* host_in,
                           void* const* dev_in, size_t in_bytes, const size_t* off,
                           void* const* dev_out, void* const* host_out, size_t out_bytes,
                           void* const* key_pages, void* const* value_pages, int32_t page_size,
                           pa_shape append_shape, float scale, int causal, pa_shape shape,
                           int32_t max_context_len, void* workspace, size_t workspace_bytes,
                           void* stream, void* copy_stream, void* out_stream,
                           float* total_ms)
{
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaStream_t cs = static_cast<cudaStream_t>(copy_stream);
    cudaStream_t os = static_cast<cudaStream_t>(out_stream);
    EventPool timing(2);
    std::vector<cudaEvent_t> sync(6, nullptr);   // in_ready[2], done[2], out_free[2]
    struct Destroy {
        std::vector<cudaEvent_t>& e;
        ~Destroy()
        {
            for (auto x : e)
                if (x)
                    cudaEventDestroy(x);
        }
    } destroy{sync};
    if (!timing.ok())
        return -1;
    for (auto& e : sync)
        if (cudaEventCreateWithFlags(&e, cudaEventDisableTiming) != cudaSuccess)
            return -1;
    cudaEvent_t* in_ready = &sync[0];
    cudaEvent_t* done = &sync[2];
    cudaEvent_t* out_free = &sync[4];
    if (cudaEventRecord(timing.ev[0], s) != cudaSuccess ||
        cudaStreamWaitEvent(cs, timing.ev[0], 0) != cudaSuccess ||
        cudaStreamWaitEvent(os, timing.ev[0], 0) != cudaSuccess)
        return -1;
    for (int k = 0; k < n_steps; ++k) {
        const int r = k & 1, c = k % n_copies;
        uint8_t* base = static_cast<uint8_t*>(dev_in[r]);
        // inputs: region r is free once step k - 2 has run
        if (k >= 2 && cudaStreamWaitEvent(cs, done[r], 0) != cudaSuccess)
            return -1;
        if (cudaMemcpyAsync(base, host_in, in_bytes, cudaMemcpyHostToDevice, cs) != cudaSuccess ||
            cudaEventRecord(in_ready[r], cs) != cudaSuccess)
            return -1;
        // the step, once its inputs are in and output buffer r has been read back
        if (cudaStreamWaitEvent(s, in_ready[r], 0) != cudaSuccess)
            return -1;
        if (k >= 2 && cudaStreamWaitEvent(s, out_free[r], 0) != cudaSuccess)
            return -1;
        pa_status st = pa_append_kv(base + off[1], base + off[2], key_pages[c], value_pages[c],
                                    reinterpret_cast<const int32_t*>(base + off[3]), page_size,
                                    append_shape, stream);
        if (st != PA_OK)
            return int(st);
        st = pa_attention(base + off[0], key_pages[c], value_pages[c],
                          reinterpret_cast<const int32_t*>(base + off[4]),
                          reinterpret_cast<const int32_t*>(base + off[5]), page_size, scale,
                          causal, dev_out[r], shape, max_context_len, workspace, workspace_bytes,
                          stream);
        if (st != PA_OK)
            return int(st);
        if (cudaEventRecord(done[r], s) != cudaSuccess)
            return -1;
        // output of step k back to the host
        if (cudaStreamWaitEvent(os, done[r], 0) != cudaSuccess ||
            cudaMemcpyAsync(host_out[r], dev_out[r], out_bytes, cudaMemcpyDeviceToHost, os) !=
                cudaSuccess ||
            cudaEventRecord(out_free[r], os) != cudaSuccess)
            return -1;
    }
    if (cudaEventRecord(timing.ev[1], os) != cudaSuccess ||
        cudaEventSynchronize(timing.ev[1]) != cudaSuccess || cudaStreamSynchronize(s) != cudaSuccess ||
        cudaStreamSynchronize(cs) != cudaSuccess)
        return -1;
    return cudaEventElapsedTime(total_ms, timing.ev[0], timing.ev[1]) == cudaSuccess ? 0 : -1;
}

// Back-to-back attention calls with no other work and no event between them:
// call k reads page-pool copy k % n_copies. Events bracket the whole loop,
// so *total_ms / n_calls is the device time of one call as a stream of
// calls runs it (each call's kernels may be scheduled while the one before
// drains). fp8 != 0: pa_decode_fp8 over e4m3 pools with k_scale / v_scale;
// otherwise pa_attention.
int pa_bench_attention_calls(int n_calls, int n_copies, void* const* key_pages,
                             void* const* value_pages, const void* query,
                             const int32_t* block_table, const int32_t* context_lens,
                             int32_t page_size, float scale, int causal, int fp8, float k_scale,
                             float v_scale, void* out, pa_shape shape, int32_t max_context_len,
                             void* workspace, size_t workspace_bytes, void* stream,
                             float* total_ms)
{
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    EventPool pool(2);
    if (!pool.ok())
        return -1;
    if (cudaEventRecord(pool.ev[0], s) != cudaSuccess)
        return -1;
    for (int k = 0; k < n_calls; ++k) {
        const int c = k % n_copies;
        const pa_status st =
            fp8 ? pa_decode_fp8(query, key_pages[c], value_pages[c], block_table, context_lens,
                                page_size, scale, k_scale, v_scale, causal, out, shape,
                                max_context_len, workspace, workspace_bytes, stream)
                : pa_attention(query, key_pages[c], value_pages[c], block_table, context_lens,
                               page_size, scale, causal, out, shape, max_context_len, workspace,
                               workspace_bytes, stream);
        if (st != PA_OK)
            return int(st);
    }
    if (cudaEventRecord(pool.ev[1], s) != cudaSuccess ||
        cudaEventSynchronize(pool.ev[1]) != cudaSuccess)
        return -1;
    return cudaEventElapsedTime(total_ms, pool.ev[0], pool.ev[1]) == cudaSuccess ? 0 : -1;
}

}  // extern "C"
