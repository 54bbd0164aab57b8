// Host-side page allocator and per-step metadata builder (host code only).
//
// The pages' serving stack keeps, per request, the list of pages it holds in
// each layer pool and the number of tokens cached; a scheduler step turns
// that into the block_table, context_lens and slot_mapping the kernels read
// (Week 3 Day 4, "Decode Metadata": allocate a page only when the tail page is
// full; prepare the batch's page metadata once per scheduler step; Tutorial
// 13, section 4 "The Request Cache": fill the tail page first, then
// allocate; release every page of a finished request exactly once; restore
// the pool when a write fails).
//
// pa_kv_cache_step runs a whole step from the host in one call: the plan,
// one copy of the packed tables, the append and the attention launch.
//
// The allocator hands out a freed page first (free list, last freed first)
// and otherwise the lowest never-used page id. A step is all-or-nothing: the
// allocations it made are undone, in reverse, when any request of the step
// cannot be placed, so a failed step leaves the cache exactly as it was.
#include <cuda_runtime.h>
#include <stdint.h>
#include <string.h>

#include <new>
#include <unordered_map>
#include <unordered_set>
#include <vector>

#include "../../include/pagedattn.h"

namespace {

struct Sequence {
    std::vector<int32_t> pages;
    int32_t len = 0;       // tokens cached
};

}  // namespace

struct pa_kv_cache {
    int32_t num_pages = 0;
    int32_t page_size = 0;
    int32_t next_fresh = 0;                 // lowest page id never handed out
    std::vector<int32_t> free_list;         // freed ids, last freed at the back
    std::unordered_map<int64_t, Sequence> seqs;
    int32_t held = 0;                       // pages held by sequences
};

namespace {

// One allocation, for undo: the page and whether it came off the free list.
struct Taken {
    int32_t page;
    bool from_free_list;
};

bool take_page(pa_kv_cache* c, std::vector<Taken>* log, int32_t* page)
{
    if (!c->free_list.empty()) {
        *page = c->free_list.back();
        c->free_list.pop_back();
        log->push_back({*page, true});
    } else if (c->next_fresh < c->num_pages) {
        *page = c->next_fresh++;
        log->push_back({*page, false});
    } else {
        return false;
    }
    ++c->held;
    return true;
}

void undo(pa_kv_cache* c, const std::vector<Taken>& log)
{
    for (size_t k = log.size(); k-- > 0;) {
        if (log[k].from_free_list)
            c->free_list.push_back(log[k].page);
        else
            --c->next_fresh;
        --c->held;
    }
}

}  // namespace

struct pa_kv_cache_snapshot {
    const pa_kv_cache* owner;
    pa_kv_cache state;
};

extern "C" {

pa_status pa_kv_cache_create(int32_t num_pages, int32_t page_size, pa_kv_cache** cache)
{
    if (!cache || num_pages <= 0 || page_size <= 0)
        return PA_ERR_INVALID_ARG;
    pa_kv_cache* c = new (std::nothrow) pa_kv_cache;
    if (!c)
        return PA_ERR_NO_PAGES;
    c->num_pages = num_pages;
    c->page_size = page_size;
    *cache = c;
    return PA_OK;
}

void pa_kv_cache_destroy(pa_kv_cache* cache) { delete cache; }

pa_status pa_kv_cache_add(pa_kv_cache* cache, int64_t seq_id)
{
    if (!cache)
        return PA_ERR_INVALID_ARG;
    if (cache->seqs.count(seq_id))
        return PA_ERR_INVALID_ARG;
    cache->seqs.emplace(seq_id, Sequence());
    return PA_OK;
}

pa_status pa_kv_cache_release(pa_kv_cache* cache, int64_t seq_id)
{
    if (!cache)
        return PA_ERR_INVALID_ARG;
    auto it = cache->seqs.find(seq_id);
    if (it == cache->seqs.end())
        return PA_ERR_INVALID_ARG;   // unknown, or released already
    for (int32_t p : it->second.pages)
        cache->free_list.push_back(p);
    cache->held -= int32_t(it->second.pages.size());
    cache->seqs.erase(it);
    return PA_OK;
}

int32_t pa_kv_cache_free_pages(const pa_kv_cache* cache)
{
    return cache ? cache->num_pages - cache->held : -1;
}

int32_t pa_kv_cache_context_len(const pa_kv_cache* cache, int64_t seq_id)
{
    if (!cache)
        return -1;
    auto it = cache->seqs.find(seq_id);
    return it == cache->seqs.end() ? -1 : it->second.len;
}

pa_status pa_kv_cache_plan(pa_kv_cache* cache, int32_t n, const int64_t* seq_ids,
                           const int32_t* new_tokens, int32_t max_pages, int32_t l_new,
                           int32_t* block_table, int32_t* context_lens, int32_t* slot_mapping)
{
    if (!cache || n < 0 || max_pages <= 0 || l_new < 0)
        return PA_ERR_INVALID_ARG;
    if (n > 0 && (!seq_ids || !new_tokens || !block_table || !context_lens ||
                  (l_new > 0 && !slot_mapping)))
        return PA_ERR_INVALID_ARG;
    // Validate every request before touching anything.
    std::unordered_set<int64_t> seen;
    for (int32_t i = 0; i < n; ++i) {
        if (new_tokens[i] < 0 || new_tokens[i] > l_new)
            return PA_ERR_INVALID_ARG;
        if (!seen.insert(seq_ids[i]).second || !cache->seqs.count(seq_ids[i]))
            return PA_ERR_INVALID_ARG;   // listed twice, or unknown
        if (int64_t(cache->seqs[seq_ids[i]].pages.size()) > max_pages)
            return PA_ERR_NO_PAGES;      // its block-table row does not fit
    }
    const int32_t ps = cache->page_size;
    std::vector<Taken> log;
    struct Before {
        Sequence* s;
        size_t pages;
        int32_t len;
    };
    std::vector<Before> before;
    before.reserve(size_t(n));
    pa_status st = PA_OK;
    for (int32_t i = 0; i < n && st == PA_OK; ++i) {
        Sequence& s = cache->seqs[seq_ids[i]];
        before.push_back({&s, s.pages.size(), s.len});
        int32_t* slots = slot_mapping ? slot_mapping + int64_t(i) * l_new : nullptr;
        for (int32_t k = 0; k < new_tokens[i]; ++k) {
            const int32_t pos = s.len;
            if (pos % ps == 0) {   // the tail page is full (or there is none)
                int32_t page;
                if (int32_t(s.pages.size()) >= max_pages || !take_page(cache, &log, &page)) {
                    st = PA_ERR_NO_PAGES;
                    break;
                }
                s.pages.push_back(page);
            }
            slots[k] = s.pages.back() * ps + pos % ps;
            ++s.len;
        }
    }
    if (st != PA_OK) {
        for (const Before& b : before) {
            b.s->pages.resize(b.pages);
            b.s->len = b.len;
        }
        undo(cache, log);
        return st;
    }
    for (int32_t i = 0; i < n; ++i) {
        const Sequence& s = cache->seqs[seq_ids[i]];
        int32_t* row = block_table + int64_t(i) * max_pages;
        const int32_t np = int32_t(s.pages.size());
        memcpy(row, s.pages.data(), size_t(np) * sizeof(int32_t));
        for (int32_t k = np; k < max_pages; ++k)
            row[k] = -1;
        context_lens[i] = s.len;
        if (slot_mapping)
            for (int32_t k = new_tokens[i]; k < l_new; ++k)
                slot_mapping[int64_t(i) * l_new + k] = -1;
    }
    return PA_OK;
}

pa_status pa_kv_cache_snapshot_take(const pa_kv_cache* cache, pa_kv_cache_snapshot** snapshot)
{
    if (!cache || !snapshot)
        return PA_ERR_INVALID_ARG;
    pa_kv_cache_snapshot* s = new (std::nothrow) pa_kv_cache_snapshot;
    if (!s)
        return PA_ERR_NO_PAGES;
    s->owner = cache;
    s->state = *cache;
    *snapshot = s;
    return PA_OK;
}

pa_status pa_kv_cache_restore(pa_kv_cache* cache, const pa_kv_cache_snapshot* snapshot)
{
    if (!cache || !snapshot || snapshot->owner != cache)
        return PA_ERR_INVALID_ARG;
    *cache = snapshot->state;
    return PA_OK;
}

void pa_kv_cache_snapshot_destroy(pa_kv_cache_snapshot* snapshot) { delete snapshot; }

size_t pa_kv_cache_step_table_bytes(int32_t n, int32_t max_pages, int32_t l_new)
{
    if (n <= 0 || max_pages <= 0 || l_new <= 0)
        return 0;
    return size_t(n) * size_t(max_pages + 1 + l_new) * sizeof(int32_t);
}

pa_status pa_kv_cache_step(pa_kv_cache* cache, int32_t n, const int64_t* seq_ids,
                           const int32_t* new_tokens, int32_t l_new, int32_t max_pages,
                           void* host_tables, void* device_tables, size_t table_bytes,
                           const void* key_new, const void* value_new, const void* query,
                           void* key_pages, void* value_pages, int32_t num_q_heads,
                           int32_t num_kv_heads, int32_t head_dim, float scale, void* out,
                           void* workspace, size_t workspace_bytes, void* stream)
{
    const size_t need = pa_kv_cache_step_table_bytes(n, max_pages, l_new);
    if (!cache || need == 0 || !host_tables || !device_tables || table_bytes < need)
        return PA_ERR_INVALID_ARG;
    // The three tables, packed: block_table [n, max_pages], context_lens [n],
    // slot_mapping [n, l_new].
    int32_t* h_bt = static_cast<int32_t*>(host_tables);
    int32_t* h_cl = h_bt + int64_t(n) * max_pages;
    int32_t* h_sm = h_cl + n;
    pa_status st = pa_kv_cache_plan(cache, n, seq_ids, new_tokens, max_pages, l_new, h_bt, h_cl,
                                    h_sm);
    if (st != PA_OK)
        return st;
    int32_t max_len = 0;
    for (int32_t i = 0; i < n; ++i)
        max_len = h_cl[i] > max_len ? h_cl[i] : max_len;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (cudaMemcpyAsync(device_tables, host_tables, need, cudaMemcpyHostToDevice, s) != cudaSuccess)
        return PA_ERR_CUDA;
    const int32_t* d_bt = static_cast<const int32_t*>(device_tables);
    const int32_t* d_cl = d_bt + int64_t(n) * max_pages;
    const int32_t* d_sm = d_cl + n;
    pa_shape shape;
    shape.batch = n;
    shape.num_q_heads = num_q_heads;
    shape.num_kv_heads = num_kv_heads;
    shape.head_dim = head_dim;
    shape.q_len = l_new;
    shape.num_pages = cache->num_pages;
    shape.max_pages = max_pages;
    st = pa_append_kv(key_new, value_new, key_pages, value_pages, d_sm, cache->page_size, shape,
                      stream);
    if (st != PA_OK)
        return st;
    return pa_attention(query, key_pages, value_pages, d_bt, d_cl, cache->page_size, scale, 1, out,
                        shape, max_len, workspace, workspace_bytes, stream);
}

}  // extern "C"
