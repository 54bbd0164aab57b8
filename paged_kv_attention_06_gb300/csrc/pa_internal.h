// Internal declarations shared by the library's translation units (host
// launchers and kernel argument blocks). Not part of the public ABI.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "../../include/pagedattn.h"

namespace pa {

// Device error bits (same values as the PA_DEVERR_* macros of the header).
constexpr unsigned PA_DEVERR_PAGE_ID_BIT = 0x1u;
constexpr unsigned PA_DEVERR_SLOT_BIT = 0x2u;
constexpr unsigned PA_DEVERR_CONTEXT_LEN_BIT = 0x4u;
constexpr unsigned PA_DEVERR_TIMEOUT_BIT = 0x8u;

// Longest a kernel waits for one pipeline phase before giving up, and the
// limit of every later wait of a block that already gave up once.
constexpr uint64_t kWaitLimitNs = 1000000000ull;
constexpr uint64_t kShortWaitLimitNs = 20000000ull;

// ---------------------------------------------------------------------------
// Write path

struct AppendArgs {
    const uint16_t* key;          // [B, H_kv, L_new, D]
    const uint16_t* value;
    uint16_t* key_pages;          // [P, H_kv, ps, D]
    uint16_t* value_pages;
    const int32_t* slot_mapping;  // [B, L_new]
    unsigned* err;
    int32_t B, L_new, H_kv, D, ps, num_pages;
    int32_t fp8;                  // 1: the pages hold e4m3 codes (one byte each)
    float k_scale, v_scale;       // e4m3 pages: code = e4m3(x / scale)
};

cudaError_t launch_append(const AppendArgs& a, cudaStream_t stream);

struct GatherArgs {
    const uint16_t* key_pages;    // [P, H_kv, ps, D]
    const uint16_t* value_pages;
    const int32_t* block_table;   // [B, max_pages]
    const int32_t* context_lens;  // [B]
    uint16_t* key_dense;          // [B, H_kv, dense_len, D]
    uint16_t* value_dense;
    unsigned* err;
    int32_t B, H_kv, D, ps, num_pages, max_pages, dense_len;
};

cudaError_t launch_gather(const GatherArgs& a, cudaStream_t stream);

// ---------------------------------------------------------------------------
// Split-KV attention (decode schedule)

// Work decomposition: the G * L query rows of a (request b, KV head h) are
// cut into tiles of 16 rows, and a "segment" is (b, h, group of TG
// consecutive row tiles); its keys are cut into granules of kDecodeTokens
// tokens, and every K/V granule loaded serves all TG tiles. All granules of
// all segments form one stream that the grid splits evenly; a segment that
// straddles blocks leaves one partial state per block, merged by a second,
// small kernel.
constexpr int kDecodeTokens = 64;
constexpr int kDecodeRows = 16;

// At most this many (request x KV head x 16-row tile) per call.
constexpr int64_t kMaxSegments = 65536;

// Row tiles per segment and segment count of a decode call: one tile per
// segment when the rows fit one tile (and always on e4m3 pools), otherwise
// 2 tiles (2 tiles of rows) or 4 (3 or more; a group of 3 tiles leaves the
// fourth slot empty).
struct DecodePlan {
    int32_t MT;      // 16-row tiles per (request, KV head): ceil(G * L / 16)
    int32_t TG;      // row tiles per segment: 1, 2 or 4
    int32_t MS;      // segments per (request, KV head): ceil(MT / TG)
    int64_t nseg;    // B * H_kv * MS
};
DecodePlan decode_plan(const pa_shape& s, bool fp8);

struct DecodeArgs {
    const uint16_t* q;            // [B, H_q, L, D]
    uint16_t* out;                // [B, H_q, L, D]
    const int32_t* block_table;   // [B, max_pages]
    const int32_t* context_lens;  // [B]
    float* partials;              // [slots][TG][m[16], l[16], acc[16][D]]
    unsigned* err;
    int32_t B, H_q, H_kv, L, D, ps, max_pages, num_pages;
    int32_t G;          // H_q / H_kv
    int32_t R;          // G * L query rows per (request, KV head)
    int32_t MS;         // segments per (request, KV head): ceil(ceil(R / 16) / TG)
    int32_t TG;         // 16-row tiles per segment (1, 2 or 4); tile t of segment
                        // ms holds rows [16 (ms TG + t), 16 (ms TG + t) + 16) of R
    int32_t box_rows;   // rows per TMA box: min(ps, 64)
    int32_t swz;        // 7: 128B-swizzled stage layout (box_rows >= 8); 0: linear
    int32_t whole_segments;  // 1: every block takes whole segments (no partials)
    int32_t piece_units;     // split weight of a piece beyond its granules (set by
                             // the launcher for the merge pass)
    int32_t dense;      // 1: K/V are dense [B, H_kv, ps, D] (request b is page b;
                        // block_table is not read)
    float scale_log2;   // scale * log2(e) (times k_scale for e4m3 pages)
    int32_t causal;
    int32_t fp8;        // 1: K/V pages hold e4m3 codes (head_dim 128)
    float v_scale;      // e4m3 pages: the value scale (1 otherwise)
    int32_t debug_unset_wait;  // test support: block 0 first waits on a barrier
                               // that nothing arrives at (times out, flags)
};

size_t decode_smem_bytes(int D, int B, bool fp8 = false, int TG = 1);
int decode_max_grid(int sm_count);
size_t decode_workspace_bytes(int64_t nseg, int grid_max, int D, int TG);
cudaError_t launch_decode(const CUtensorMap& key_map, const CUtensorMap& value_map,
                          const CUtensorMap& q_map, const DecodeArgs& a, int grid, int device,
                          cudaStream_t stream);

// ---------------------------------------------------------------------------
// Prefill on the 5th-generation tensor cores (D = 128, page_size >= 8)

struct PrefillArgs {
    uint16_t* out;                // [B, H_q, L, D]
    const int32_t* block_table;   // [B, max_pages]
    const int32_t* context_lens;  // [B]
    unsigned* err;
    int32_t B, H_q, H_kv, L, ps, max_pages, num_pages;
    int32_t G;          // H_q / H_kv
    int32_t n_qtiles;   // ceil(L / 128)
    int32_t box_rows;   // rows per K/V TMA box: min(ps, 128)
    float scale_log2;
    int32_t causal;
    float out_scale;    // the output is out_scale * softmax . V (e4m3 copies: v_scale)
    int32_t D;          // head_dim: 128 (64 on the pairs kernel only)
    // The pools, read row by row on the pairs kernel when a page holds fewer
    // than 8 tokens (otherwise through the tensor maps).
    const uint16_t* key_pages;    // [P, H_kv, ps, D]
    const uint16_t* value_pages;
    // Pairs kernel, tail pieces (head_dim 128; state == nullptr: none): per
    // donor block slot, part (0: the item's last tiles, 1: its first tiles)
    // and head, O / l in bf16 [16 chunks of 8 columns][128 rows] and (m, l)
    // per row; per slot, head and softmax warp one arrival word (the launch's
    // stamp in the high 32 bits, the arrivals in the low 32).
    uint4* state;                 // [grid][2][2][16][128]
    float2* state_ml;             // [grid][2][2][128]
    unsigned long long* arrive;   // [grid][2][4]
    uint64_t stamp;               // this launch's stamp (never 0)
    int32_t piece_last;           // test setting: receiving blocks run the piece last
};

// Prefill over e4m3 pools: bf16 copies of the visible K/V tokens, in pages
// of 128 tokens; copy page b * P2 + p holds tokens [128 p, 128 p + 128) of
// request b.
struct Fp8PagesArgs {
    const uint8_t* key_pages;     // [P, H_kv, ps, 128] e4m3 codes
    const uint8_t* value_pages;
    const int32_t* block_table;   // [B, max_pages]
    const int32_t* context_lens;  // [B]
    uint16_t* key_out;            // [B * P2, H_kv, 128, 128] bf16
    uint16_t* value_out;
    int32_t* table_out;           // [B, P2]: b * P2 + p
    unsigned* err;
    int32_t B, H_kv, ps, max_pages, num_pages;
    int32_t P2;                   // copy pages per request: ceil(max_context_len / 128)
};
int64_t fp8_copy_pages(int64_t max_context_len);
cudaError_t launch_fp8_pages_to_bf16(const Fp8PagesArgs& a, cudaStream_t stream);

// Stamps for the publish flags of kernels that hand partial states between
// blocks: distinct for every launch of this process, the first one
// seeded from a clock reading so that flags left in a workspace by an earlier
// process are not mistaken for this launch's. Never 0; 48 bits.
uint64_t next_launch_stamp();

// Prefill with the K/V tiles of all (request, head pair, query tile) items
// split evenly over a persistent grid (one block per SM, all resident); an
// item cut by a block boundary is finished by the block that holds its first
// tiles, which merges the states the later pieces left in the workspace.
struct SplitPrefillArgs {
    uint16_t* out;                // [B, H_q, L, 128]
    const int32_t* block_table;   // [B, max_pages]
    const int32_t* context_lens;  // [B]
    unsigned* err;
    float* state;                 // [grid][head 2][32][128][4]
    float2* state_ml;             // [grid][head 2][128] (m, l)
    unsigned long long* flags;    // [grid][head 2][4 warps]: stamp when written
    uint64_t stamp;               // this launch's stamp (never 0)
    int32_t B, H_q, H_kv, L, ps, max_pages, num_pages;
    int32_t G;          // H_q / H_kv (>= 2; odd: the last pair repeats its head)
    int32_t n_qtiles;   // ceil(L / 128)
    int32_t box_rows;   // rows per K/V TMA box: min(ps, 128)
    float scale_log2;
    int32_t causal;
    float out_scale;    // the output is out_scale * softmax . V (e4m3 copies: v_scale)
};

size_t prefill_split_smem_bytes();
size_t prefill_split_workspace_bytes(int grid);
cudaError_t launch_prefill_split(const CUtensorMap& q_map, const CUtensorMap& key_map,
                                 const CUtensorMap& value_map, SplitPrefillArgs a, int grid,
                                 void* workspace, int device, cudaStream_t stream);

size_t prefill_smem_bytes();
size_t prefill_pairs_smem_bytes(int D);
// Workspace of the pairs kernel's tail pieces on a grid of `grid` blocks.
size_t prefill_pairs_workspace_bytes(int grid);
// out_map: the output as a 3-D bf16 tensor {D, L, B * H_q}, boxes of 64
// columns x 32 rows, 128-byte swizzle (the kernel stores through it).
// grid_cap: blocks at most (the SM count). workspace (optional, 256-byte
// aligned, any contents): room for tail pieces (prefill_pairs_workspace_bytes
// of the grid); without it, whole items only.
cudaError_t launch_prefill_pairs(const CUtensorMap& q_map, const CUtensorMap& key_map,
                                 const CUtensorMap& value_map, const CUtensorMap& out_map,
                                 const PrefillArgs& a, int device, int grid_cap, void* workspace,
                                 size_t workspace_bytes, cudaStream_t stream);
cudaError_t launch_prefill(const CUtensorMap& q_map, const CUtensorMap& key_map,
                           const CUtensorMap& value_map, const PrefillArgs& a, int device,
                           cudaStream_t stream);

// Host-side checks of a decode call (everything pa_decode rejects before
// launching, except the workspace), and its number of segments.
pa_status validate_decode(const void* query, const void* key_pages, const void* value_pages,
                          const int32_t* block_table, const int32_t* context_lens,
                          int32_t page_size, float scale, const void* out, const pa_shape& s);
int64_t decode_segment_count(const pa_shape& s);

}  // namespace pa
