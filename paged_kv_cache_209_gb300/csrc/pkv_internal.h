// Host-side interfaces between the C ABI layer (pkv_api.cu) and the kernel
// translation units. Not part of the public ABI.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include <nvtx3/nvToolsExt.h>

#include "pkv.h"

namespace pkv {

// An NVTX range named after the API call, open for the call's host-side
// duration (argument checks and kernel launches). Profilers (Nsight Systems,
// Nsight Compute with --nvtx) show it; without a profiler attached a push or
// pop costs one indirect call.
struct NvtxRange {
    explicit NvtxRange(const char* name) { nvtxRangePushA(name); }
    ~NvtxRange() { nvtxRangePop(); }
    NvtxRange(const NvtxRange&) = delete;
    NvtxRange& operator=(const NvtxRange&) = delete;
};

// ---------------------------------------------------------------- KV moves
cudaError_t launch_append(const void* k, const void* v, const int64_t* slots, int64_t num_tokens, void* k_cache,
                          void* v_cache, const pkv_cache_desc& d, unsigned int* status, cudaStream_t s);
cudaError_t launch_copy_blocks(const int64_t* pairs, int64_t num_pairs, void* k_cache, void* v_cache,
                               const pkv_cache_desc& d, unsigned int* status, cudaStream_t s);

// Validation kernels for PKV_FLAG_CHECKED: OR a PKV_ERR_* code into *verdict
// (the ordering RANGE < OVERLAP does not matter: any nonzero is a rejection).
cudaError_t launch_check_slots(const int64_t* slots, int64_t num_tokens, int64_t num_slots, unsigned int* verdict,
                               cudaStream_t s);
cudaError_t launch_check_pairs(const int64_t* pairs, int64_t num_pairs, int64_t num_blocks, unsigned int* verdict,
                               cudaStream_t s);
// Context lengths must lie in [min_len, max_blocks * 16]: min_len is 1 for the
// decode calls (a zero-length context is no decode query) and 0 where a
// sequence may carry no queries (multi-query calls).
cudaError_t launch_check_decode(const int32_t* tables, int32_t max_blocks, const int32_t* lens, int32_t batch,
                                int64_t num_blocks, int32_t min_len, unsigned int* verdict, cudaStream_t s);

constexpr unsigned int kVerdictRange = 1u;
constexpr unsigned int kVerdictOverlap = 2u;

// ---------------------------------------------------------------- decode
struct DecodeArgs {
    const void* q;
    const void* k_cache;
    const void* v_cache;
    const int32_t* tables;
    const int32_t* lens;
    void* out;
    float* partials;  // fp32 pieces of cut segments: [num_ctas][2 slots][4 warps][G*D/4 + 2G]
    int* counters;    // [batch][kv_heads][4 warps]; zero between calls
    void* trace;      // per-CTA timestamps (PKV_TRACE builds only)
    unsigned int* status;
    int64_t num_blocks;
    int32_t max_blocks;
    int32_t batch;
    int32_t q_heads;
    int32_t kv_heads;
    int32_t head_dim;
    int32_t group;  // q_heads / kv_heads
    int32_t dtype;
    int32_t num_ctas;
    int32_t test_stall;  // PKV_FLAG_TEST_STALL: the producer issues nothing
    // cost model of the CTA split (set by launch_decode): a segment of nb blocks
    // costs nb + (nb < seg_cost_below ? seg_cost : 0) + max(seg_min_cost - nb, 0)
    int32_t seg_cost;
    int32_t seg_cost_below;
    int32_t seg_min_cost;
    float scale;
    // Shared-prefix groups (null for a plain call). A sequence with a group
    // attends only its own blocks past the group's shared ones here, and its
    // rows go to fold_o / fold_lse instead of out, for the chunk-first pass
    // to combine with the shared part.
    const int32_t* prefix_group;  // [batch]: group of sequence i, or -1
    const int32_t* group_blocks;  // [num_groups]: whole blocks the group shares
    int32_t num_groups;
    int32_t max_group_blocks;     // host-side bound on group_blocks[]
    float* fold_o;                // [batch][q_heads][head_dim]: normalised output over the own tokens
    float* fold_lse;              // [batch][q_heads]: log2-sum-exp of the scaled logits, -inf if none
};

// Which kernel a decode call runs and on how many CTAs.
struct DecodePlan {
    int kernel;    // 1 CUDA-core, 2 tensor-core
    int stages;    // ring depth of the tensor-core kernel
    int num_ctas;  // CTAs of the split kernel
    size_t smem;   // dynamic shared memory of the split kernel
};

// Largest batch one launch handles (sequence prefix sums live in shared
// memory); pkv_decode_attention splits bigger batches.
constexpr int kMaxBatchPerLaunch = 1024;

// Workspace: 256-byte header (reserved), merge counters, piece slots.
struct WorkspaceLayout {
    size_t counters_offset, partials_offset, trace_offset, total;
};
WorkspaceLayout decode_workspace_layout(int batch, int kv_heads, int num_ctas, int group, int head_dim);
// `prefixed`: the call carries shared-prefix groups (a per-sequence block
// offset in shared memory; the tensor-core kernel only).
int decode_plan(const pkv_cache_desc& d, int32_t batch, int32_t q_heads, int32_t max_blocks,
                const pkv_decode_opts* opts, DecodePlan* plan, bool prefixed = false);
cudaError_t launch_decode(const DecodeArgs& a, const DecodePlan& plan, cudaStream_t s);

// 2-D TMA view of a bf16 pool: rows of head_dim elements (one token of one
// KV head), 16-row x 64-column boxes, 128-byte swizzle.
bool make_pool_map(CUtensorMap* map, const void* pool, int64_t rows, int head_dim);
// 2-D TMA view of `rows` rows of `inner` elements (PKV_INT8: uint8, else
// float32) `row_bytes` apart; boxes of box_inner x box_rows; l2_promote
// widens L2 fetches of a box to 256 bytes.
bool make_map_2d(CUtensorMap* map, int dtype, const void* base, uint64_t inner, uint64_t rows, uint64_t row_bytes,
                 uint32_t box_inner, uint32_t box_rows, bool swizzle128, bool l2_promote);

// ---------------------------------------------------------------- shared-prefix decode
// Chunk-first pass: for every group, the queries of all its members against
// the group's shared blocks, combined with the members' own-token results
// (fold_o / fold_lse, written by the decode kernel in prefixed mode).
struct PrefixArgs {
    const void* q;
    const void* k_cache;
    const void* v_cache;
    const int32_t* tables;
    const int32_t* lens;
    const int32_t* prefix_group;
    const int32_t* group_blocks;
    const float* fold_o;
    const float* fold_lse;
    void* out;
    float* partials;  // [tiles][kv_heads][chunks][rows per tile][head_dim + 2]
    int* counters;    // [tiles][kv_heads][4 warps]; zero between calls
    void* trace;      // per-CTA timestamps (PKV_TRACE builds only)
    unsigned int* status;
    int64_t num_blocks;
    int32_t max_blocks;
    int32_t batch;
    int32_t num_groups;
    int32_t max_group_blocks;
    int32_t q_heads;
    int32_t kv_heads;
    int32_t head_dim;
    int32_t group;         // q_heads / kv_heads
    int32_t tiles;         // grid x: upper bound on 64-row tiles over all groups
    int32_t chunks;        // grid y: shared-block chunks per group
    int32_t chunk_blocks;  // blocks per chunk
    float scale;
    // causal multi-query (chunked prefill) mode of the tcgen05 kernel: the
    // queries of sequence i are rows qstart[i] .. qstart[i+1]-1 of q / out
    const int32_t* qstart;
    int32_t max_query_len;
};

// Grid and workspace of the chunk-first pass for a launch of `batch`
// sequences (at most kMaxBatchPerLaunch).
struct PrefixPlan {
    int kernel;  // 1 mma.sync (64-row tiles), 2 tcgen05 (128-row tiles)
    int rows;    // query rows per tile
    int tiles, chunks, chunk_blocks;
    size_t counters_offset, partials_offset, fold_o_offset, fold_lse_offset, trace_offset, total;
};
PrefixPlan prefix_plan(int batch, int num_groups, int q_heads, int kv_heads, int head_dim, int max_group_blocks,
                       size_t base_offset, int kernel);
cudaError_t launch_prefix(const PrefixArgs& a, int kernel, cudaStream_t s);
// Causal multi-query attention with many query rows per (sequence, KV head)
// on the tcgen05 kernel: 128-row query tiles, the context split over a
// cluster; fills a.tiles / a.chunks / a.chunk_blocks.
cudaError_t launch_prefill(PrefixArgs& a, cudaStream_t s);
cudaError_t launch_check_groups(const int32_t* tables, int32_t max_blocks, const int32_t* lens,
                                const int32_t* prefix_group, const int32_t* group_blocks, int32_t num_groups,
                                int32_t max_group_blocks, int32_t batch, unsigned int* verdict, cudaStream_t s);

int device_sm_count();

// ---------------------------------------------------------------- low-bit KV
cudaError_t launch_append_q8(const void* k, const void* v, const int64_t* slots, int64_t num_tokens, void* k_codes,
                             void* v_codes, float* scales, const pkv_cache_desc& d,
                             unsigned int* status, cudaStream_t s);
cudaError_t launch_copy_scales(const int64_t* pairs, int64_t num_pairs, float* scales,
                               const pkv_cache_desc& d, unsigned int* status, cudaStream_t s);

// ---------------------------------------------------------------- multi-query decode
// Several causal queries per sequence; see pkv_multiquery.cu.
struct MqArgs {
    const void* q;          // [query_start[batch]][q_heads][head_dim] bf16
    const void* k_cache;
    const void* v_cache;
    const int32_t* tables;
    const int32_t* lens;
    const int32_t* qstart;  // [batch + 1]: first query row of each sequence (absolute rows of q / out);
                            // null: one query per sequence at row i (decode)
    void* out;
    float* partials;        // [num_ctas][2 slots][4 row groups][8 rows][head_dim + 2]
    int* counters;          // [batch][kv_heads][4 row groups]; zero between calls
    unsigned int* status;
    int64_t num_blocks;
    int32_t max_blocks;
    int32_t batch;
    int32_t q_heads;
    int32_t kv_heads;
    int32_t head_dim;
    int32_t group;
    int32_t num_ctas;
    int32_t max_query_len;  // queries per sequence, at most (32 / group)
    int32_t wpu;            // warps per unit: 1, 2 or 4 row groups of 8 (from max_query_len * group)
    float scale;
    // int8 pools (q8 != 0): k_cache / v_cache are the code pools, with this scale
    // pool: [num_blocks][kv_heads][2 (K, V)][16] float
    const float* scales;
    int32_t q8;
    int32_t test_stall;  // PKV_FLAG_TEST_STALL: the producer issues nothing
};
constexpr int kMqMaxRows = 32;      // query rows per (sequence, KV head) of the mma.sync kernel
constexpr int kMaxQueryLen = 65536;  // queries per sequence in one multi-query call
int mq_num_ctas(int head_dim, int batch, const pkv_decode_opts* opts, bool q8 = false);
size_t mq_workspace_bytes(int batch, int kv_heads, int head_dim, int num_ctas, size_t* counters_offset,
                          size_t* partials_offset);
cudaError_t launch_multiquery(const MqArgs& a, cudaStream_t s);
cudaError_t launch_check_queries(const int32_t* lens, const int32_t* qstart, int32_t batch, int32_t max_query_len,
                                 unsigned int* verdict, cudaStream_t s);

}  // namespace pkv
