// Host-side interfaces between the C ABI layer (pkv_api.cu) and the kernel
// translation units. Not part of the public ABI.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "pkv.h"

namespace pkv {

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
cudaError_t launch_check_decode(const int32_t* tables, int32_t max_blocks, const int32_t* lens, int32_t batch,
                                int64_t num_blocks, unsigned int* verdict, cudaStream_t s);

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
    float scale;
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
int decode_plan(const pkv_cache_desc& d, int32_t batch, int32_t q_heads, int32_t max_blocks,
                const pkv_decode_opts* opts, DecodePlan* plan);
cudaError_t launch_decode(const DecodeArgs& a, const DecodePlan& plan, cudaStream_t s);

int device_sm_count();

}  // namespace pkv
