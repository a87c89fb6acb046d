// Slot-mapped append and copy-on-write block copy (plus the validation
// kernels of PKV_FLAG_CHECKED).
//
// Both moves are pure byte copies in 16-byte vectors: a (token, KV head) row
// of head_dim elements is 128..512 bytes, a whole block of one pool is
// num_kv_heads * 16 rows. Consecutive threads take consecutive vectors of one
// row, so every warp reads and writes whole 32-byte sectors.
#include "pkv_device.cuh"
#include "pkv_internal.h"

namespace pkv {
namespace {

constexpr int kThreads = 256;

int grid_for(int64_t work, int threads) {
    const int64_t want = (work + threads - 1) / threads;
    const int64_t cap = static_cast<int64_t>(device_sm_count()) * 16;
    return static_cast<int>(want < cap ? (want < 1 ? 1 : want) : cap);
}

// Token t, head h, vector c of k/v goes to pool vector
// ((slot/16 * Hkv + h) * 16 + slot%16) * vecs_per_row + c.
__global__ void __launch_bounds__(kThreads) append_kernel(const uint4* __restrict__ k, const uint4* __restrict__ v,
                                                          const int64_t* __restrict__ slots, int64_t per_pool,
                                                          uint4* __restrict__ kc, uint4* __restrict__ vc,
                                                          int64_t num_slots, int kv_heads, int vecs_per_row,
                                                          unsigned int* status) {
    grid_dependency_wait();  // a block copy before us may target the same block
    allow_dependents();
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    for (int64_t idx = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; idx < 2 * per_pool;
         idx += stride) {
        const bool is_v = idx >= per_pool;
        const int64_t r = is_v ? idx - per_pool : idx;
        const int64_t row = r / vecs_per_row;
        const int c = static_cast<int>(r - row * vecs_per_row);
        const int64_t t = row / kv_heads;
        const int h = static_cast<int>(row - t * kv_heads);
        const int64_t s = slots[t];
        if (s < 0) continue;
        if (s >= num_slots) {
            if (!is_v && h == 0 && c == 0) atomicOr(status, PKV_DEVERR_RANGE);
            continue;
        }
        const int64_t dst = (((s >> 4) * kv_heads + h) * 16 + (s & 15)) * vecs_per_row + c;
        if (is_v)
            vc[dst] = v[r];
        else
            kc[dst] = k[r];
    }
}

__global__ void __launch_bounds__(kThreads) copy_kernel(const int64_t* __restrict__ pairs, int64_t num_pairs,
                                                        uint4* __restrict__ kc, uint4* __restrict__ vc,
                                                        int64_t num_blocks, int64_t block_vecs,
                                                        unsigned int* status) {
    grid_dependency_wait();
    allow_dependents();
    const int64_t per_pair = 2 * block_vecs;
    const int64_t total = num_pairs * per_pair;
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    for (int64_t idx = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; idx < total; idx += stride) {
        const int64_t p = idx / per_pair;
        int64_t c = idx - p * per_pair;
        const bool is_v = c >= block_vecs;
        if (is_v) c -= block_vecs;
        const int64_t src = pairs[2 * p];
        const int64_t dst = pairs[2 * p + 1];
        if (src < 0 || src >= num_blocks || dst < 0 || dst >= num_blocks) {
            if (c == 0 && !is_v) atomicOr(status, PKV_DEVERR_RANGE);
            continue;
        }
        uint4* pool = is_v ? vc : kc;
        pool[dst * block_vecs + c] = pool[src * block_vecs + c];
    }
}

__global__ void check_slots_kernel(const int64_t* __restrict__ slots, int64_t n, int64_t num_slots,
                                   unsigned int* verdict) {
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n; i += stride) {
        const int64_t s = slots[i];
        if (s < 0) continue;
        if (s >= num_slots) atomicOr(verdict, kVerdictRange);
        for (int64_t j = i + 1; j < n; ++j)
            if (slots[j] == s) {
                atomicOr(verdict, kVerdictOverlap);
                break;
            }
    }
}

__global__ void check_pairs_kernel(const int64_t* __restrict__ pairs, int64_t n, int64_t num_blocks,
                                   unsigned int* verdict) {
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n; i += stride) {
        const int64_t src = pairs[2 * i], dst = pairs[2 * i + 1];
        if (src < 0 || src >= num_blocks || dst < 0 || dst >= num_blocks) atomicOr(verdict, kVerdictRange);
        for (int64_t j = 0; j < n; ++j) {
            if (j != i && pairs[2 * j + 1] == dst) atomicOr(verdict, kVerdictOverlap);
            if (pairs[2 * j] == dst) atomicOr(verdict, kVerdictOverlap);
        }
    }
}

__global__ void check_decode_kernel(const int32_t* __restrict__ tables, int32_t max_blocks,
                                    const int32_t* __restrict__ lens, int32_t batch, int64_t num_blocks,
                                    int32_t min_len, unsigned int* verdict) {
    for (int i = blockIdx.x; i < batch; i += gridDim.x) {
        const int32_t n = lens[i];
        if (n < min_len || static_cast<int64_t>(n) > static_cast<int64_t>(max_blocks) * 16) {
            if (threadIdx.x == 0) atomicOr(verdict, kVerdictRange);
            continue;
        }
        const int nb = (n + 15) / 16;
        for (int b = threadIdx.x; b < nb; b += blockDim.x) {
            const int32_t id = tables[static_cast<int64_t>(i) * max_blocks + b];
            if (id < 0 || id >= num_blocks) atomicOr(verdict, kVerdictRange);
        }
    }
}

int elem_bytes(int dtype) { return dtype == PKV_BF16 ? 2 : (dtype == PKV_INT8 ? 1 : 4); }

}  // namespace

cudaError_t launch_append(const void* k, const void* v, const int64_t* slots, int64_t num_tokens, void* k_cache,
                          void* v_cache, const pkv_cache_desc& d, unsigned int* status, cudaStream_t s) {
    const int vecs_per_row = d.head_dim * elem_bytes(d.dtype) / 16;
    const int64_t per_pool = num_tokens * d.num_kv_heads * vecs_per_row;
    return launch_pdl(append_kernel, dim3(grid_for(2 * per_pool, kThreads)), dim3(kThreads), 0, s,
                      static_cast<const uint4*>(k), static_cast<const uint4*>(v), slots, per_pool,
                      static_cast<uint4*>(k_cache), static_cast<uint4*>(v_cache), d.num_blocks * 16, d.num_kv_heads,
                      vecs_per_row, status);
}

cudaError_t launch_copy_blocks(const int64_t* pairs, int64_t num_pairs, void* k_cache, void* v_cache,
                               const pkv_cache_desc& d, unsigned int* status, cudaStream_t s) {
    const int64_t block_vecs = static_cast<int64_t>(d.num_kv_heads) * 16 * d.head_dim * elem_bytes(d.dtype) / 16;
    return launch_pdl(copy_kernel, dim3(grid_for(num_pairs * 2 * block_vecs, kThreads)), dim3(kThreads), 0, s,
                      pairs, num_pairs, static_cast<uint4*>(k_cache), static_cast<uint4*>(v_cache), d.num_blocks,
                      block_vecs, status);
}

cudaError_t launch_check_slots(const int64_t* slots, int64_t n, int64_t num_slots, unsigned int* verdict,
                               cudaStream_t s) {
    check_slots_kernel<<<grid_for(n, 128), 128, 0, s>>>(slots, n, num_slots, verdict);
    return cudaGetLastError();
}

cudaError_t launch_check_pairs(const int64_t* pairs, int64_t n, int64_t num_blocks, unsigned int* verdict,
                               cudaStream_t s) {
    check_pairs_kernel<<<grid_for(n, 128), 128, 0, s>>>(pairs, n, num_blocks, verdict);
    return cudaGetLastError();
}

cudaError_t launch_check_decode(const int32_t* tables, int32_t max_blocks, const int32_t* lens, int32_t batch,
                                int64_t num_blocks, int32_t min_len, unsigned int* verdict, cudaStream_t s) {
    const int grid = batch < 1024 ? batch : 1024;
    check_decode_kernel<<<grid, 256, 0, s>>>(tables, max_blocks, lens, batch, num_blocks, min_len, verdict);
    return cudaGetLastError();
}

}  // namespace pkv
