// Low-bit (int8) paged KV: the quantizing slot-mapped append and the scale
// half of the copy-on-write block copy.
//
// Per row (one token of one KV head, head_dim coordinates), symmetric
// quantization as in the notebook's project demo (`fake_quantize_rows`),
// with the scale stored as a float32: scale = max|x| / 127 (IEEE float32
// division; 1 for a zero row), code = clip(rint(x / scale), -127, 127) with
// the quotient taken in float64 against that stored scale and rounded half to
// even, so the codes are a function of what the cache keeps. A row of bf16
// inputs is exact in float32, so its maximum is too.
//
// The float64 decision is reproduced exactly in float32 arithmetic (FP64 is
// slow on this part): x and the scale carry 24-bit significands, so x / scale
// is either exactly a half-integer or at least 2^-25 away from one, farther
// than the float64 rounding of the quotient (< 2^-46 at |q| < 128) can move
// it; the float64 rint is therefore the nearest integer to the exact quotient,
// ties to even. A float32 quotient gives a candidate within one of it, and two
// fused multiply-adds decide the sides of c - 1/2 and c + 1/2 exactly (the
// sign of a fused x - (c +- 1/2) * scale is that of the exact difference,
// and it is zero only for a tie). Normal-range inputs; subnormal scales (rows
// below ~1e-36) are outside what this argument covers.
//
// Layouts: K codes [num_blocks][Hkv][16][D] (token rows), V codes
// [num_blocks][Hkv][D][16] (the 16 token codes of one coordinate together,
// the order the decode kernel feeds the tensor cores), scales
// [num_blocks][Hkv][2][16] float32 (per block and head one 128-byte record:
// the K-row scales, then the V-row scales).
#include <math.h>

#include "pkv_device.cuh"
#include "pkv_internal.h"

namespace pkv {
namespace {

// Nearest integer to the exact x / scale, ties to even, clipped to +-127.
__device__ __forceinline__ int code_of(float x, float scale) {
    float c = rintf(__fdiv_rn(x, scale));
    const float up = fmaf(-(c + 0.5f), scale, x);  // sign of x - (c + 1/2) scale
    const float dn = fmaf(-(c - 0.5f), scale, x);  // sign of x - (c - 1/2) scale
    const bool odd = (static_cast<int>(c) & 1) != 0;
    if (up > 0.f || (up == 0.f && odd)) c += 1.f;
    else if (dn < 0.f || (dn == 0.f && odd)) c -= 1.f;
    return static_cast<int>(fminf(fmaxf(c, -127.f), 127.f));
}

// One warp per (token, KV head, pool): lane l holds coordinates
// [l * D/32, (l+1) * D/32).
template <int D>
__global__ void __launch_bounds__(64) append_q8_kernel(const __nv_bfloat16* __restrict__ k,
                                                        const __nv_bfloat16* __restrict__ v,
                                                        const int64_t* __restrict__ slots, int64_t num_tokens,
                                                        int8_t* __restrict__ kc, int8_t* __restrict__ vc,
                                                        float* __restrict__ scales, int64_t num_slots, int kv_heads,
                                                        unsigned int* status) {
    constexpr int kPer = D / 32;
    grid_dependency_wait();  // a block copy before us may target the same block
    allow_dependents();
    const int lane = threadIdx.x & 31;
    const int64_t rows = num_tokens * kv_heads * 2;
    const int64_t wstride = static_cast<int64_t>(gridDim.x) * (blockDim.x >> 5);
    for (int64_t w = static_cast<int64_t>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5); w < rows;
         w += wstride) {
        const bool is_v = w >= num_tokens * kv_heads;
        const int64_t r = is_v ? w - num_tokens * kv_heads : w;  // token * kv_heads + head
        const int64_t t = r / kv_heads;
        const int h = static_cast<int>(r - t * kv_heads);
        const int64_t s = slots[t];
        if (s < 0) continue;
        if (s >= num_slots) {
            if (!is_v && h == 0 && lane == 0) atomicOr(status, PKV_DEVERR_RANGE);
            continue;
        }
        const __nv_bfloat16* src = (is_v ? v : k) + r * D + lane * kPer;
        float x[kPer];
        float amax = 0.f;
#pragma unroll
        for (int e = 0; e < kPer; ++e) {
            x[e] = __bfloat162float(src[e]);
            amax = fmaxf(amax, fabsf(x[e]));
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
        const float scale = amax > 0.f ? __fdiv_rn(amax, 127.0f) : 1.0f;
        int8_t c[kPer];
#pragma unroll
        for (int e = 0; e < kPer; ++e) c[e] = static_cast<int8_t>(code_of(x[e], scale));
        const int64_t blk = s >> 4, slot = s & 15;
        const int64_t bh = blk * kv_heads + h;
        if (!is_v) {
            int8_t* dst = kc + (bh * 16 + slot) * D + lane * kPer;
#pragma unroll
            for (int e = 0; e < kPer; ++e) dst[e] = c[e];
        } else {
#pragma unroll
            for (int e = 0; e < kPer; ++e) vc[(bh * D + lane * kPer + e) * 16 + slot] = c[e];
        }
        if (lane == 0) scales[(bh * 2 + (is_v ? 1 : 0)) * 16 + slot] = scale;  // the (block, head) record
    }
}

// Copy-on-write of the scales: a block's records are kv_heads * 32 contiguous
// floats (K and V rows of every head), moved as float4.
__global__ void __launch_bounds__(256) copy_scales_kernel(const int64_t* __restrict__ pairs, int64_t num_pairs,
                                                          float4* __restrict__ scales, int64_t num_blocks,
                                                          int per_block, unsigned int* status) {
    grid_dependency_wait();
    allow_dependents();
    const int64_t total = num_pairs * per_block;
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    for (int64_t idx = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; idx < total; idx += stride) {
        const int64_t p = idx / per_block;
        const int64_t c = idx - p * per_block;
        const int64_t src = pairs[2 * p], dst = pairs[2 * p + 1];
        if (src < 0 || src >= num_blocks || dst < 0 || dst >= num_blocks) {
            if (c == 0) atomicOr(status, PKV_DEVERR_RANGE);
            continue;
        }
        scales[dst * per_block + c] = scales[src * per_block + c];
    }
}

int grid_of(int64_t work, int per_block) {
    const int64_t want = (work + per_block - 1) / per_block;
    const int64_t cap = static_cast<int64_t>(device_sm_count()) * 16;
    return static_cast<int>(want < cap ? (want < 1 ? 1 : want) : cap);
}

}  // namespace

cudaError_t launch_append_q8(const void* k, const void* v, const int64_t* slots, int64_t num_tokens, void* k_codes,
                             void* v_codes, float* scales, const pkv_cache_desc& d, unsigned int* status,
                             cudaStream_t s) {
    const int64_t warps = num_tokens * d.num_kv_heads * 2;
    const int grid = grid_of(warps, 2);  // 64-thread CTAs: a decode step's few hundred rows reach every SM
    const int64_t num_slots = d.num_blocks * 16;
    const auto* kb = static_cast<const __nv_bfloat16*>(k);
    const auto* vb = static_cast<const __nv_bfloat16*>(v);
    auto* kc = static_cast<int8_t*>(k_codes);
    auto* vc = static_cast<int8_t*>(v_codes);
    if (d.head_dim == 128)
        return launch_pdl(append_q8_kernel<128>, dim3(grid), dim3(64), 0, s, kb, vb, slots, num_tokens, kc, vc,
                          scales, num_slots, d.num_kv_heads, status);
    return launch_pdl(append_q8_kernel<64>, dim3(grid), dim3(64), 0, s, kb, vb, slots, num_tokens, kc, vc, scales,
                      num_slots, d.num_kv_heads, status);
}

cudaError_t launch_copy_scales(const int64_t* pairs, int64_t num_pairs, float* scales, const pkv_cache_desc& d,
                               unsigned int* status, cudaStream_t s) {
    const int per_block = d.num_kv_heads * 32 / 4;  // float4 per block
    const int grid = grid_of(num_pairs * per_block, 256);
    return launch_pdl(copy_scales_kernel, dim3(grid), dim3(256), 0, s, pairs, num_pairs,
                      reinterpret_cast<float4*>(scales), d.num_blocks, per_block, status);
}

}  // namespace pkv
