// pkv_decode_attention_noalloc: decode attention for callers that cannot
// allocate device memory.
//
// pkv_decode_attention needs a caller-provided workspace (the fp32 pieces of
// context segments split across CTAs and the counters that decide which CTA
// merges them). Some callers have no way to provide one: a plugin that runs
// inside a host framework whose memory pool it does not own, code on a
// latency-critical path where cudaMalloc's implicit device synchronisation is
// not acceptable, or a deployment with a fixed device-memory budget set at
// start-up. For them this file holds a fixed scratch array in the library
// itself and runs the same decode kernel on it.
//
// The array below lives in device memory on every GPU that loads the library,
// from module load until the process exits. Its size is the hard limit of
// this entry point.
#include <mutex>

#include "pkv.h"
#include "pkv_internal.h"

// PKV_NOALLOC_SCRATCH_BYTES (4 MiB) of workspace shared by every call of
// pkv_decode_attention_noalloc on a device. Static device memory starts out
// zero-filled.
static __device__ __align__(256) unsigned char g_pkv_noalloc_scratch[PKV_NOALLOC_SCRATCH_BYTES];

namespace {

constexpr int kMaxDevices = 64;

// Device address of the scratch array for the current device. In host code
// the array's name is only a host-side stand-in, so the address is looked up
// once per device (with that device current) and cached. Returns nullptr if
// the lookup fails.
unsigned char* scratch_address() {
    static std::mutex mu;
    static unsigned char* addr[kMaxDevices] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    std::lock_guard<std::mutex> lock(mu);
    if (addr[dev] == nullptr) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_pkv_noalloc_scratch) != cudaSuccess) return nullptr;
        addr[dev] = static_cast<unsigned char*>(p);
    }
    return addr[dev];
}

}  // namespace

extern "C" pkv_status pkv_decode_attention_noalloc(const void* q, const void* k_cache, const void* v_cache,
                                                   const int32_t* block_tables, int32_t max_blocks_per_seq,
                                                   const int32_t* context_lens, int32_t batch,
                                                   int32_t num_q_heads, float scale, void* out,
                                                   const pkv_cache_desc* desc, uint32_t flags,
                                                   const pkv_decode_opts* opts, void* stream) {
    if (desc == nullptr) return PKV_ERR_NULL;
    if (batch == 0) return pkv_decode_attention(q, k_cache, v_cache, block_tables, max_blocks_per_seq,
                                                context_lens, batch, num_q_heads, scale, out, nullptr, 0, desc,
                                                flags, opts, stream);
    const size_t need = pkv_decode_workspace_size(batch, num_q_heads, max_blocks_per_seq, desc, opts);
    if (need == 0) {
        // invalid geometry or options: let the regular entry point name the fault
        const pkv_status st = pkv_decode_attention(q, k_cache, v_cache, block_tables, max_blocks_per_seq,
                                                   context_lens, batch, num_q_heads, scale, out, nullptr, 0, desc,
                                                   flags, opts, stream);
        return st != PKV_OK ? st : PKV_ERR_SHAPE;
    }
    // Sizes whose workspace would not fit the fixed array are refused.
    if (need > PKV_NOALLOC_SCRATCH_BYTES) return PKV_ERR_WORKSPACE;
    unsigned char* scratch = scratch_address();
    if (scratch == nullptr) return PKV_ERR_CUDA;
    // The array keeps whatever the last call left in it. The merge counters
    // must start at zero; a completed call leaves them at zero, but one that
    // stopped early may not, so clear them every time (a memset, no
    // allocation).
    // Header and counters sit before the piece slots, whatever the CTA count.
    const size_t counters_bytes = pkv::decode_workspace_layout(batch, desc->num_kv_heads, 0,
                                                                num_q_heads / desc->num_kv_heads, desc->head_dim)
                                      .partials_offset;
    if (cudaMemsetAsync(scratch, 0, counters_bytes, static_cast<cudaStream_t>(stream)) != cudaSuccess)
        return PKV_ERR_CUDA;
    return pkv_decode_attention(q, k_cache, v_cache, block_tables, max_blocks_per_seq, context_lens, batch,
                                num_q_heads, scale, out, scratch, PKV_NOALLOC_SCRATCH_BYTES, desc, flags, opts,
                                stream);
}
