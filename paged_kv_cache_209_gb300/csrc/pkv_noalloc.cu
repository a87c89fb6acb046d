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
#include <cuda.h>

#include <mutex>

#include "pkv.h"
#include "pkv_internal.h"

// PKV_NOALLOC_SCRATCH_BYTES (4 MiB) of workspace shared by every call of
// pkv_decode_attention_noalloc on a device. Static device memory starts out
// zero-filled.
static __device__ __align__(256) unsigned char g_pkv_noalloc_scratch[PKV_NOALLOC_SCRATCH_BYTES];

namespace {

constexpr int kMaxDevices = 64;

using CtxGetCurrentFn = CUresult (*)(CUcontext*);
using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long*);

// Process-unique id of the context current on this thread (0 if the driver
// cannot say). A cudaDeviceReset destroys the device's primary context, and
// the array with it; the runtime's next call creates a new context with a new
// id, where the array has a new address.
unsigned long long current_context_id() {
    static CtxGetCurrentFn get_current = nullptr;
    static CtxGetIdFn get_id = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_current = reinterpret_cast<CtxGetCurrentFn>(f);
        f = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_id = reinterpret_cast<CtxGetIdFn>(f);
    });
    if (get_current == nullptr || get_id == nullptr) return 0;
    CUcontext ctx = nullptr;
    unsigned long long id = 0;
    if (get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr || get_id(ctx, &id) != CUDA_SUCCESS) return 0;
    return id;
}

// Device address of the scratch array for the current device. In host code
// the array's name is only a host-side stand-in, so the address is looked up
// (with the device current) at set-up: on the first call on a device, and
// again on the first call after the device's context was replaced (a
// cudaDeviceReset). Returns nullptr if the lookup fails.
unsigned char* scratch_address() {
    static std::mutex mu;
    static unsigned char* addr[kMaxDevices] = {};
    static unsigned long long ctx_of[kMaxDevices] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    unsigned long long ctx = current_context_id();
    if (ctx == 0 && cudaSetDevice(dev) == cudaSuccess) ctx = current_context_id();  // make the primary context current
    std::lock_guard<std::mutex> lock(mu);
    if (addr[dev] == nullptr || ctx != ctx_of[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_pkv_noalloc_scratch) != cudaSuccess) return nullptr;
        addr[dev] = static_cast<unsigned char*>(p);
        ctx_of[dev] = ctx;
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
    pkv::NvtxRange nvtx_range("pkv_decode_attention_noalloc");
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
