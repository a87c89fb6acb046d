// The extern "C" entry points declared in include/pkv.h: argument
// validation, the optional checked mode, and dispatch to the kernels.
//
// Validation order follows the pages' rule for a rejected input: everything
// that can be checked on the host is checked before any work is enqueued, and
// in checked mode the device-resident indices are verified (and the call
// waits for the verdict) before any output byte is written.
#include <math.h>
#include <mutex>

#include "pkv.h"
#include "pkv_internal.h"

// Sticky device status ([0], PKV_DEVERR_* bits) and the verdict word of the
// current checked call ([1]). One copy per device.
static __device__ unsigned int g_pkv_status[2];

namespace pkv {

namespace {

constexpr int kMaxDevices = 64;

struct DeviceInfo {
    unsigned int* status = nullptr;
    int sm_count = 0;
};

DeviceInfo& device_info() {
    static std::mutex mu;
    static DeviceInfo info[kMaxDevices];
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 0 || dev >= kMaxDevices) dev = 0;
    std::lock_guard<std::mutex> lock(mu);
    DeviceInfo& d = info[dev];
    if (d.status == nullptr) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_pkv_status) == cudaSuccess) d.status = static_cast<unsigned int*>(p);
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess) d.sm_count = n;
    }
    return d;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Query heads of an attention call: a positive multiple of the KV heads, at
// most PKV_MAX_Q_HEADS (query-row counts per (sequence, KV head) stay 32-bit).
bool q_heads_ok(int32_t num_q_heads, const pkv_cache_desc* d) {
    return num_q_heads >= 1 && num_q_heads <= PKV_MAX_Q_HEADS && num_q_heads % d->num_kv_heads == 0;
}

// Block-table width of an attention call: the tokens of one sequence
// (max_blocks * 16) and the blocks of one launch's sequences (at most
// kMaxBatchPerLaunch of them, prefix-summed on the device) are 32-bit counts.
bool table_width_ok(int32_t batch, int32_t max_blocks) {
    const int64_t per_launch = batch < kMaxBatchPerLaunch ? batch : kMaxBatchPerLaunch;
    return max_blocks >= 1 && static_cast<int64_t>(max_blocks) * 16 < (int64_t(1) << 31) &&
           per_launch * max_blocks < (int64_t(1) << 31);
}

pkv_status check_desc(const pkv_cache_desc* d) {
    if (d == nullptr) return PKV_ERR_NULL;
    if (d->block_size != 16 || d->num_blocks < 1 || d->num_kv_heads < 1) return PKV_ERR_SHAPE;
    if (d->head_dim != 64 && d->head_dim != 128) return PKV_ERR_SHAPE;
    if (d->dtype != PKV_F32 && d->dtype != PKV_BF16) return PKV_ERR_DTYPE;
    // Rows of one pool (block, head, slot) are addressed with 32-bit coordinates.
    if (d->num_blocks * d->num_kv_heads * 16 >= (int64_t(1) << 31)) return PKV_ERR_SHAPE;
    return PKV_OK;
}

// Runs one validation launch in checked mode and waits for its verdict. The
// verdict word is one per device, so checked calls from different host
// threads take turns (each waits for its verdict before releasing it).
template <typename F>
pkv_status run_checked(F launch, cudaStream_t s) {
    static std::mutex verdict_mu;
    std::lock_guard<std::mutex> lock(verdict_mu);
    unsigned int* status = device_info().status;
    if (status == nullptr) return PKV_ERR_CUDA;
    unsigned int* verdict = status + 1;
    if (cudaMemsetAsync(verdict, 0, sizeof(unsigned int), s) != cudaSuccess) return PKV_ERR_CUDA;
    if (launch(verdict) != cudaSuccess) return PKV_ERR_CUDA;
    unsigned int host = 0;
    if (cudaMemcpyAsync(&host, verdict, sizeof(unsigned int), cudaMemcpyDeviceToHost, s) != cudaSuccess)
        return PKV_ERR_CUDA;
    if (cudaStreamSynchronize(s) != cudaSuccess) return PKV_ERR_CUDA;
    if (host & kVerdictRange) return PKV_ERR_RANGE;
    if (host & kVerdictOverlap) return PKV_ERR_OVERLAP;
    return PKV_OK;
}

pkv_status check_desc_q8(const pkv_cache_desc* d, bool attention) {
    if (d == nullptr) return PKV_ERR_NULL;
    if (d->block_size != 16 || d->num_blocks < 1 || d->num_kv_heads < 1) return PKV_ERR_SHAPE;
    if (d->head_dim != 128 && (attention || d->head_dim != 64)) return PKV_ERR_SHAPE;
    if (d->dtype != PKV_INT8) return PKV_ERR_DTYPE;
    if (d->num_blocks * d->num_kv_heads * d->head_dim >= (int64_t(1) << 31)) return PKV_ERR_SHAPE;
    return PKV_OK;
}

}  // namespace

int device_sm_count() {
    const int n = device_info().sm_count;
    return n > 0 ? n : 1;
}

}  // namespace pkv

using namespace pkv;

extern "C" {

const char* pkv_status_string(pkv_status s) {
    switch (s) {
        case PKV_OK: return "PKV_OK";
        case PKV_ERR_NULL: return "PKV_ERR_NULL";
        case PKV_ERR_SHAPE: return "PKV_ERR_SHAPE";
        case PKV_ERR_DTYPE: return "PKV_ERR_DTYPE";
        case PKV_ERR_ALIGN: return "PKV_ERR_ALIGN";
        case PKV_ERR_RANGE: return "PKV_ERR_RANGE";
        case PKV_ERR_OVERLAP: return "PKV_ERR_OVERLAP";
        case PKV_ERR_WORKSPACE: return "PKV_ERR_WORKSPACE";
        case PKV_ERR_TIMEOUT: return "PKV_ERR_TIMEOUT";
        case PKV_ERR_CUDA: return "PKV_ERR_CUDA";
        case PKV_ERR_UNSUPPORTED: return "PKV_ERR_UNSUPPORTED";
        case PKV_ERR_OUT_OF_BLOCKS: return "PKV_ERR_OUT_OF_BLOCKS";
        case PKV_ERR_UNKNOWN_SEQUENCE: return "PKV_ERR_UNKNOWN_SEQUENCE";
        case PKV_ERR_EXISTS: return "PKV_ERR_EXISTS";
        case PKV_ERR_INVARIANT: return "PKV_ERR_INVARIANT";
    }
    return "PKV_ERR_UNKNOWN";
}

int32_t pkv_version(void) { return 100; }

pkv_status pkv_append(const void* k, const void* v, const int64_t* slot_mapping, int64_t num_tokens, void* k_cache,
                      void* v_cache, const pkv_cache_desc* desc, uint32_t flags, void* stream) {
    NvtxRange nvtx_range("pkv_append");
    pkv_status st = check_desc(desc);
    if (st != PKV_OK) return st;
    if (num_tokens < 0) return PKV_ERR_SHAPE;
    if (k_cache == nullptr || v_cache == nullptr) return PKV_ERR_NULL;
    if (!aligned16(k_cache) || !aligned16(v_cache)) return PKV_ERR_ALIGN;
    if (num_tokens == 0) return PKV_OK;
    if (k == nullptr || v == nullptr || slot_mapping == nullptr) return PKV_ERR_NULL;
    if (!aligned16(k) || !aligned16(v) || (reinterpret_cast<uintptr_t>(slot_mapping) & 7u)) return PKV_ERR_ALIGN;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    unsigned int* status = device_info().status;
    if (status == nullptr) return PKV_ERR_CUDA;
    if (flags & PKV_FLAG_CHECKED) {
        if (num_tokens > 16384) return PKV_ERR_UNSUPPORTED;
        const int64_t num_slots = desc->num_blocks * 16;
        st = run_checked([&](unsigned int* verdict) { return launch_check_slots(slot_mapping, num_tokens, num_slots, verdict, s); }, s);
        if (st != PKV_OK) return st;
    }
    return launch_append(k, v, slot_mapping, num_tokens, k_cache, v_cache, *desc, status, s) == cudaSuccess
               ? PKV_OK
               : PKV_ERR_CUDA;
}

pkv_status pkv_copy_blocks(const int64_t* pairs, int64_t num_pairs, void* k_cache, void* v_cache,
                           const pkv_cache_desc* desc, uint32_t flags, void* stream) {
    NvtxRange nvtx_range("pkv_copy_blocks");
    pkv_status st = check_desc(desc);
    if (st != PKV_OK) return st;
    if (num_pairs < 0) return PKV_ERR_SHAPE;
    if (k_cache == nullptr || v_cache == nullptr) return PKV_ERR_NULL;
    if (!aligned16(k_cache) || !aligned16(v_cache)) return PKV_ERR_ALIGN;
    if (num_pairs == 0) return PKV_OK;
    if (pairs == nullptr) return PKV_ERR_NULL;
    if (reinterpret_cast<uintptr_t>(pairs) & 7u) return PKV_ERR_ALIGN;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    unsigned int* status = device_info().status;
    if (status == nullptr) return PKV_ERR_CUDA;
    if (flags & PKV_FLAG_CHECKED) {
        if (num_pairs > 16384) return PKV_ERR_UNSUPPORTED;
        st = run_checked([&](unsigned int* verdict) { return launch_check_pairs(pairs, num_pairs, desc->num_blocks, verdict, s); }, s);
        if (st != PKV_OK) return st;
    }
    return launch_copy_blocks(pairs, num_pairs, k_cache, v_cache, *desc, status, s) == cudaSuccess ? PKV_OK
                                                                                                   : PKV_ERR_CUDA;
}

size_t pkv_decode_workspace_size(int32_t batch, int32_t num_q_heads, int32_t max_blocks_per_seq,
                                 const pkv_cache_desc* desc, const pkv_decode_opts* opts) {
    if (check_desc(desc) != PKV_OK || batch < 0 || !q_heads_ok(num_q_heads, desc))
        return 0;
    DecodePlan plan;
    if (decode_plan(*desc, batch, num_q_heads, max_blocks_per_seq, opts, &plan) != PKV_OK) return 0;
    return decode_workspace_layout(batch, desc->num_kv_heads, plan.num_ctas, num_q_heads / desc->num_kv_heads,
                                   desc->head_dim)
        .total;
}

pkv_status pkv_decode_attention(const void* q, const void* k_cache, const void* v_cache, const int32_t* block_tables,
                                int32_t max_blocks_per_seq, const int32_t* context_lens, int32_t batch,
                                int32_t num_q_heads, float scale, void* out, void* workspace,
                                size_t workspace_bytes, const pkv_cache_desc* desc, uint32_t flags,
                                const pkv_decode_opts* opts, void* stream) {
    NvtxRange nvtx_range("pkv_decode_attention");
    pkv_status st = check_desc(desc);
    if (st != PKV_OK) return st;
    if (batch < 0 || !q_heads_ok(num_q_heads, desc)) return PKV_ERR_SHAPE;
    if (!isfinite(scale)) return PKV_ERR_SHAPE;
    if (opts != nullptr && opts->num_ctas < 0) return PKV_ERR_SHAPE;
    if ((flags & PKV_FLAG_TEST_STALL) && !(opts != nullptr && opts->kernel == 2)) return PKV_ERR_UNSUPPORTED;
    if (batch == 0) return PKV_OK;
    if (!table_width_ok(batch, max_blocks_per_seq)) return PKV_ERR_SHAPE;
    if (!q || !k_cache || !v_cache || !block_tables || !context_lens || !out || !workspace) return PKV_ERR_NULL;
    if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(out) ||
        (reinterpret_cast<uintptr_t>(block_tables) & 3u) || (reinterpret_cast<uintptr_t>(context_lens) & 3u) ||
        (reinterpret_cast<uintptr_t>(workspace) & 255u))
        return PKV_ERR_ALIGN;
    DecodePlan plan;
    const int rc = decode_plan(*desc, batch, num_q_heads, max_blocks_per_seq, opts, &plan);
    if (rc != PKV_OK) return static_cast<pkv_status>(rc);
    const int G = num_q_heads / desc->num_kv_heads;
    const WorkspaceLayout wl = decode_workspace_layout(batch, desc->num_kv_heads, plan.num_ctas, G, desc->head_dim);
    if (workspace_bytes < wl.total) return PKV_ERR_WORKSPACE;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    unsigned int* status = device_info().status;
    if (status == nullptr) return PKV_ERR_CUDA;
    if (flags & PKV_FLAG_CHECKED) {
        st = run_checked([&](unsigned int* verdict) {
            return launch_check_decode(block_tables, max_blocks_per_seq, context_lens, batch, desc->num_blocks,
                                       1, verdict, s);
        }, s);
        if (st != PKV_OK) return st;
    }
    const int elem = desc->dtype == PKV_BF16 ? 2 : 4;
    const int64_t row = static_cast<int64_t>(num_q_heads) * desc->head_dim * elem;
    for (int32_t b0 = 0; b0 < batch; b0 += kMaxBatchPerLaunch) {
        const int32_t nb = batch - b0 < kMaxBatchPerLaunch ? batch - b0 : kMaxBatchPerLaunch;
        DecodeArgs a{};
        a.q = static_cast<const char*>(q) + b0 * row;
        a.k_cache = k_cache;
        a.v_cache = v_cache;
        a.tables = block_tables + static_cast<int64_t>(b0) * max_blocks_per_seq;
        a.lens = context_lens + b0;
        a.out = static_cast<char*>(out) + b0 * row;
        a.partials = reinterpret_cast<float*>(static_cast<char*>(workspace) + wl.partials_offset);
        a.counters = reinterpret_cast<int*>(static_cast<char*>(workspace) + wl.counters_offset);
        a.trace = wl.trace_offset ? static_cast<char*>(workspace) + wl.trace_offset : nullptr;
        a.status = status;
        a.num_blocks = desc->num_blocks;
        a.max_blocks = max_blocks_per_seq;
        a.batch = nb;
        a.q_heads = num_q_heads;
        a.kv_heads = desc->num_kv_heads;
        a.head_dim = desc->head_dim;
        a.group = G;
        a.dtype = desc->dtype;
        a.num_ctas = plan.num_ctas;
        a.test_stall = (flags & PKV_FLAG_TEST_STALL) ? 1 : 0;
        a.scale = scale;
        if (launch_decode(a, plan, s) != cudaSuccess) return PKV_ERR_CUDA;
    }
    return PKV_OK;
}

size_t pkv_decode_prefixed_workspace_size(int32_t batch, int32_t num_q_heads, int32_t max_blocks_per_seq,
                                          int32_t num_groups, int32_t max_group_blocks, const pkv_cache_desc* desc,
                                          const pkv_decode_opts* opts) {
    if (check_desc(desc) != PKV_OK || batch < 0 || !q_heads_ok(num_q_heads, desc)) return 0;
    if (num_groups < 0 || num_groups > kMaxBatchPerLaunch || max_group_blocks < 0) return 0;
    DecodePlan plan;
    if (decode_plan(*desc, batch, num_q_heads, max_blocks_per_seq, opts, &plan, true) != PKV_OK) return 0;
    const int G = num_q_heads / desc->num_kv_heads;
    const size_t base = decode_workspace_layout(batch, desc->num_kv_heads, plan.num_ctas, G, desc->head_dim).total;
    if (plan.kernel != 2 || num_groups == 0) return base;
    return prefix_plan(batch, num_groups, num_q_heads, desc->num_kv_heads, desc->head_dim, max_group_blocks, base,
                       opts ? opts->prefix_kernel : 0)
        .total;
}

pkv_status pkv_decode_attention_prefixed(const void* q, const void* k_cache, const void* v_cache,
                                         const int32_t* block_tables, int32_t max_blocks_per_seq,
                                         const int32_t* context_lens, int32_t batch, int32_t num_q_heads,
                                         float scale, const int32_t* prefix_group, const int32_t* group_blocks,
                                         int32_t num_groups, int32_t max_group_blocks, void* out, void* workspace,
                                         size_t workspace_bytes, const pkv_cache_desc* desc, uint32_t flags,
                                         const pkv_decode_opts* opts, void* stream) {
    NvtxRange nvtx_range("pkv_decode_attention_prefixed");
    pkv_status st = check_desc(desc);
    if (st != PKV_OK) return st;
    if (num_groups < 0 || max_group_blocks < 0 || max_group_blocks > max_blocks_per_seq) return PKV_ERR_SHAPE;
    if (num_groups > kMaxBatchPerLaunch) return PKV_ERR_UNSUPPORTED;
    if (flags & PKV_FLAG_TEST_STALL) return PKV_ERR_UNSUPPORTED;
    if (num_groups > 0 && batch > 0) {
        if (prefix_group == nullptr || group_blocks == nullptr) return PKV_ERR_NULL;
        if ((reinterpret_cast<uintptr_t>(prefix_group) & 3u) || (reinterpret_cast<uintptr_t>(group_blocks) & 3u))
            return PKV_ERR_ALIGN;
    }
    if (batch < 0 || !q_heads_ok(num_q_heads, desc)) return PKV_ERR_SHAPE;
    DecodePlan plan;
    int rc = decode_plan(*desc, batch, num_q_heads, max_blocks_per_seq, opts, &plan, true);
    if (rc != PKV_OK) return static_cast<pkv_status>(rc);
    // Without groups, or where only the CUDA-core kernel applies, the groups
    // are only a hint: the plain call computes the same result.
    if (num_groups == 0 || plan.kernel != 2 || batch == 0) {
        if (num_groups > 0 && batch > 0 && (flags & PKV_FLAG_CHECKED)) {
            cudaStream_t s = static_cast<cudaStream_t>(stream);
            if (max_blocks_per_seq < 1) return PKV_ERR_SHAPE;
            st = run_checked([&](unsigned int* verdict) {
                return launch_check_groups(block_tables, max_blocks_per_seq, context_lens, prefix_group,
                                           group_blocks, num_groups, max_group_blocks, batch, verdict, s);
            }, s);
            if (st != PKV_OK) return st;
        }
        return pkv_decode_attention(q, k_cache, v_cache, block_tables, max_blocks_per_seq, context_lens, batch,
                                    num_q_heads, scale, out, workspace, workspace_bytes, desc, flags, opts, stream);
    }
    if (!isfinite(scale)) return PKV_ERR_SHAPE;
    if (opts != nullptr && opts->num_ctas < 0) return PKV_ERR_SHAPE;
    if (!table_width_ok(batch, max_blocks_per_seq)) return PKV_ERR_SHAPE;
    if (!q || !k_cache || !v_cache || !block_tables || !context_lens || !out || !workspace) return PKV_ERR_NULL;
    if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(out) ||
        (reinterpret_cast<uintptr_t>(block_tables) & 3u) || (reinterpret_cast<uintptr_t>(context_lens) & 3u) ||
        (reinterpret_cast<uintptr_t>(workspace) & 255u))
        return PKV_ERR_ALIGN;
    const int G = num_q_heads / desc->num_kv_heads;
    const WorkspaceLayout wl = decode_workspace_layout(batch, desc->num_kv_heads, plan.num_ctas, G, desc->head_dim);
    if (opts != nullptr && (opts->prefix_kernel < 0 || opts->prefix_kernel > 2)) return PKV_ERR_UNSUPPORTED;
    const PrefixPlan pp = prefix_plan(batch, num_groups, num_q_heads, desc->num_kv_heads, desc->head_dim,
                                      max_group_blocks, wl.total, opts ? opts->prefix_kernel : 0);
    if (workspace_bytes < pp.total) return PKV_ERR_WORKSPACE;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    unsigned int* status = device_info().status;
    if (status == nullptr) return PKV_ERR_CUDA;
    if (flags & PKV_FLAG_CHECKED) {
        st = run_checked([&](unsigned int* verdict) {
            cudaError_t e = launch_check_decode(block_tables, max_blocks_per_seq, context_lens, batch,
                                                desc->num_blocks, 1, verdict, s);
            if (e != cudaSuccess) return e;
            return launch_check_groups(block_tables, max_blocks_per_seq, context_lens, prefix_group, group_blocks,
                                       num_groups, max_group_blocks, batch, verdict, s);
        }, s);
        if (st != PKV_OK) return st;
    }
    char* ws = static_cast<char*>(workspace);
    const int64_t row = static_cast<int64_t>(num_q_heads) * desc->head_dim * 2;
    for (int32_t b0 = 0; b0 < batch; b0 += kMaxBatchPerLaunch) {
        const int32_t nb = batch - b0 < kMaxBatchPerLaunch ? batch - b0 : kMaxBatchPerLaunch;
        DecodeArgs a{};
        a.q = static_cast<const char*>(q) + b0 * row;
        a.k_cache = k_cache;
        a.v_cache = v_cache;
        a.tables = block_tables + static_cast<int64_t>(b0) * max_blocks_per_seq;
        a.lens = context_lens + b0;
        a.out = static_cast<char*>(out) + b0 * row;
        a.partials = reinterpret_cast<float*>(ws + wl.partials_offset);
        a.counters = reinterpret_cast<int*>(ws + wl.counters_offset);
        a.trace = wl.trace_offset ? ws + wl.trace_offset : nullptr;
        a.status = status;
        a.num_blocks = desc->num_blocks;
        a.max_blocks = max_blocks_per_seq;
        a.batch = nb;
        a.q_heads = num_q_heads;
        a.kv_heads = desc->num_kv_heads;
        a.head_dim = desc->head_dim;
        a.group = G;
        a.dtype = desc->dtype;
        a.num_ctas = plan.num_ctas;
        a.test_stall = 0;
        a.scale = scale;
        a.prefix_group = prefix_group + b0;
        a.group_blocks = group_blocks;
        a.num_groups = num_groups;
        a.max_group_blocks = max_group_blocks;
        a.fold_o = reinterpret_cast<float*>(ws + pp.fold_o_offset);
        a.fold_lse = reinterpret_cast<float*>(ws + pp.fold_lse_offset);
        if (launch_decode(a, plan, s) != cudaSuccess) return PKV_ERR_CUDA;
        PrefixArgs pa{};
        pa.q = a.q;
        pa.k_cache = k_cache;
        pa.v_cache = v_cache;
        pa.tables = a.tables;
        pa.lens = a.lens;
        pa.prefix_group = a.prefix_group;
        pa.group_blocks = group_blocks;
        pa.fold_o = a.fold_o;
        pa.fold_lse = a.fold_lse;
        pa.out = a.out;
        pa.partials = reinterpret_cast<float*>(ws + pp.partials_offset);
        pa.counters = reinterpret_cast<int*>(ws + pp.counters_offset);
        pa.trace = pp.trace_offset ? ws + pp.trace_offset : nullptr;
        pa.status = status;
        pa.num_blocks = desc->num_blocks;
        pa.max_blocks = max_blocks_per_seq;
        pa.batch = nb;
        pa.num_groups = num_groups;
        pa.max_group_blocks = max_group_blocks;
        pa.q_heads = num_q_heads;
        pa.kv_heads = desc->num_kv_heads;
        pa.head_dim = desc->head_dim;
        pa.group = G;
        pa.tiles = pp.tiles;
        pa.chunks = pp.chunks;
        pa.chunk_blocks = pp.chunk_blocks;
        pa.scale = scale;
        if (launch_prefix(pa, pp.kernel, s) != cudaSuccess) return PKV_ERR_CUDA;
    }
    return PKV_OK;
}

size_t pkv_multiquery_workspace_size(int32_t batch, int32_t num_q_heads, int32_t max_blocks_per_seq,
                                     int32_t max_query_len, const pkv_cache_desc* desc,
                                     const pkv_decode_opts* opts) {
    (void)max_blocks_per_seq;
    if (check_desc(desc) != PKV_OK || batch < 0 || !q_heads_ok(num_q_heads, desc)) return 0;
    const int G = num_q_heads / desc->num_kv_heads;
    if (desc->dtype != PKV_BF16 || max_query_len < 1 || max_query_len > kMaxQueryLen) return 0;
    if (max_query_len * G > kMqMaxRows) return 256;  // tensor-core prefill path: combines on chip
    size_t co = 0, po = 0;
    return mq_workspace_bytes(batch, desc->num_kv_heads, desc->head_dim, mq_num_ctas(desc->head_dim, batch, opts),
                              &co, &po);
}

pkv_status pkv_multiquery_attention(const void* q, const void* k_cache, const void* v_cache,
                                    const int32_t* block_tables, int32_t max_blocks_per_seq,
                                    const int32_t* context_lens, const int32_t* query_start, int32_t batch,
                                    int32_t num_q_heads, int32_t max_query_len, float scale, void* out,
                                    void* workspace, size_t workspace_bytes, const pkv_cache_desc* desc,
                                    uint32_t flags, const pkv_decode_opts* opts, void* stream) {
    NvtxRange nvtx_range("pkv_multiquery_attention");
    pkv_status st = check_desc(desc);
    if (st != PKV_OK) return st;
    if (batch < 0 || !q_heads_ok(num_q_heads, desc)) return PKV_ERR_SHAPE;
    if (!isfinite(scale) || max_query_len < 1) return PKV_ERR_SHAPE;
    if (opts != nullptr && opts->num_ctas < 0) return PKV_ERR_SHAPE;
    const int G = num_q_heads / desc->num_kv_heads;
    if (desc->dtype != PKV_BF16) return PKV_ERR_DTYPE;
    if (max_query_len > kMaxQueryLen) return PKV_ERR_UNSUPPORTED;
    const bool prefill = max_query_len * G > kMqMaxRows;  // many query rows: the tcgen05 kernel
    if (prefill && (flags & PKV_FLAG_TEST_STALL)) return PKV_ERR_UNSUPPORTED;  // the hook is the split kernel's
    if (batch == 0) return PKV_OK;
    if (!table_width_ok(batch, max_blocks_per_seq)) return PKV_ERR_SHAPE;
    if (!q || !k_cache || !v_cache || !block_tables || !context_lens || !query_start || !out || !workspace)
        return PKV_ERR_NULL;
    if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(out) ||
        (reinterpret_cast<uintptr_t>(block_tables) & 3u) || (reinterpret_cast<uintptr_t>(context_lens) & 3u) ||
        (reinterpret_cast<uintptr_t>(query_start) & 3u) || (reinterpret_cast<uintptr_t>(workspace) & 255u))
        return PKV_ERR_ALIGN;
    const int num_ctas = prefill ? 0 : mq_num_ctas(desc->head_dim, batch, opts);
    size_t co = 0, po = 0;
    const size_t need =
        prefill ? 256 : mq_workspace_bytes(batch, desc->num_kv_heads, desc->head_dim, num_ctas, &co, &po);
    if (workspace_bytes < need) return PKV_ERR_WORKSPACE;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    unsigned int* status = device_info().status;
    if (status == nullptr) return PKV_ERR_CUDA;
    if (flags & PKV_FLAG_CHECKED) {
        st = run_checked([&](unsigned int* verdict) {
            cudaError_t e = launch_check_decode(block_tables, max_blocks_per_seq, context_lens, batch,
                                                desc->num_blocks, 0, verdict, s);
            if (e != cudaSuccess) return e;
            return launch_check_queries(context_lens, query_start, batch, max_query_len, verdict, s);
        }, s);
        if (st != PKV_OK) return st;
    }
    if (prefill) {
        for (int32_t b0 = 0; b0 < batch; b0 += kMaxBatchPerLaunch) {
            PrefixArgs pa{};
            pa.q = q;
            pa.k_cache = k_cache;
            pa.v_cache = v_cache;
            pa.tables = block_tables + static_cast<int64_t>(b0) * max_blocks_per_seq;
            pa.lens = context_lens + b0;
            pa.qstart = query_start + b0;
            pa.out = out;
            pa.status = status;
            pa.num_blocks = desc->num_blocks;
            pa.max_blocks = max_blocks_per_seq;
            pa.batch = batch - b0 < kMaxBatchPerLaunch ? batch - b0 : kMaxBatchPerLaunch;
            pa.q_heads = num_q_heads;
            pa.kv_heads = desc->num_kv_heads;
            pa.head_dim = desc->head_dim;
            pa.group = G;
            pa.max_query_len = max_query_len;
            pa.scale = scale;
            if (launch_prefill(pa, s) != cudaSuccess) return PKV_ERR_CUDA;
        }
        return PKV_OK;
    }
    char* ws = static_cast<char*>(workspace);
    for (int32_t b0 = 0; b0 < batch; b0 += kMaxBatchPerLaunch) {
        const int32_t nb = batch - b0 < kMaxBatchPerLaunch ? batch - b0 : kMaxBatchPerLaunch;
        MqArgs a{};
        a.q = q;
        a.k_cache = k_cache;
        a.v_cache = v_cache;
        a.tables = block_tables + static_cast<int64_t>(b0) * max_blocks_per_seq;
        a.lens = context_lens + b0;
        a.qstart = query_start + b0;
        a.out = out;
        a.partials = reinterpret_cast<float*>(ws + po);
        a.counters = reinterpret_cast<int*>(ws + co);
        a.status = status;
        a.num_blocks = desc->num_blocks;
        a.max_blocks = max_blocks_per_seq;
        a.batch = nb;
        a.q_heads = num_q_heads;
        a.kv_heads = desc->num_kv_heads;
        a.head_dim = desc->head_dim;
        a.group = G;
        a.num_ctas = num_ctas;
        a.max_query_len = max_query_len;
        const int row_groups = (max_query_len * G + 7) / 8;
        a.wpu = row_groups <= 1 ? 1 : (row_groups <= 2 ? 2 : 4);
        a.test_stall = (flags & PKV_FLAG_TEST_STALL) ? 1 : 0;
        a.scale = scale;
        if (launch_multiquery(a, s) != cudaSuccess) return PKV_ERR_CUDA;
    }
    return PKV_OK;
}

pkv_status pkv_append_q8(const void* k, const void* v, const int64_t* slot_mapping, int64_t num_tokens, void* k_codes,
                         void* v_codes, float* scales, const pkv_cache_desc* desc, uint32_t flags, void* stream) {
    NvtxRange nvtx_range("pkv_append_q8");
    pkv_status st = check_desc_q8(desc, false);
    if (st != PKV_OK) return st;
    if (num_tokens < 0) return PKV_ERR_SHAPE;
    if (!k_codes || !v_codes || !scales) return PKV_ERR_NULL;
    if (!aligned16(k_codes) || !aligned16(v_codes) || !aligned16(scales)) return PKV_ERR_ALIGN;
    if (num_tokens == 0) return PKV_OK;
    if (k == nullptr || v == nullptr || slot_mapping == nullptr) return PKV_ERR_NULL;
    if (!aligned16(k) || !aligned16(v) || (reinterpret_cast<uintptr_t>(slot_mapping) & 7u)) return PKV_ERR_ALIGN;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    unsigned int* status = device_info().status;
    if (status == nullptr) return PKV_ERR_CUDA;
    if (flags & PKV_FLAG_CHECKED) {
        if (num_tokens > 16384) return PKV_ERR_UNSUPPORTED;
        const int64_t num_slots = desc->num_blocks * 16;
        st = run_checked([&](unsigned int* verdict) { return launch_check_slots(slot_mapping, num_tokens, num_slots, verdict, s); }, s);
        if (st != PKV_OK) return st;
    }
    return launch_append_q8(k, v, slot_mapping, num_tokens, k_codes, v_codes, scales, *desc, status, s) ==
                   cudaSuccess
               ? PKV_OK
               : PKV_ERR_CUDA;
}

pkv_status pkv_copy_blocks_q8(const int64_t* pairs, int64_t num_pairs, void* k_codes, void* v_codes, float* scales,
                              const pkv_cache_desc* desc, uint32_t flags, void* stream) {
    NvtxRange nvtx_range("pkv_copy_blocks_q8");
    pkv_status st = check_desc_q8(desc, false);
    if (st != PKV_OK) return st;
    if (num_pairs < 0) return PKV_ERR_SHAPE;
    if (!k_codes || !v_codes || !scales) return PKV_ERR_NULL;
    if (!aligned16(k_codes) || !aligned16(v_codes) || !aligned16(scales)) return PKV_ERR_ALIGN;
    if (num_pairs == 0) return PKV_OK;
    if (pairs == nullptr) return PKV_ERR_NULL;
    if (reinterpret_cast<uintptr_t>(pairs) & 7u) return PKV_ERR_ALIGN;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    unsigned int* status = device_info().status;
    if (status == nullptr) return PKV_ERR_CUDA;
    if (flags & PKV_FLAG_CHECKED) {
        if (num_pairs > 16384) return PKV_ERR_UNSUPPORTED;
        st = run_checked([&](unsigned int* verdict) { return launch_check_pairs(pairs, num_pairs, desc->num_blocks, verdict, s); }, s);
        if (st != PKV_OK) return st;
    }
    // the code pools move as whole blocks of num_kv_heads * 16 * head_dim bytes (either layout)
    if (launch_copy_blocks(pairs, num_pairs, k_codes, v_codes, *desc, status, s) != cudaSuccess) return PKV_ERR_CUDA;
    return launch_copy_scales(pairs, num_pairs, scales, *desc, status, s) == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}

size_t pkv_decode_q8_workspace_size(int32_t batch, int32_t num_q_heads, int32_t max_blocks_per_seq,
                                    int32_t max_query_len, const pkv_cache_desc* desc, const pkv_decode_opts* opts) {
    (void)max_blocks_per_seq;
    if (check_desc_q8(desc, true) != PKV_OK || batch < 0 || !q_heads_ok(num_q_heads, desc))
        return 0;
    const int G = num_q_heads / desc->num_kv_heads;
    if (max_query_len < 1 || max_query_len * G > kMqMaxRows) return 0;
    size_t co = 0, po = 0;
    return mq_workspace_bytes(batch, desc->num_kv_heads, desc->head_dim,
                              mq_num_ctas(desc->head_dim, batch, opts, true), &co, &po);
}

pkv_status pkv_decode_attention_q8(const void* q, const void* k_codes, const void* v_codes, const float* scales,
                                   const int32_t* block_tables, int32_t max_blocks_per_seq,
                                   const int32_t* context_lens, const int32_t* query_start, int32_t batch,
                                   int32_t num_q_heads, int32_t max_query_len, float scale, void* out,
                                   void* workspace, size_t workspace_bytes, const pkv_cache_desc* desc,
                                   uint32_t flags, const pkv_decode_opts* opts, void* stream) {
    NvtxRange nvtx_range("pkv_decode_attention_q8");
    pkv_status st = check_desc_q8(desc, true);
    if (st != PKV_OK) return st;
    if (batch < 0 || !q_heads_ok(num_q_heads, desc)) return PKV_ERR_SHAPE;
    if (!isfinite(scale) || max_query_len < 1) return PKV_ERR_SHAPE;
    if (opts != nullptr && opts->num_ctas < 0) return PKV_ERR_SHAPE;
    const int G = num_q_heads / desc->num_kv_heads;
    if (max_query_len * G > kMqMaxRows) return PKV_ERR_UNSUPPORTED;
    if (query_start == nullptr && max_query_len != 1) return PKV_ERR_SHAPE;
    if (batch == 0) return PKV_OK;
    if (!table_width_ok(batch, max_blocks_per_seq)) return PKV_ERR_SHAPE;
    if (!q || !k_codes || !v_codes || !scales || !block_tables || !context_lens || !out || !workspace)
        return PKV_ERR_NULL;
    if (!aligned16(q) || !aligned16(k_codes) || !aligned16(v_codes) || !aligned16(scales) || !aligned16(out) || (reinterpret_cast<uintptr_t>(block_tables) & 3u) ||
        (reinterpret_cast<uintptr_t>(context_lens) & 3u) || (reinterpret_cast<uintptr_t>(query_start) & 3u) ||
        (reinterpret_cast<uintptr_t>(workspace) & 255u))
        return PKV_ERR_ALIGN;
    const int num_ctas = mq_num_ctas(desc->head_dim, batch, opts, true);
    size_t co = 0, po = 0;
    const size_t need = mq_workspace_bytes(batch, desc->num_kv_heads, desc->head_dim, num_ctas, &co, &po);
    if (workspace_bytes < need) return PKV_ERR_WORKSPACE;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    unsigned int* status = device_info().status;
    if (status == nullptr) return PKV_ERR_CUDA;
    if (flags & PKV_FLAG_CHECKED) {
        st = run_checked([&](unsigned int* verdict) {
            cudaError_t e = launch_check_decode(block_tables, max_blocks_per_seq, context_lens, batch,
                                                desc->num_blocks, query_start ? 0 : 1, verdict, s);
            if (e != cudaSuccess || query_start == nullptr) return e;
            return launch_check_queries(context_lens, query_start, batch, max_query_len, verdict, s);
        }, s);
        if (st != PKV_OK) return st;
    }
    char* ws = static_cast<char*>(workspace);
    const int64_t row = static_cast<int64_t>(num_q_heads) * desc->head_dim * 2;
    for (int32_t b0 = 0; b0 < batch; b0 += kMaxBatchPerLaunch) {
        const int32_t nb = batch - b0 < kMaxBatchPerLaunch ? batch - b0 : kMaxBatchPerLaunch;
        MqArgs a{};
        // with query offsets the rows are absolute; without, row i of this launch is sequence b0 + i
        a.q = query_start ? q : static_cast<const char*>(q) + b0 * row;
        a.out = query_start ? out : static_cast<char*>(out) + b0 * row;
        a.qstart = query_start ? query_start + b0 : nullptr;
        a.k_cache = k_codes;
        a.v_cache = v_codes;
        a.scales = scales;
        a.q8 = 1;
        a.tables = block_tables + static_cast<int64_t>(b0) * max_blocks_per_seq;
        a.lens = context_lens + b0;
        a.partials = reinterpret_cast<float*>(ws + po);
        a.counters = reinterpret_cast<int*>(ws + co);
        a.status = status;
        a.num_blocks = desc->num_blocks;
        a.max_blocks = max_blocks_per_seq;
        a.batch = nb;
        a.q_heads = num_q_heads;
        a.kv_heads = desc->num_kv_heads;
        a.head_dim = desc->head_dim;
        a.group = G;
        a.num_ctas = num_ctas;
        a.max_query_len = max_query_len;
        const int row_groups = (max_query_len * G + 7) / 8;
        a.wpu = row_groups <= 1 ? 1 : (row_groups <= 2 ? 2 : 4);
        a.test_stall = (flags & PKV_FLAG_TEST_STALL) ? 1 : 0;
        a.scale = scale;
        if (launch_multiquery(a, s) != cudaSuccess) return PKV_ERR_CUDA;
    }
    return PKV_OK;
}

pkv_status pkv_device_status(uint32_t* bits_out, int clear, void* stream) {
    unsigned int* status = device_info().status;
    if (status == nullptr) return PKV_ERR_CUDA;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    unsigned int host = 0;
    if (cudaMemcpyAsync(&host, status, sizeof(unsigned int), cudaMemcpyDeviceToHost, s) != cudaSuccess)
        return PKV_ERR_CUDA;
    if (cudaStreamSynchronize(s) != cudaSuccess) return PKV_ERR_CUDA;
    if (clear) {
        if (cudaMemsetAsync(status, 0, sizeof(unsigned int), s) != cudaSuccess) return PKV_ERR_CUDA;
        if (cudaStreamSynchronize(s) != cudaSuccess) return PKV_ERR_CUDA;
    }
    if (bits_out) *bits_out = host;
    return PKV_OK;
}

}  // extern "C"
