/*
 * pkv.h -- C ABI of the paged KV-cache decode path for GB300 (sm_103a).
 *
 * The problem (release page "NeuralOps v1.3.4: Serving Primitives & KV Cache
 * Optimization", Architectural Breakdown 1 "Paged KV Cache Engine"): attention
 * K/V memory is cut into fixed 16-token physical blocks; a per-sequence block
 * table maps logical tokens to physical blocks; new tokens are written
 * through a slot mapping; a block is added only when a sequence crosses a
 * block boundary. "Notebook 10. KV cache and serving: bytes, pages, and
 * ceilings", section 5, adds prefix sharing with copy-on-write of a shared
 * partial final block.
 *
 * Cache layout (one layer): two pools, K and V, each
 *     pool[num_blocks][num_kv_heads][16][head_dim]
 * contiguous, row-major, elements of `dtype`, base address 16-byte aligned
 * (1024-byte alignment recommended). A slot id is `block_id * 16 + offset`.
 * Logical token t of sequence i lives in block block_tables[i][t / 16] at
 * offset t % 16.
 *
 * Conventions shared by every call:
 *  - All pointers named *device* are CUDA device pointers on the current
 *    device; the caller owns every buffer (including the workspace) and the
 *    library allocates no device memory.
 *  - Work is enqueued on `stream` (a cudaStream_t; NULL = legacy default
 *    stream) and returns without waiting, except in PKV_FLAG_CHECKED mode.
 *  - Host-visible arguments are validated before anything is enqueued. A call
 *    that returns an error status has written no byte of any output buffer
 *    (notebook "PyTorch bridge - B17": inputs are checked before any state
 *    changes, and a rejected input leaves the old state as it was; notebook
 *    section 5: running out of blocks never leaves a half-updated pool).
 *  - Indices that live in device memory (slot ids, block ids, context
 *    lengths, copy pairs) are checked on the device:
 *      * default (fast) mode: an out-of-range entry is never dereferenced; it
 *        is skipped (append/copy) or treated as an absent token (attention),
 *        and bit PKV_DEVERR_RANGE is set in the sticky device status that
 *        pkv_device_status() reads.
 *      * PKV_FLAG_CHECKED: a validation kernel runs first, the call waits for
 *        it, and a bad index returns PKV_ERR_RANGE / PKV_ERR_OVERLAP with
 *        nothing written.
 *  - Every wait inside a kernel is bounded; if one runs out the kernel stops,
 *    sets PKV_DEVERR_TIMEOUT in the sticky device status and returns.
 *  - Attention calls take num_q_heads, a positive multiple of the pool's
 *    num_kv_heads and at most PKV_MAX_Q_HEADS (else PKV_ERR_SHAPE; the
 *    workspace-size queries return 0), so that row and tile counts such as
 *    max_query_len * num_q_heads / num_kv_heads stay 32-bit. Likewise
 *    max_blocks_per_seq * 16 and max_blocks_per_seq * min(batch, 1024) must
 *    stay below 2^31 (else PKV_ERR_SHAPE).
 */
#ifndef PKV_H
#define PKV_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define PKV_API __attribute__((visibility("default")))
#else
#define PKV_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    PKV_OK = 0,
    PKV_ERR_NULL = 1,        /* a required pointer is NULL                     */
    PKV_ERR_SHAPE = 2,       /* a size or geometry field is invalid            */
    PKV_ERR_DTYPE = 3,       /* unsupported element type                       */
    PKV_ERR_ALIGN = 4,       /* a pointer is not 16-byte aligned               */
    PKV_ERR_RANGE = 5,       /* a device-resident index is out of range        */
    PKV_ERR_OVERLAP = 6,     /* duplicate slots / copy destinations            */
    PKV_ERR_WORKSPACE = 7,   /* workspace NULL or smaller than required        */
    PKV_ERR_TIMEOUT = 8,     /* a bounded in-kernel wait ran out               */
    PKV_ERR_CUDA = 9,        /* a CUDA runtime call failed                     */
    PKV_ERR_UNSUPPORTED = 10, /* valid request this build does not implement   */
    PKV_ERR_OUT_OF_BLOCKS = 11, /* block pool: not enough free blocks            */
    PKV_ERR_UNKNOWN_SEQUENCE = 12, /* block pool: no such sequence               */
    PKV_ERR_EXISTS = 13,      /* block pool: the sequence already exists         */
    PKV_ERR_INVARIANT = 14    /* block pool: an internal invariant is broken     */
} pkv_status;

/* PKV_INT8: the low-bit pools of pkv_append_q8 / pkv_decode_attention_q8
 * (int8 codes plus one float32 scale per token row of a KV head). */
typedef enum { PKV_F32 = 0, PKV_BF16 = 1, PKV_INT8 = 2 } pkv_dtype;

/* Geometry of one layer's K and V pools. */
typedef struct {
    int64_t num_blocks;    /* physical blocks in each pool, >= 1              */
    int32_t block_size;    /* tokens per block; must be 16                     */
    int32_t num_kv_heads;  /* KV heads stored per token, >= 1                  */
    int32_t head_dim;      /* 64 or 128                                        */
    int32_t dtype;         /* pkv_dtype of pools, new K/V, q and out           */
} pkv_cache_desc;

/* flags */
#define PKV_FLAG_CHECKED 1u    /* validate device-resident indices first (syncs) */
/* Test hook for failure detection, on pkv_decode_attention with the
 * tensor-core kernel (opts->kernel == 2), on pkv_multiquery_attention up to 32
 * query rows per (sequence, KV head) and on pkv_decode_attention_q8: the
 * kernel's producer warp issues no copies, so every consumer wait runs out
 * after 20 ms instead of 2 s. The call itself returns PKV_OK; the sticky device
 * status then reports PKV_DEVERR_TIMEOUT and `out` holds no result. Nothing is
 * in flight when the kernel returns. Elsewhere the flag is PKV_ERR_UNSUPPORTED. */
#define PKV_FLAG_TEST_STALL 0x80000000u

/* Bits of the sticky device status (pkv_device_status). */
/* Largest num_q_heads an attention call accepts. */
#define PKV_MAX_Q_HEADS 1024

#define PKV_DEVERR_TIMEOUT 1u
#define PKV_DEVERR_RANGE 2u

/* Decode tuning. Pass NULL for the defaults. */
typedef struct {
    int32_t kernel;     /* 0 = choose; 1 = CUDA-core kernel; 2 = tensor-core
                           (mma.sync) kernel: bf16 only, head_dim 64/128,
                           at most 8 query heads per KV head               */
    int32_t num_ctas;   /* 0 = one wave of resident CTAs; > 0 forces that
                           many CTAs (tests use it to force context splits) */
    int32_t stages;     /* tensor-core kernel ring depth: 0 = default (8), 8 or 12 */
    int32_t prefix_kernel; /* shared-prefix pass of pkv_decode_attention_prefixed:
                              0 = choose (2); 1 = mma.sync kernel, 64-row tiles;
                              2 = tcgen05 kernel, 128-row tiles              */
} pkv_decode_opts;

/*
 * pkv_append -- slot-mapped write of one step's new K/V.
 * (release page, Highlights "slot mapping" and Architectural Breakdown 1
 * "Fragment-Free Growth"; notebook section 5 `append`.)
 *
 * For each token t < num_tokens with s = slot_mapping[t] >= 0, and each KV
 * head h:  k_cache[s/16][h][s%16][:] = k[t][h][:]  and the same for v.
 * s < 0 skips the token (padding).
 *
 *   k, v          device, [num_tokens][num_kv_heads][head_dim] of desc->dtype,
 *                 contiguous, 16-byte aligned. Read only.
 *   slot_mapping  device, int64 [num_tokens]. Read only.
 *   k_cache,
 *   v_cache       device pools (layout above). Written at the named slots only.
 *   num_tokens    >= 0; 0 enqueues nothing.
 * Errors: NULL pointers, bad geometry, misalignment (host-side); with
 * PKV_FLAG_CHECKED also a slot >= num_blocks*16 (PKV_ERR_RANGE) or the same
 * slot named twice (PKV_ERR_OVERLAP; checked for num_tokens <= 16384, larger
 * checked calls return PKV_ERR_UNSUPPORTED). In fast mode a repeated slot
 * receives one of the tokens, unspecified which.
 */
PKV_API pkv_status pkv_append(const void* k, const void* v, const int64_t* slot_mapping,
                      int64_t num_tokens, void* k_cache, void* v_cache,
                      const pkv_cache_desc* desc, uint32_t flags, void* stream);

/*
 * pkv_copy_blocks -- whole-block copy for copy-on-write.
 * (notebook section 5: before a sequence appends into a shared partial final
 * block it takes a private replacement; this call moves the data.)
 *
 * For each pair p < num_pairs: block pairs[p][1] of both pools becomes a copy
 * of block pairs[p][0] (all KV heads, all 16 slots, K and V). The copies act
 * as one step: destinations must be distinct and must not also be sources.
 *
 *   src_dst_pairs device, int64 [num_pairs][2] = {src, dst}. Read only.
 *   num_pairs     >= 0; 0 enqueues nothing (a valid no-op).
 * Errors: as pkv_append; with PKV_FLAG_CHECKED a block id outside
 * [0, num_blocks) gives PKV_ERR_RANGE and a repeated destination or a
 * destination that is also a source gives PKV_ERR_OVERLAP (num_pairs <= 16384).
 */
PKV_API pkv_status pkv_copy_blocks(const int64_t* src_dst_pairs, int64_t num_pairs,
                           void* k_cache, void* v_cache,
                           const pkv_cache_desc* desc, uint32_t flags, void* stream);

/*
 * pkv_decode_workspace_size -- bytes of device workspace pkv_decode_attention
 * needs for these sizes and options on the current device.
 *
 * The workspace holds the fp32 pieces of context segments that the kernel
 * splits across CTAs and one counter per (sequence, KV head, warp) that
 * finds the CTA which merges them. Zero-fill it once before its first use
 * (cudaMemset); every completed call leaves the counters at zero again. Use
 * one workspace per in-flight call, and zero it again after a call that set
 * PKV_DEVERR_TIMEOUT.
 */
PKV_API size_t pkv_decode_workspace_size(int32_t batch, int32_t num_q_heads,
                                 int32_t max_blocks_per_seq,
                                 const pkv_cache_desc* desc,
                                 const pkv_decode_opts* opts);

/*
 * pkv_decode_attention -- one decode query per sequence against its paged
 * context, grouped-query heads.
 * (notebook project demo, Demo 2 `attention`: softmax of the scaled logits
 * with the maximum subtracted, times V; notebook section 3: K/V storage scales
 * with the KV heads, the work with the query heads.)
 *
 * For sequence i < batch, query head h < num_q_heads, G = num_q_heads /
 * num_kv_heads, j = h / G, n = context_lens[i]:
 *     s_t = scale * dot(q[i][h], K_j(t)),  t < n
 *     out[i][h] = sum_t softmax(s)_t * V_j(t)
 * where K_j(t) / V_j(t) is row t % 16 of KV head j in block
 * block_tables[i][t / 16]. n == 0 gives a zero row in the default mode (a
 * query with no keys; notebook section 3 notes it does not occur in a real
 * decode, so PKV_FLAG_CHECKED rejects it, below). Accumulation is fp32;
 * out is written once, rounded to nearest-even into desc->dtype. One kernel
 * launch per 1024 sequences.
 *
 *   q             device, [batch][num_q_heads][head_dim], desc->dtype.
 *   block_tables  device, int32 [batch][max_blocks_per_seq]; entries at
 *                 index >= ceil(n/16) are never read.
 *   context_lens  device, int32 [batch], 0 <= n <= max_blocks_per_seq*16
 *                 (1 <= n with PKV_FLAG_CHECKED).
 *   out           device, [batch][num_q_heads][head_dim], desc->dtype.
 *   workspace     device, >= pkv_decode_workspace_size(...) bytes, 256-byte
 *                 aligned, zero-filled before its first use (see above).
 *   opts          NULL or tuning (above).
 * Errors: host-side checks as above plus num_q_heads % num_kv_heads != 0
 * (PKV_ERR_SHAPE) and a short workspace (PKV_ERR_WORKSPACE); with
 * PKV_FLAG_CHECKED a context length outside [1, max_blocks_per_seq*16] or a
 * block id outside [0, num_blocks) among the blocks a sequence uses gives
 * PKV_ERR_RANGE. batch may exceed any internal limit: the call splits it.
 * `opts` is an addition to the pages' argument list (q, caches, tables,
 * lengths, scale, out): kernel choice and CTA count for tests and tuning;
 * NULL keeps the defaults.
 */
PKV_API pkv_status pkv_decode_attention(const void* q, const void* k_cache, const void* v_cache,
                                const int32_t* block_tables, int32_t max_blocks_per_seq,
                                const int32_t* context_lens, int32_t batch,
                                int32_t num_q_heads, float scale, void* out,
                                void* workspace, size_t workspace_bytes,
                                const pkv_cache_desc* desc, uint32_t flags,
                                const pkv_decode_opts* opts, void* stream);

/*
 * pkv_decode_prefixed_workspace_size -- bytes of device workspace
 * pkv_decode_attention_prefixed needs (same zero-fill rule as above: zero it
 * once before first use; completed calls leave their counters at zero).
 * num_groups and max_group_blocks as in that call. Returns 0 for invalid sizes.
 */
PKV_API size_t pkv_decode_prefixed_workspace_size(int32_t batch, int32_t num_q_heads,
                                                  int32_t max_blocks_per_seq, int32_t num_groups,
                                                  int32_t max_group_blocks,
                                                  const pkv_cache_desc* desc,
                                                  const pkv_decode_opts* opts);

/*
 * pkv_decode_attention_prefixed -- pkv_decode_attention for a batch in which
 * groups of sequences share leading blocks, computed in two phases.
 * (paper-search page, ChunkAttention abstract: KV split into chunks that
 * requests with a common prompt prefix share, and a "two-phase partition"
 * kernel that reads a shared chunk once for all of them; notebook section 5
 * `share_prefix`: the target's table begins with the source's first
 * ceil(prefix/B) blocks, and section 7, prefix reuse.)
 *
 * Sequence i is a member of group g = prefix_group[i] when 0 <= g <
 * num_groups, 0 <= group_blocks[g] <= max_group_blocks and its context holds
 * group_blocks[g] whole blocks (16 * group_blocks[g] <= context_lens[i]).
 * The caller guarantees that the first group_blocks[g] entries of every
 * member's block table are the same physical blocks. Phase 1 attends the
 * queries of all members of a group together over those shared blocks (each
 * shared block is read once per 64 query rows: 64 / G members); phase 2
 * attends each sequence over the rest of its context; the two partials are
 * combined by their log-sum-exp weights. A sequence with prefix_group[i] < 0,
 * or one that names a group but fails the membership rule (this also sets
 * PKV_DEVERR_RANGE), is attended in one pass.
 *
 * The result equals pkv_decode_attention's on the same arguments, up to
 * fp32 rounding order: the groups change the work, not the output. A shared
 * partial last block is not shared here: its tokens belong to phase 2.
 *
 *   prefix_group      device, int32 [batch]: group of each sequence, or -1.
 *   group_blocks      device, int32 [num_groups]: shared whole blocks per group.
 *   num_groups        0..1024 (more: PKV_ERR_UNSUPPORTED); 0 = plain call.
 *   max_group_blocks  host-side bound on group_blocks[], <= max_blocks_per_seq;
 *                     sizes the split of the shared blocks over CTAs.
 *   workspace         >= pkv_decode_prefixed_workspace_size(...) bytes,
 *                     256-byte aligned, zero-filled before its first use.
 * Other arguments, results and errors are pkv_decode_attention's. Phase 1
 * runs on the tensor-core path (bf16, head_dim 64/128, G <= 8); elsewhere the
 * groups are ignored and the call is pkv_decode_attention. With
 * PKV_FLAG_CHECKED it also returns PKV_ERR_RANGE, writing nothing, when a
 * sequence names a group but fails the membership rule or its table does not
 * begin with the group's first member's group_blocks[g] entries. Two kernel
 * launches per 1024 sequences.
 */
PKV_API pkv_status pkv_decode_attention_prefixed(const void* q, const void* k_cache, const void* v_cache,
                                                 const int32_t* block_tables, int32_t max_blocks_per_seq,
                                                 const int32_t* context_lens, int32_t batch,
                                                 int32_t num_q_heads, float scale,
                                                 const int32_t* prefix_group, const int32_t* group_blocks,
                                                 int32_t num_groups, int32_t max_group_blocks, void* out,
                                                 void* workspace, size_t workspace_bytes,
                                                 const pkv_cache_desc* desc, uint32_t flags,
                                                 const pkv_decode_opts* opts, void* stream);

/*
 * pkv_multiquery_workspace_size -- bytes of device workspace
 * pkv_multiquery_attention needs (zero-fill once before first use; completed
 * calls leave its counters at zero). Returns 0 for sizes the call rejects.
 */
PKV_API size_t pkv_multiquery_workspace_size(int32_t batch, int32_t num_q_heads, int32_t max_blocks_per_seq,
                                             int32_t max_query_len, const pkv_cache_desc* desc,
                                             const pkv_decode_opts* opts);

/*
 * pkv_multiquery_attention -- several causal queries per sequence against its
 * paged context, in one pass over the cache.
 * (release page, Architectural Breakdown 2: the target model verifies the K
 * draft tokens in a single parallel pass; notebook section 7: a cached-prefix
 * suffix attends to every cached position and causally within itself, and the
 * chunks of a prefill together hold exactly the causal pairs of the prompt.)
 *
 * Sequence i holds n = context_lens[i] tokens, the last nq = query_start[i+1]
 * - query_start[i] of which are this step's new tokens (appended before the
 * call). Query t < nq, at row query_start[i] + t of q and out, attends to
 * tokens 0 .. n - nq + t:
 *     out[r][h] = sum_p softmax_p(scale * dot(q[r][h], K_j(p))) V_j(p),  p <= n - nq + t
 * with K_j / V_j gathered through block_tables[i] as in pkv_decode_attention.
 * One query per sequence is pkv_decode_attention. fp32 accumulation, one
 * rounding to bf16.
 *
 *   q, out        device, bf16 [query_start[batch]][num_q_heads][head_dim].
 *   query_start   device, int32 [batch + 1], non-decreasing row offsets.
 *   max_query_len host bound on nq, 1 <= max_query_len <= 65536 (else
 *                 PKV_ERR_UNSUPPORTED). Up to 32 query rows per (sequence,
 *                 KV head) (max_query_len * num_q_heads / num_kv_heads) run
 *                 on the split decode kernel; more (a chunked prefill) run on
 *                 the 5th-generation tensor cores: 128-row query tiles, the
 *                 context split over a thread-block cluster whose CTAs combine
 *                 their partials on chip (that path uses only 256 bytes of the
 *                 workspace).
 *   workspace     >= pkv_multiquery_workspace_size(...) bytes, 256-byte
 *                 aligned, zero-filled before its first use.
 * Errors: as pkv_decode_attention; bf16 caches only (else PKV_ERR_DTYPE). A
 * sequence whose query count lies outside [0, min(n, max_query_len)] gets no
 * output rows and sets PKV_DEVERR_RANGE; with PKV_FLAG_CHECKED the call
 * returns PKV_ERR_RANGE instead, having written nothing. The split decode
 * kernel reads every K/V byte once for all the queries of its sequence; the
 * prefill path reads a sequence's K/V once per 128-row query tile.
 */
PKV_API pkv_status pkv_multiquery_attention(const void* q, const void* k_cache, const void* v_cache,
                                            const int32_t* block_tables, int32_t max_blocks_per_seq,
                                            const int32_t* context_lens, const int32_t* query_start,
                                            int32_t batch, int32_t num_q_heads, int32_t max_query_len,
                                            float scale, void* out, void* workspace, size_t workspace_bytes,
                                            const pkv_cache_desc* desc, uint32_t flags,
                                            const pkv_decode_opts* opts, void* stream);

/*
 * Low-bit (int8) paged KV.
 * (notebook section 8: fewer bits per coordinate shrink the bytes per token in
 * proportion; notebook project demo `fake_quantize_rows`: per row, limit =
 * 2^(bits-1) - 1, scale = max|x| / limit (1 for a zero row), codes =
 * clip(rint(x / scale), -limit, limit), value = code * scale.)
 *
 * A row is one token of one KV head (head_dim coordinates); bits = 8, limit =
 * 127. The scale is stored as a float32, computed as float32(max|x|) / 127 in
 * float32; each code is rint(x / scale) in float64 (half to even) against that
 * stored scale, clipped to [-127, 127]. The cached row stands for code * scale.
 * Pools (desc->dtype = PKV_INT8, head_dim 64 or 128 for the append, 128 for
 * the attention, block_size 16), caller-allocated, device:
 *   k_codes   int8  [num_blocks][num_kv_heads][16][head_dim]   (token rows)
 *   v_codes   int8  [num_blocks][num_kv_heads][head_dim][16]   (coordinate rows)
 *   scales    float [num_blocks][num_kv_heads][2][16]: one 128-byte record per
 *             (block, KV head), the 16 K-row scales ([..][0][slot]) then the
 *             16 V-row scales ([..][1][slot])
 * 132 bytes per (token, KV head, pool) at head_dim 128, against 256 for bf16.
 * The two scale rows of a (block, head) share one record so that attention
 * reads one whole 128-byte line for them: with a pool per side, each 64-byte
 * row was half of a line that DRAM delivered whole (3.9 % more DRAM traffic
 * than the bytes used, and 3 % more time, on the 8K Llama layer).
 */

/*
 * pkv_append_q8 -- slot-mapped quantizing append: for each token t with
 * s = slot_mapping[t] >= 0 and each KV head h, row (t, h) of k (bf16
 * [num_tokens][num_kv_heads][head_dim]) is quantized into k_codes and its scale at
 * block s/16, slot s%16 (scale in scales[s/16][h][0][s%16]), and the same for v
 * (scales[s/16][h][1][s%16]). Arguments and errors as
 * pkv_append (PKV_FLAG_CHECKED validates the slots first).
 */
PKV_API pkv_status pkv_append_q8(const void* k, const void* v, const int64_t* slot_mapping, int64_t num_tokens,
                                 void* k_codes, void* v_codes, float* scales,
                                 const pkv_cache_desc* desc, uint32_t flags, void* stream);

/*
 * pkv_copy_blocks_q8 -- copy-on-write block copy of the low-bit pools: codes
 * and scales of every pair {src, dst}, with pkv_copy_blocks's rules.
 */
PKV_API pkv_status pkv_copy_blocks_q8(const int64_t* src_dst_pairs, int64_t num_pairs, void* k_codes,
                                      void* v_codes, float* scales,
                                      const pkv_cache_desc* desc, uint32_t flags, void* stream);

/*
 * pkv_decode_q8_workspace_size -- bytes of workspace pkv_decode_attention_q8
 * needs (zero-fill once before first use; completed calls leave its counters at
 * zero). max_query_len as in pkv_multiquery_attention (1 for plain decode).
 */
PKV_API size_t pkv_decode_q8_workspace_size(int32_t batch, int32_t num_q_heads, int32_t max_blocks_per_seq,
                                            int32_t max_query_len, const pkv_cache_desc* desc,
                                            const pkv_decode_opts* opts);

/*
 * pkv_decode_attention_q8 -- decode (or causal multi-query) attention over the
 * low-bit pools: the result pkv_multiquery_attention (query_start non-NULL) or
 * pkv_decode_attention (query_start NULL: one query per sequence, a sequence
 * with no tokens gets a zero row) would give over the values the cached rows
 * stand for (code * scale). q and out are bf16 as in those calls; fp32
 * accumulation, one rounding to bf16. The products run on f16 tensor cores:
 * the codes and q (each row scaled by a power of two) are exact there, the
 * softmax weights times the V scale are rounded to f16. head_dim 128, at most
 * 32 query rows per (sequence, KV head). Errors, checked mode and the device
 * status bits as in pkv_multiquery_attention; query_start NULL with
 * max_query_len != 1 is PKV_ERR_SHAPE.
 */
PKV_API pkv_status pkv_decode_attention_q8(const void* q, const void* k_codes, const void* v_codes,
                                           const float* scales,
                                           const int32_t* block_tables, int32_t max_blocks_per_seq,
                                           const int32_t* context_lens, const int32_t* query_start,
                                           int32_t batch, int32_t num_q_heads, int32_t max_query_len,
                                           float scale, void* out, void* workspace, size_t workspace_bytes,
                                           const pkv_cache_desc* desc, uint32_t flags,
                                           const pkv_decode_opts* opts, void* stream);

/*
 * pkv_decode_attention_noalloc -- pkv_decode_attention without a
 * caller-provided workspace. The pages have no counterpart to this call; it
 * exists for callers that cannot allocate device memory: plugins running
 * inside a framework whose memory pool they do not own, latency-critical
 * paths that cannot take cudaMalloc's implicit synchronisation, deployments
 * with a device-memory budget fixed at start-up.
 *
 * Arguments, results and errors are those of pkv_decode_attention, minus
 * `workspace` / `workspace_bytes`. The workspace is a fixed array of
 * PKV_NOALLOC_SCRATCH_BYTES inside the library, held in device memory by
 * every GPU that loads the library until the process exits. A call whose
 * workspace (pkv_decode_workspace_size) would exceed it returns
 * PKV_ERR_WORKSPACE and writes nothing.
 *
 *  - The call allocates nothing: no cudaMalloc, cudaFree or allocating
 *    library routine. It clears the array's merge counters with one
 *    cudaMemsetAsync on `stream` before the kernel.
 *  - Every call on a device shares the one array: calls that can overlap on
 *    the GPU (different streams without ordering between them) race and give
 *    wrong results. Order them, e.g. issue them on one stream.
 *  - The first call on each device looks up the array's device address (with
 *    that device current) and caches it; make that first call before any
 *    stream capture begins. cudaDeviceReset destroys the array with the
 *    device's context; the first call after it (in the new context) looks the
 *    address up again, so it too belongs before any capture.
 */
#define PKV_NOALLOC_SCRATCH_BYTES (4u * 1024u * 1024u)
PKV_API pkv_status pkv_decode_attention_noalloc(const void* q, const void* k_cache, const void* v_cache,
                                                const int32_t* block_tables, int32_t max_blocks_per_seq,
                                                const int32_t* context_lens, int32_t batch,
                                                int32_t num_q_heads, float scale, void* out,
                                                const pkv_cache_desc* desc, uint32_t flags,
                                                const pkv_decode_opts* opts, void* stream);

/* ------------------------------------------------------------------------
 * Block pool: the host-side page table that decides where tokens go.
 * ("Notebook 10. KV cache and serving: bytes, pages, and ceilings",
 * section 5 "Page pool: prefix sharing and copy-on-write"; release page,
 * Architectural Breakdown 1: physical block allocator, block table,
 * fragment-free growth; Highlights: dynamic block reclamation.)
 *
 * The pool tracks, per physical block, how many sequences reference it, and
 * per sequence its length and block table. It stores no K/V: it produces the
 * slot ids for pkv_append, the copy-on-write pairs for pkv_copy_blocks and the
 * block tables for pkv_decode_attention.
 *  - A fresh pool hands out block ids in `pop_order` (default 0, 1, 2, ...);
 *    freed blocks are reused most-recently-freed first.
 *  - An append first counts the blocks it needs (one private replacement if
 *    the sequence's last block is partial and shared, plus one per 16 new
 *    tokens past the last block's room) and fails with PKV_ERR_OUT_OF_BLOCKS,
 *    leaving the pool unchanged, if too few are free.
 *  - Appending into a shared partial last block first replaces it with a
 *    private block (copy-on-write); the call reports the pair (old, new) the
 *    cache must copy before the new tokens are written.
 *  - share_prefix creates a sequence whose first tokens are another's, by
 *    referencing the source's first ceil(prefix / block_size) blocks.
 *  - release drops a sequence; blocks nobody references return to the pool.
 * Sequence ids are caller-chosen int64 values. A pool is not thread-safe.
 * Host memory only; no CUDA call is made.
 * ---------------------------------------------------------------------- */
typedef struct pkv_pool pkv_pool;

typedef struct {
    int64_t total_blocks;
    int64_t free_blocks;
    int64_t allocated_blocks;          /* referenced by at least one sequence   */
    int64_t physical_capacity_tokens;  /* allocated_blocks * block_size         */
    int64_t physical_payload_tokens;   /* live slots, each block counted once   */
    int64_t logical_tokens;            /* sum of sequence lengths               */
    int64_t internal_waste_tokens;     /* capacity - payload                    */
    int64_t sharing_savings_tokens;    /* logical - payload                     */
    int64_t sequences;
} pkv_pool_stats;

/* total_blocks in [1, 2^31); block_size >= 1 (16 for the kernels); pop_order
 * NULL or a permutation of [0, total_blocks). *out receives the pool. */
PKV_API pkv_status pkv_pool_create(int64_t total_blocks, int32_t block_size, const int64_t* pop_order,
                                   pkv_pool** out);
PKV_API void pkv_pool_destroy(pkv_pool* pool);
/* Register an empty sequence (PKV_ERR_EXISTS if the id is taken). */
PKV_API pkv_status pkv_pool_add_sequence(pkv_pool* pool, int64_t seq);
/* Grow `seq` by `tokens` tokens. slots_out (NULL or `tokens` entries) gets the
 * slot ids of the new tokens; copy_pair_out (NULL or 2 entries) the
 * copy-on-write pair {old, new} when *num_pairs_out is 1. */
PKV_API pkv_status pkv_pool_append(pkv_pool* pool, int64_t seq, int64_t tokens, int64_t* slots_out,
                                   int64_t* copy_pair_out, int32_t* num_pairs_out);
/* One append per listed sequence, in list order (the decode step). slots_out
 * gets sum(tokens) slot ids in list order; pairs_out ([n][2]) the copy-on-write
 * pairs, *num_pairs_out of them. Each append is preflighted on its own: on
 * PKV_ERR_OUT_OF_BLOCKS the first *num_done_out appends have been applied. */
PKV_API pkv_status pkv_pool_append_batch(pkv_pool* pool, const int64_t* seqs, const int64_t* tokens, int64_t n,
                                         int64_t* slots_out, int64_t* pairs_out, int64_t* num_pairs_out,
                                         int64_t* num_done_out);
/* Create `target` sharing the first `prefix_tokens` tokens of `source`. */
PKV_API pkv_status pkv_pool_share_prefix(pkv_pool* pool, int64_t source, int64_t target, int64_t prefix_tokens);
/* Drop `seq`; its unreferenced blocks become free (most recently freed first). */
PKV_API pkv_status pkv_pool_release(pkv_pool* pool, int64_t seq);
PKV_API pkv_status pkv_pool_sequence_length(const pkv_pool* pool, int64_t seq, int64_t* length_out);
/* Block table of `seq`: *num_blocks_out entries are written if they fit in
 * `capacity` (else PKV_ERR_SHAPE and only *num_blocks_out is set). */
PKV_API pkv_status pkv_pool_page_table(const pkv_pool* pool, int64_t seq, int32_t* table_out, int64_t capacity,
                                       int64_t* num_blocks_out);
/* Tables of n sequences as rows of `width` int32 entries padded with -1, and
 * their lengths: the block_tables / context_lens of pkv_decode_attention. */
PKV_API pkv_status pkv_pool_block_tables(const pkv_pool* pool, const int64_t* seqs, int64_t n, int32_t* tables_out,
                                         int64_t width, int32_t* lens_out);
PKV_API pkv_status pkv_pool_get_stats(const pkv_pool* pool, pkv_pool_stats* out);
/* Check every invariant of section 5 (free list, table lengths, reference
 * counts, fills); PKV_ERR_INVARIANT if one is broken. */
PKV_API pkv_status pkv_pool_validate(const pkv_pool* pool);

/*
 * pkv_device_status -- read (and with clear != 0, reset) the sticky device
 * status of the current device: an OR of PKV_DEVERR_* bits set by kernels
 * since the last clear. Waits for `stream`. Returns PKV_OK or PKV_ERR_CUDA.
 *
 * The status is one word per device, shared by every caller, stream and
 * thread of the process that uses the library on that device: a bit set by
 * any call's kernel stays set (no later call clears it, successful or not)
 * until some caller clears it here. A clear therefore also clears bits that
 * other callers' kernels set; a caller that needs its own verdict should
 * read without clearing, or use PKV_FLAG_CHECKED, whose verdict is returned
 * by the call itself. Reading waits only for `stream`: kernels still running
 * on other streams may set bits after the read.
 */
PKV_API pkv_status pkv_device_status(uint32_t* bits_out, int clear, void* stream);

/* Human-readable name of a status code (static string). */
PKV_API const char* pkv_status_string(pkv_status status);

/* ABI version: major * 10000 + minor * 100 + patch. */
PKV_API int32_t pkv_version(void);

#ifdef __cplusplus
}
#endif
#endif /* PKV_H */
