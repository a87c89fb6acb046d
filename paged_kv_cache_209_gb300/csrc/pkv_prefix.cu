// Chunk-first pass of the shared-prefix (two-phase) decode.
//
// A group is a set of sequences whose block tables begin with the same
// group_blocks[p] physical blocks (notebook section 5: share_prefix gives the
// target the source's leading blocks). The decode kernel, in prefixed mode,
// has already attended every member over its own tokens past those blocks
// and left the normalised result with its log2-sum-exp in fold_o / fold_lse.
// The kernels here attend the queries of all members of a group together
// over the shared blocks -- each shared K/V block is read once per tile of
// query rows instead of once per sequence -- and combine the two partials by
// their log-sum-exp weights into the output rows (paper-search page,
// ChunkAttention abstract: "two-phase partition", shared chunks first, then
// each sequence).
//
// Work decomposition (both kernels). The query rows of group p are (member
// m, query head g of KV head h) in member order, row r = m * G + g. CTA
// (x, y, z) takes row tile x of the list of all groups' tiles (each group's
// rows padded to whole tiles), chunk y of the group's shared blocks and KV
// head z. A group whose shared blocks fit in one chunk is finished by its CTA
// directly; otherwise each chunk leaves an fp32 partial (unnormalised O,
// running max m, sum l) per row, and the last of the chunks' warps to finish
// a set of rows (an atomic counter per tile, head and warp) merges them.
//
// prefix_umma_kernel (default): 128-row tiles on the 5th-generation tensor
// cores, one role per warp. Two TMA warps stream 64-token steps (four
// blocks) of K and of V through separate shared-memory rings; two warps
// issue the score products of even and of odd steps,
//     S[128][64]  = Q[128][D] K^T      (tcgen05.mma, fp32 accumulator in tensor
//                                        memory, four S/P buffers)
// and two the products of the two 32-token halves of P,
//     O[128][D]  += P[128][32] V[32][D] (P as bf16 hi + lo written by the softmax
//                                        over its own S columns in tensor memory,
//                                        V read MN-major straight from the TMA
//                                        layout, one O accumulator per half)
// while eight softmax warps, one thread per (query row, token half), load S
// rows from tensor memory, run the online softmax (base 2, lazy rescale of O
// in tensor memory) and store P. The two halves of a row are combined at the
// end.
//
// prefix_mma_kernel: 64-row tiles, four warps of 16 rows each on mma.sync
// (m16n8k16) with the S accumulator fragments reused as the A operand of P;
// kept as a second implementation that the tests compare with.
#include <math.h>
#include <mutex>

#include "pkv_device.cuh"
#include "pkv_internal.h"

namespace pkv {
namespace {

constexpr float kLog2e = 1.4426950408889634f;
constexpr int kMaxChunks = 32;
// Sleep between probes of a wait that runs ahead of need (the score issuers
// waiting for a free S/P buffer, the copy warps for a free stage).
#ifndef PKV_AHEAD_SLEEP_NS
#define PKV_AHEAD_SLEEP_NS 64
#endif
constexpr unsigned int kAheadSleepNs = PKV_AHEAD_SLEEP_NS;
constexpr int kMaxCluster = 8;  // CTAs (chunks) per cluster of the tcgen05 kernel: the portable maximum
constexpr int kMaxGroups = kMaxBatchPerLaunch;

__device__ __forceinline__ float ninf() { return __int_as_float(0xff800000); }


// Build-time tracing (PKV_TRACE): each CTA of the tcgen05 kernel records
// %globaltimer stamps in a row of 16 words: [0] entry, [1] tile located,
// [2] tensor memory and Q ready, [3] softmax loop done, [5] exit of thread 0,
// [7] 1 for a CTA with work; sums over the steps of: [8] softmax wait for S,
// [9] S load from tensor memory, [10] softmax arithmetic (with the P
// stores), [11] softmax waits for PV products (O rescale), [12] wait for the
// P stores and arrival, [13] P.V issuer wait for P, [4] P.V issuer wait for
// V, [14] score issuer wait for K, [6] score issuer wait for its S/P buffer
// (the P.V product four steps back), [15] K copy warp wait for a free stage.
#ifdef PKV_TRACE
// Launches without a workspace slot for the stamps (chunked prefill) write
// them here instead, for the first 65536 CTAs.
__device__ unsigned long long g_px_trace[65536 * 16];
#define PX_CTA() ((blockIdx.z * gridDim.y + blockIdx.y) * gridDim.x + blockIdx.x)
#define PX_STAMP(a, i, v)                                                                    \
    do {                                                                                     \
        if ((a).trace != nullptr)                                                            \
            (reinterpret_cast<unsigned long long*>((a).trace))[PX_CTA() * 16 + (i)] = (v);   \
        else if (PX_CTA() < 65536)                                                           \
            g_px_trace[PX_CTA() * 16 + (i)] = (v);                                           \
    } while (0)
#define PX_T(var) const unsigned long long var = global_ns()
// Per-step stamps of the first CTA (steps < 256), after the per-CTA rows:
// [0] score issue start, [1] score issue end, [2] softmax sees S, [3] softmax
// arrives on P (warp 0, lane 0), [4] P.V issue start, [5] P.V issue end.
#define PX_STEP(j, k)                                                                      \
    do {                                                                                   \
        if (PX_CTA() == 0 && (j) < 256) g_px_trace[65536 * 8 + (j) * 8 + (k)] = global_ns(); \
    } while (0)
#define PX_ADD(acc, v) acc += (v)
#else
#define PX_STAMP(a, i, v) ((void)0)
#define PX_T(var) ((void)0)
#define PX_STEP(j, k) ((void)0)
#define PX_ADD(acc, v) ((void)0)
#endif

// Members of one tile: at most rows / G + 2.
__host__ __device__ constexpr int member_slots(int rows) { return rows + 8; }

// Shared prologue of both kernels (all threads; contains __syncthreads).
// Counts the members of every group, finds the group and tile of this CTA's
// x index and the tile's members in member order, and the chunk of shared
// blocks of this CTA's y index. info[]: [0] group, [1] tile within the group,
// [2] first member of the group, [3] shared blocks, [4] chunks of the group,
// [5] rows of the tile, [6] first member of the tile. Returns (for the whole
// CTA) 0 when x names no tile, 1 when the tile exists but its group has no
// chunk y (info and members are set), 2 when the CTA has work.
//
// `stage` holds 2 * kMaxBatchPerLaunch + kMaxGroups ints: the context lengths
// (clamped to the tables), the group ids and the group block counts, read from
// global memory once, side by side, so that nothing below waits on a chain of
// dependent global loads.
template <int kRowsPerTile>
__device__ int locate_tile(const PrefixArgs& a, int* info, int* members, int* counts, int* stage) {
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int G = a.group;
    const int cap = a.max_blocks * 16;
    int* s_len = stage;
    int* s_grp = stage + kMaxBatchPerLaunch;
    int* s_gb = stage + 2 * kMaxBatchPerLaunch;
    if (threadIdx.x == 0) {
        info[0] = -1;
        info[2] = 0;
    }
    for (int i = threadIdx.x; i < a.batch; i += blockDim.x) {
        const int n = a.lens[i];
        s_len[i] = n < 0 ? 0 : (n > cap ? cap : n);
        s_grp[i] = a.prefix_group[i];
    }
    for (int g = threadIdx.x; g < a.num_groups; g += blockDim.x) {
        counts[g] = 0;
        s_gb[g] = a.group_blocks[g];
    }
    __syncthreads();
    auto member_blocks = [&](int i) {
        return prefix_member_blocks(s_grp, s_gb, a.num_groups, a.max_group_blocks, s_len[i], i);
    };
    for (int i = threadIdx.x; i < a.batch; i += blockDim.x)
        if (member_blocks(i) >= 0) atomicAdd(&counts[s_grp[i]], 1);
    __syncthreads();
    if (warp == 0) {
        // tile x -> (group, tile within the group): prefix sums of the groups' tile counts
        int carry = 0;
        for (int base = 0; base < a.num_groups; base += 32) {
            const int g = base + lane;
            const int t = g < a.num_groups ? (counts[g] * G + kRowsPerTile - 1) / kRowsPerTile : 0;
            int x = t;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int y = __shfl_up_sync(0xffffffffu, x, o);
                if (lane >= o) x += y;
            }
            const int excl = carry + x - t;
            if (t > 0 && static_cast<int>(blockIdx.x) >= excl && static_cast<int>(blockIdx.x) < excl + t) {
                info[0] = g;
                info[1] = static_cast<int>(blockIdx.x) - excl;
            }
            carry += __shfl_sync(0xffffffffu, x, 31);
        }
    }
    __syncthreads();
    const int p = info[0];
    if (p < 0) return 0;
    const int nb = s_gb[p];  // in [0, max_group_blocks]: p has members
    const int nch = nb > 0 ? (nb + a.chunk_blocks - 1) / a.chunk_blocks : 1;
    const int r0 = info[1] * kRowsPerTile;
    const int nrows = min(kRowsPerTile, counts[p] * G - r0);
    const int m0 = r0 / G;
    const int m1 = (r0 + nrows - 1) / G + 1;
    if (warp == 0) {
        int rank = 0;
        for (int base = 0; base < a.batch; base += 32) {
            const int i = base + lane;
            const bool is = i < a.batch && s_grp[i] == p && member_blocks(i) >= 0;
            const unsigned int bal = __ballot_sync(0xffffffffu, is);
            const int r = rank + __popc(bal & ((1u << lane) - 1u));
            if (is) {
                if (r == 0) info[2] = i;
                if (r >= m0 && r < m1) members[r - m0] = i;
            }
            rank += __popc(bal);
        }
        if (lane == 0) {
            info[3] = nb;
            info[4] = nch;
            info[5] = nrows;
            info[6] = m0;
        }
    }
    __syncthreads();
    return static_cast<int>(blockIdx.y) < nch ? 2 : 1;
}

// Prologue of the causal multi-query (chunked prefill) mode (all threads;
// contains __syncthreads). The query rows of sequence i are (query t, query
// head g of KV head h), row r = t G + g, in 128-row tiles; query t of a
// sequence with n tokens and nq queries sees tokens 0 .. n - nq + t. Finds
// the sequence and tile of this CTA's x index. info[]: [1] tile within the
// sequence, [2] sequence, [3] blocks the tile's last row sees, [4] chunks of
// them, [5] rows of the tile, [7] n, [8] nq, [9] first query row of the
// sequence. Returns 0 when x names no tile, 1 when the tile has no chunk y,
// 2 when the CTA has work. A sequence whose query range is malformed
// (negative, more queries than tokens or than max_query_len) gets no tiles
// and sets PKV_DEVERR_RANGE.
template <int kRowsPerTile>
__device__ int locate_prefill_tile(const PrefixArgs& a, int* info, int* stage) {
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int G = a.group;
    const int cap = a.max_blocks * 16;
    int* s_tiles = stage;  // tiles of each sequence
    if (threadIdx.x == 0) info[0] = -1;
    for (int i = threadIdx.x; i < a.batch; i += blockDim.x) {
        const int n = a.lens[i];
        const int q0 = a.qstart[i];
        const int nq = a.qstart[i + 1] - q0;
        const bool bad = n < 0 || n > cap || q0 < 0 || nq < 0 || nq > n || nq > a.max_query_len;
        if (bad && blockIdx.x == 0 && blockIdx.y == 0 && blockIdx.z == 0) atomicOr(a.status, PKV_DEVERR_RANGE);
        s_tiles[i] = bad ? 0 : (nq * G + kRowsPerTile - 1) / kRowsPerTile;
    }
    __syncthreads();
    if (warp == 0) {
        int carry = 0;
        for (int base = 0; base < a.batch; base += 32) {
            const int i = base + lane;
            const int t = i < a.batch ? s_tiles[i] : 0;
            int x = t;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int y = __shfl_up_sync(0xffffffffu, x, o);
                if (lane >= o) x += y;
            }
            const int excl = carry + x - t;
            if (t > 0 && static_cast<int>(blockIdx.x) >= excl && static_cast<int>(blockIdx.x) < excl + t) {
                info[0] = i;
                info[1] = static_cast<int>(blockIdx.x) - excl;
            }
            carry += __shfl_sync(0xffffffffu, x, 31);
        }
    }
    __syncthreads();
    const int i = info[0];
    if (i < 0) return 0;
    if (threadIdx.x == 0) {
        const int n = a.lens[i];
        const int q0 = a.qstart[i];
        const int nq = a.qstart[i + 1] - q0;
        const int r0 = info[1] * kRowsPerTile;
        const int nrows = min(kRowsPerTile, nq * G - r0);
        const int seen = n - nq + (r0 + nrows - 1) / G + 1;  // tokens the tile's last row sees, >= 1
        const int nb = (seen + 15) / 16;
        info[2] = i;
        info[3] = nb;
        info[4] = (nb + a.chunk_blocks - 1) / a.chunk_blocks;
        info[5] = nrows;
        info[6] = 0;
        info[7] = n;
        info[8] = nq;
        info[9] = q0;
    }
    __syncthreads();
    return static_cast<int>(blockIdx.y) < info[4] ? 2 : 1;
}

// A CTA without work leaves at once, except CTA (0, 0, 0), which first waits
// for the kernel before it: this grid must not complete (and release the next
// kernel in the stream) before that one has.
__device__ __forceinline__ void idle_exit() {
    if (blockIdx.x == 0 && blockIdx.y == 0 && blockIdx.z == 0) grid_dependency_wait();
}

template <int D, int NST>
struct Px {
    static constexpr int kRows = 64;  // query rows per tile
    static constexpr int kStages = NST;
    static constexpr int kConsumers = 4;
    static constexpr int kThreads = (kConsumers + 1) * 32;
    static constexpr int kHalves = D / 64;
    static constexpr int kPoolBytes = 16 * D * 2;
    static constexpr int kStageBytes = 2 * kPoolBytes;  // K then V
    // shared memory (offsets from a 1024-byte aligned base): the ring,
    // full[NST] and empty[NST], stage flags and the abort flag, then
    // info[8], the tile's members and the per-group member counts.
    static constexpr int kOffBars = kStages * kStageBytes;
    static constexpr int kOffFlags = kOffBars + 2 * kStages * 8;
    static constexpr int kOffInts = kOffFlags + (kStages + 1) * 4;
    static constexpr size_t kSmem =
        1024 + kOffInts + (8 + member_slots(kRows) + kMaxGroups + 2 * kMaxBatchPerLaunch + kMaxGroups) * 4;
};

template <int D, int NST>
__global__ void __launch_bounds__(Px<D, NST>::kThreads)
    prefix_mma_kernel(const PrefixArgs a, const __grid_constant__ CUtensorMap tmK,
                      const __grid_constant__ CUtensorMap tmV) {
    using C = Px<D, NST>;
    constexpr int kTileRows = C::kRows;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::kOffBars);
    uint64_t* empty = full + C::kStages;
    int* stage_ok = reinterpret_cast<int*>(smem + C::kOffFlags);
    volatile int* abort_flag = stage_ok + C::kStages;
    int* info = reinterpret_cast<int*>(smem + C::kOffInts);
    int* members = info + 8;
    int* counts = members + member_slots(kTileRows);
    int* stage = counts + kMaxGroups;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int G = a.group;
    const int h = blockIdx.z;
    const int chunk = blockIdx.y;

    if (threadIdx.x == 0) {
        for (int s = 0; s < C::kStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], C::kConsumers);
        }
        *abort_flag = 0;
        fence_barrier_init();
    }
    if (threadIdx.x == 32) {
        tma_prefetch_desc(&tmK);
        tma_prefetch_desc(&tmV);
    }
    // Inputs only until the fold: the kernel before this one (the decode
    // kernel) lets it start once all its CTAs have passed their own wait on
    // the kernels before them, so the K/V blocks are complete.
    allow_dependents();
    if (locate_tile<kTileRows>(a, info, members, counts, stage) != 2) {
        idle_exit();
        return;
    }
    const int nb = info[3];
    const int nch = info[4];
    const int nrows = info[5];
    const int m0 = info[6];
    const int r0 = info[1] * kTileRows;
    const int blk0 = chunk * a.chunk_blocks;
    const int nblk = nb > 0 ? min(a.chunk_blocks, nb - blk0) : 0;

    if (warp == C::kConsumers) {
        // ------------------------------------------------ producer warp
        const uint64_t policy = l2_evict_last_policy();
        const int32_t* trow = a.tables + static_cast<long long>(info[2]) * a.max_blocks + blk0;
        bool ok = true;
        int k = 0;
        for (int b0 = 0; ok && b0 < nblk; b0 += 32) {
            const int ids = b0 + lane < nblk ? __ldg(trow + b0 + lane) : 0;
            const int cnt = min(32, nblk - b0);
            for (int e = 0; e < cnt; ++e, ++k) {
                const int bid = __shfl_sync(0xffffffffu, ids, e);
                int good = 1;
                if (lane == 0) {
                    const int s = k % C::kStages;
                    const uint32_t par = static_cast<uint32_t>((k / C::kStages) & 1) ^ 1u;
                    if (!mbar_wait(&empty[s], par, a.status, abort_flag)) {
                        good = 0;
                    } else if (bid >= 0 && bid < a.num_blocks) {
                        stage_ok[s] = 1;
                        mbar_arrive_expect_tx(&full[s], C::kStageBytes);
                        uint8_t* st = smem + s * C::kStageBytes;
                        const int y = (bid * a.kv_heads + h) * 16;
#pragma unroll
                        for (int hf = 0; hf < C::kHalves; ++hf)
                            tma_load_2d(st + hf * 2048, &tmK, hf * 64, y, &full[s], policy);
#pragma unroll
                        for (int hf = 0; hf < C::kHalves; ++hf)
                            tma_load_2d(st + C::kPoolBytes + hf * 2048, &tmV, hf * 64, y, &full[s], policy);
                    } else {
                        stage_ok[s] = 0;
                        atomicOr(a.status, PKV_DEVERR_RANGE);
                        mbar_arrive(&full[s]);
                    }
                }
                good = __shfl_sync(0xffffffffu, good, 0);
                if (!good) {
                    ok = false;
                    break;
                }
            }
        }
        if (!ok && lane == 0) {  // after an abort: wait (bounded) for the copies still in flight
            const int first = k > C::kStages ? k - C::kStages : 0;
            for (int u = first; u < k; ++u)
                mbar_wait(&full[u % C::kStages], static_cast<uint32_t>((u / C::kStages) & 1), a.status, nullptr);
        }
        grid_dependency_wait();
        return;
    }

    // ---------------------------------------------------- consumer warps
    const int gid = lane >> 2;  // fragment row group
    const int tig = lane & 3;   // thread in group
    const int q8 = lane >> 3, r8 = lane & 7;
    const int k_row = r8 + 8 * (q8 & 1);   // K: token row of this lane's ldmatrix address
    const int k_chunk = q8 >> 1;           // K: +0 / +1 16-byte chunk within a k-step
    const int v_row = r8 + 8 * (q8 >> 1);  // V: token row
    const int v_chunk = q8 & 1;            // V: +0 / +1 chunk within a 16-column step
    const int rw = warp * 16;              // first tile row of this warp
    const bool live = rw < nrows;
    const float scale_log2 = a.scale * kLog2e;

    // The warp's rows gid and gid + 8: output row index (sequence * q_heads +
    // query head) and whether the row exists.
    long long row_idx[2];
    bool row_ok[2];
#pragma unroll
    for (int hr = 0; hr < 2; ++hr) {
        const int r = rw + gid + 8 * hr;
        row_ok[hr] = r < nrows;
        const int R = r0 + (row_ok[hr] ? r : 0);
        const int m = R / G;
        row_idx[hr] = static_cast<long long>(members[m - m0]) * a.q_heads + h * G + (R - m * G);
    }
    // Q as the A operand: [k-step][a0..a3] = (row gid, cols 2tig..+1), (gid+8, ..),
    // (gid, cols 2tig+8..+9), (gid+8, ..)
    uint32_t qa[D / 16][4];
    {
        const uint32_t* qa0 = reinterpret_cast<const uint32_t*>(static_cast<const __nv_bfloat16*>(a.q) + row_idx[0] * D);
        const uint32_t* qa1 = reinterpret_cast<const uint32_t*>(static_cast<const __nv_bfloat16*>(a.q) + row_idx[1] * D);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
            qa[kk][0] = row_ok[0] ? __ldg(qa0 + 8 * kk + tig) : 0u;
            qa[kk][1] = row_ok[1] ? __ldg(qa1 + 8 * kk + tig) : 0u;
            qa[kk][2] = row_ok[0] ? __ldg(qa0 + 8 * kk + 4 + tig) : 0u;
            qa[kk][3] = row_ok[1] ? __ldg(qa1 + 8 * kk + 4 + tig) : 0u;
        }
    }
    float o[D / 8][4];
#pragma unroll
    for (int i = 0; i < D / 8; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
    float ma = ninf(), mb = ninf(), la = 0.f, lb = 0.f;  // rows gid / gid + 8

    for (int k = 0; k < nblk; ++k) {
        const int s = k % C::kStages;
        if (!mbar_wait(&full[s], static_cast<uint32_t>((k / C::kStages) & 1), a.status, abort_flag)) {
            grid_dependency_wait();
            return;
        }
        if (stage_ok[s] && live) {
            const uint32_t kbase = smem_u32(smem + s * C::kStageBytes);
            const uint32_t vbase = kbase + C::kPoolBytes;
            // ---- S = Q K^T: n-tile 0 (tokens 0-7) and 1 (8-15), even and odd k-steps apart
            float s0[4] = {0.f, 0.f, 0.f, 0.f}, s1[4] = {0.f, 0.f, 0.f, 0.f};
            float t0[4] = {0.f, 0.f, 0.f, 0.f}, t1[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
                const int gc = 2 * kk + k_chunk;
                const uint32_t addr = kbase + (gc >> 3) * 2048 + k_row * 128 + (((gc & 7) ^ r8) << 4);
                uint32_t b00, b10, b01, b11;  // [n-tile][B register]
                ldmatrix_x4(addr, b00, b10, b01, b11);
                if (kk & 1) {
                    mma_bf16_16816(t0, qa[kk][0], qa[kk][1], qa[kk][2], qa[kk][3], b00, b01);
                    mma_bf16_16816(t1, qa[kk][0], qa[kk][1], qa[kk][2], qa[kk][3], b10, b11);
                } else {
                    mma_bf16_16816(s0, qa[kk][0], qa[kk][1], qa[kk][2], qa[kk][3], b00, b01);
                    mma_bf16_16816(s1, qa[kk][0], qa[kk][1], qa[kk][2], qa[kk][3], b10, b11);
                }
            }
            // row gid: tokens 2tig, 2tig+1, 8+2tig, 9+2tig; row gid+8 the same
            float xa[4] = {(s0[0] + t0[0]) * scale_log2, (s0[1] + t0[1]) * scale_log2,
                           (s1[0] + t1[0]) * scale_log2, (s1[1] + t1[1]) * scale_log2};
            float xb[4] = {(s0[2] + t0[2]) * scale_log2, (s0[3] + t0[3]) * scale_log2,
                           (s1[2] + t1[2]) * scale_log2, (s1[3] + t1[3]) * scale_log2};
            // lazy rescale, as in the decode kernel: only when a score exceeds
            // the running maximum by more than 8 (a factor 256)
            float mxa = fmaxf(fmaxf(xa[0], xa[1]), fmaxf(xa[2], xa[3]));
            float mxb = fmaxf(fmaxf(xb[0], xb[1]), fmaxf(xb[2], xb[3]));
            if (__any_sync(0xffffffffu, mxa > ma + 8.f || mxb > mb + 8.f)) {
#pragma unroll
                for (int off = 1; off < 4; off <<= 1) {
                    mxa = fmaxf(mxa, __shfl_xor_sync(0xffffffffu, mxa, off));
                    mxb = fmaxf(mxb, __shfl_xor_sync(0xffffffffu, mxb, off));
                }
                const float na = fmaxf(ma, mxa), nbm = fmaxf(mb, mxb);
                const float ala = ma == ninf() ? 0.f : ex2(ma - na);
                const float alb = mb == ninf() ? 0.f : ex2(mb - nbm);
                la *= ala;
                lb *= alb;
#pragma unroll
                for (int i = 0; i < D / 8; ++i) {
                    o[i][0] *= ala;
                    o[i][1] *= ala;
                    o[i][2] *= alb;
                    o[i][3] *= alb;
                }
                ma = na;
                mb = nbm;
            }
            float pa[4], pb[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                pa[j] = ex2(xa[j] - ma);
                pb[j] = ex2(xb[j] - mb);
            }
            la += (pa[0] + pa[1]) + (pa[2] + pa[3]);
            lb += (pb[0] + pb[1]) + (pb[2] + pb[3]);
            // ---- P as the A operand (hi + lo): (gid, tok 2tig..), (gid+8, ..), (gid, tok 8+2tig..), (gid+8, ..)
            const uint32_t h0 = pack_bf16x2(pa[0], pa[1]), h1 = pack_bf16x2(pb[0], pb[1]);
            const uint32_t h2 = pack_bf16x2(pa[2], pa[3]), h3 = pack_bf16x2(pb[2], pb[3]);
            const uint32_t l0 = pack_bf16x2(pa[0] - bf16lo_to_f32(h0), pa[1] - bf16hi_to_f32(h0));
            const uint32_t l1 = pack_bf16x2(pb[0] - bf16lo_to_f32(h1), pb[1] - bf16hi_to_f32(h1));
            const uint32_t l2 = pack_bf16x2(pa[2] - bf16lo_to_f32(h2), pa[3] - bf16hi_to_f32(h2));
            const uint32_t l3 = pack_bf16x2(pb[2] - bf16lo_to_f32(h3), pb[3] - bf16hi_to_f32(h3));
            // ---- O += P V: V^T fragments by transposed ldmatrix
#pragma unroll
            for (int i = 0; i < D / 16; ++i) {
                const int gc = 2 * i + v_chunk;
                const uint32_t addr = vbase + (gc >> 3) * 2048 + v_row * 128 + (((gc & 7) ^ r8) << 4);
                uint32_t v0, v1, v2, v3;  // (tok 0-7, cols 16i..), (0-7, 16i+8..), (8-15, 16i..), (8-15, 16i+8..)
                ldmatrix_x4_trans(addr, v0, v1, v2, v3);
                mma_bf16_16816(o[2 * i], h0, h1, h2, h3, v0, v2);
                mma_bf16_16816(o[2 * i], l0, l1, l2, l3, v0, v2);
                mma_bf16_16816(o[2 * i + 1], h0, h1, h2, h3, v1, v3);
                mma_bf16_16816(o[2 * i + 1], l0, l1, l2, l3, v1, v3);
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[s]);
    }
    if (!live) {
        grid_dependency_wait();
        return;
    }
#pragma unroll
    for (int off = 1; off < 4; off <<= 1) {
        la += __shfl_xor_sync(0xffffffffu, la, off);
        lb += __shfl_xor_sync(0xffffffffu, lb, off);
    }

    const long long tile_head = static_cast<long long>(h) * gridDim.x + blockIdx.x;
    const int ra = rw + gid, rb = ra + 8;
    if (nch > 1) {
        // ---- publish this chunk's partial of the warp's rows; the last warp merges
        constexpr int kSlot = kTileRows * (D + 2);
        float* slot = a.partials + (tile_head * a.chunks + chunk) * kSlot;
#pragma unroll
        for (int i = 0; i < D / 8; ++i) {
            const int d = 8 * i + 2 * tig;
            __stcg(reinterpret_cast<float2*>(slot + ra * D + d), make_float2(o[i][0], o[i][1]));
            __stcg(reinterpret_cast<float2*>(slot + rb * D + d), make_float2(o[i][2], o[i][3]));
        }
        if (tig == 0) {
            __stcg(slot + kTileRows * D + ra, ma);
            __stcg(slot + kTileRows * D + rb, mb);
            __stcg(slot + kTileRows * D + kTileRows + ra, la);
            __stcg(slot + kTileRows * D + kTileRows + rb, lb);
        }
        __threadfence();
        __syncwarp();
        int* counter = a.counters + tile_head * 4 + warp;
        int old = 0;
        if (lane == 0) old = atomicAdd(counter, 1);
        old = __shfl_sync(0xffffffffu, old, 0);
        if (old != nch - 1) {
            grid_dependency_wait();
            return;
        }
        __threadfence();
        for (int c = 0; c < nch; ++c) {
            if (c == chunk) continue;
            const float* sl = a.partials + (tile_head * a.chunks + c) * kSlot;
            const float mca = __ldcg(sl + kTileRows * D + ra), mcb = __ldcg(sl + kTileRows * D + rb);
            const float lca = __ldcg(sl + kTileRows * D + kTileRows + ra);
            const float lcb = __ldcg(sl + kTileRows * D + kTileRows + rb);
            const float na = fmaxf(ma, mca), nbm = fmaxf(mb, mcb);
            const float ba = na == ninf() ? 0.f : na, bb = nbm == ninf() ? 0.f : nbm;
            const float sa = ma == ninf() ? 0.f : ex2(ma - ba), sb = mb == ninf() ? 0.f : ex2(mb - bb);
            const float wa = mca == ninf() ? 0.f : ex2(mca - ba), wb = mcb == ninf() ? 0.f : ex2(mcb - bb);
            la = la * sa + lca * wa;
            lb = lb * sb + lcb * wb;
#pragma unroll
            for (int i = 0; i < D / 8; ++i) {
                const int d = 8 * i + 2 * tig;
                const float2 ca = __ldcg(reinterpret_cast<const float2*>(sl + ra * D + d));
                const float2 cb = __ldcg(reinterpret_cast<const float2*>(sl + rb * D + d));
                o[i][0] = o[i][0] * sa + ca.x * wa;
                o[i][1] = o[i][1] * sa + ca.y * wa;
                o[i][2] = o[i][2] * sb + cb.x * wb;
                o[i][3] = o[i][3] * sb + cb.y * wb;
            }
            ma = na;
            mb = nbm;
        }
        if (lane == 0) *counter = 0;  // ready for the next call
    }

    // ---- fold in each member's own-token partial and write the output rows
    grid_dependency_wait();  // fold_o / fold_lse come from the decode kernel
#pragma unroll
    for (int hr = 0; hr < 2; ++hr) {
        if (!row_ok[hr]) continue;
        const float m = hr ? mb : ma;
        const float l = hr ? lb : la;
        const float ls = __ldcg(a.fold_lse + row_idx[hr]);
        const float mp = l > 0.f ? m : ninf();
        const float M = fmaxf(mp, ls);
        float wp = 0.f, ws = 0.f;
        if (M != ninf()) {
            wp = mp == ninf() ? 0.f : ex2(mp - M);
            ws = ls == ninf() ? 0.f : ex2(ls - M);
        }
        const float den = l * wp + ws;
        const float inv = den > 0.f ? 1.f / den : 0.f;
        wp *= inv;
        ws *= inv;
        const float* fo = a.fold_o + row_idx[hr] * D;
        uint32_t* out = reinterpret_cast<uint32_t*>(static_cast<__nv_bfloat16*>(a.out) + row_idx[hr] * D);
#pragma unroll
        for (int i = 0; i < D / 8; ++i) {
            const int d = 8 * i + 2 * tig;
            const float2 f = __ldcg(reinterpret_cast<const float2*>(fo + d));
            out[d / 2] = pack_bf16x2(o[i][2 * hr] * wp + f.x * ws, o[i][2 * hr + 1] * wp + f.y * ws);
        }
    }
}

// ------------------------------------------------------------------ tcgen05 kernel
template <int D>
struct Ux {
    static constexpr int kRows = 128;                // M: query rows per tile = tensor-memory lanes
    static constexpr int kTok = 64;                  // N of S = Q K^T: tokens per step
    static constexpr int kBlk = kTok / 16;           // blocks per step
    static constexpr int kHalves = D / 64;           // 64-column (128-byte) halves of a row
    // Ring depths (a K stage is released by its score product, a V stage by
    // its P.V product). Six K stages measured slower than four on the
    // chunked-prefill workload: the loads come mostly from L2, and more of
    // them in flight did not arrive sooner.
    static constexpr int kKStages = D == 128 ? 4 : 6;
    static constexpr int kVStages = D == 128 ? 4 : 6;
    static constexpr int kHalfBytes = kTok * 128;    // one half of the 64 token rows of a step
    static constexpr int kKBytes = kHalves * kHalfBytes;  // one stage of K (or of V)
    static constexpr int kQBytes = kHalves * kRows * 128;
    // Shared memory (offsets from a 1024-byte aligned base; every operand
    // tile starts on a 1024-byte boundary, as the 128-byte swizzle wants):
    // Q [halves][128 rows][128 B]; the K ring, then the V ring, each stage
    // [halves][64 token rows][128 B] (the TMA layout of four 16-row boxes);
    // the exchange of the two token halves' row states; the mbarriers; then
    // info[16], the tile's members, the per-group member counts and the
    // staged lookup inputs.
    static constexpr int kOffQ = 0;
    static constexpr int kOffK = kOffQ + kQBytes;
    static constexpr int kOffV = kOffK + kKStages * kKBytes;
    static constexpr int kRingBytes = (kKStages + kVStages) * kKBytes;
    static constexpr int kOffX = kOffK + kRingBytes;
    static constexpr int kOffBars = kOffX + 3 * kRows * 4;
    // k_full, k_empty (per K stage), v_full, v_empty (per V stage), s_full, p_full (two token halves),
    // o_done (per S/P buffer), final (two P.V issuers, two score issuers)
    static constexpr int kNumBufs = 4;  // S/P buffers in tensor memory
    static constexpr int kNumBars = 2 * (kKStages + kVStages) + 4 * kNumBufs + 4;
    static constexpr int kOffInts = kOffBars + kNumBars * 8;
    static constexpr size_t kSmem =
        1024 + kOffInts + (16 + member_slots(kRows) + kMaxGroups + 2 * kMaxBatchPerLaunch + kMaxGroups) * 4;
    // warps 0-7 softmax: warp w takes rows 32 (w % 4) .. + 31 (its tensor-memory
    // lanes) and token half w / 4 of every step; warps 8 and 11 copy K and V
    // (separate rings: a K stage is free once its score product is done, long
    // before the V stage of the same step); warps 9 and 12 issue the P.V
    // products of token halves 0 and 1, warps 10 and 13 the score products of
    // even and odd steps. A wait that follows tensor-core issues in the same
    // thread returns only once the tensor pipe has drained, so each issuing
    // thread's waits leave a gap in its stream; with four issuers the others
    // fill it.
    static constexpr int kSoftmaxWarps = 8;
    static constexpr int kTmaWarp = 8;
    static constexpr int kMmaWarp = 9;     // P.V, token half 0 (and the tensor-memory allocation)
    static constexpr int kSWarp = 10;      // scores, even steps
    static constexpr int kTmaVWarp = 11;
    static constexpr int kMmaWarp1 = 12;   // P.V, token half 1
    static constexpr int kSWarp1 = 13;     // scores, odd steps
    static constexpr int kThreads = 448;
    // S/P buffers b < kNumBufs at columns 64 b: S_j (fp32, 64 tokens) in buffer
    // j % kNumBufs, then P_j written over it (each softmax thread overwrites
    // only the 32 columns of its own token half once it has read them: bf16
    // pairs, hi in the first 16 columns, lo in the next 16). Then O.
    static constexpr uint32_t kColS = 0;
    static constexpr uint32_t kColO = kNumBufs * kTok;  // O of token half 0: [kColO, kColO + D); half 1: next D
    static constexpr uint32_t kTmemCols = 512;
    static_assert(kColO + 2 * D <= kTmemCols, "tensor-memory columns");
};

// PF (chunked prefill): the queries of one sequence over its own context
// with a causal limit per row, written straight to the output (no fold).
template <int D, bool PF>
__global__ void __launch_bounds__(Ux<D>::kThreads, 1)
    prefix_umma_kernel(const PrefixArgs a, const __grid_constant__ CUtensorMap tmK,
                       const __grid_constant__ CUtensorMap tmV) {
    using C = Ux<D>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* k_full = reinterpret_cast<uint64_t*>(smem + C::kOffBars);
    uint64_t* k_empty = k_full + C::kKStages;
    uint64_t* v_full = k_empty + C::kKStages;
    uint64_t* v_empty = v_full + C::kVStages;
    uint64_t* s_full = v_empty + C::kVStages;       // [buffers]: buffer b holds a finished S
    uint64_t* p_full = s_full + C::kNumBufs;        // [2][buffers]: token half t of P written over it
                                                    // (one arrival per softmax warp of the half)
    uint64_t* o_done = p_full + 2 * C::kNumBufs;    // [buffers]: both P.V products reading it have completed
    uint64_t* final_bar = o_done + C::kNumBufs;     // [2]: every P.V product of an issuer has completed
    uint64_t* final_s = final_bar + 2;              // [2]: every score product of an issuer has completed
    int* info = reinterpret_cast<int*>(smem + C::kOffInts);
    int* members = info + 16;
    int* counts = members + member_slots(C::kRows);
    int* stage = counts + kMaxGroups;
    volatile int* abort_flag = info + 14;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(info + 15);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int G = a.group;
    const int h = blockIdx.z;
    const int chunk = blockIdx.y;

    if (threadIdx.x == 0) {
        PX_STAMP(a, 0, global_ns());
        PX_STAMP(a, 7, 0);
        for (int s = 0; s < C::kKStages; ++s) {
            mbar_init(&k_full[s], 1);
            mbar_init(&k_empty[s], 1);
        }
        for (int s = 0; s < C::kVStages; ++s) {
            mbar_init(&v_full[s], 1);
            mbar_init(&v_empty[s], 2);  // released by both P.V issuers
        }
        for (int b = 0; b < C::kNumBufs; ++b) {
            mbar_init(&s_full[b], 1);
            mbar_init(&p_full[b], C::kSoftmaxWarps / 2);
            mbar_init(&p_full[C::kNumBufs + b], C::kSoftmaxWarps / 2);
            mbar_init(&o_done[b], 2);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&final_bar[i], 1);
            mbar_init(&final_s[i], 1);
        }
        *abort_flag = 0;
        fence_barrier_init();
    }
    if (threadIdx.x == 32 * C::kTmaWarp) {
        tma_prefetch_desc(&tmK);
        tma_prefetch_desc(&tmV);
    }
    allow_dependents();  // inputs only until the fold (see the mma.sync kernel)
    // chunked prefill reads the K/V rows the append before it wrote
    if constexpr (PF) grid_dependency_wait();
    const int where = PF ? locate_prefill_tile<C::kRows>(a, info, stage)
                         : locate_tile<C::kRows>(a, info, members, counts, stage);
    if (where == 0) {  // no tile: the same for every CTA of the cluster
        idle_exit();
        return;
    }
    // From here every thread of the CTA reaches the final __syncthreads (so
    // the tensor memory allocated below is always freed) and both cluster
    // barriers. A CTA whose group has no chunk y streams nothing and only
    // takes its share of the combine.
    const int nb = info[3];
    const int nrows = info[5];
    const int m0 = info[6];
    const int r0 = info[1] * C::kRows;
    const int blk0 = chunk * a.chunk_blocks;
    const int nblk = (where == 2 && nb > 0) ? min(a.chunk_blocks, nb - blk0) : 0;
    const int nsteps = (nblk + C::kBlk - 1) / C::kBlk;
    if (threadIdx.x == 0) {
        PX_STAMP(a, 1, global_ns());
        PX_STAMP(a, 7, 1);
    }

    if (warp == C::kMmaWarp) {
        tmem_alloc(tmem_slot, C::kTmemCols);
        tmem_relinquish();
    }
    // Q rows into shared memory (K-major, 128-byte swizzle); thread r < 128
    // loads row r. The TMA warps do not wait for this: they start streaming
    // K and V at once.
    long long row_idx = 0;
    bool row_ok = false;
    if (warp < 4) {
        const int r = threadIdx.x;
        row_ok = r < nrows;
        const int R = r0 + (row_ok ? r : 0);
        if constexpr (PF) {
            const int t = R / G;
            row_idx = static_cast<long long>(info[9] + t) * a.q_heads + h * G + (R - t * G);
        } else {
            const int m = R / G;
            row_idx = static_cast<long long>(members[m - m0]) * a.q_heads + h * G + (R - m * G);
        }
        const uint4* src = reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(a.q) + row_idx * D);
        uint8_t* qs = smem + C::kOffQ;
#pragma unroll
        for (int c = 0; c < D / 8; ++c) {
            const uint4 v = row_ok ? __ldg(src + c) : make_uint4(0u, 0u, 0u, 0u);
            *reinterpret_cast<uint4*>(qs + (c >> 3) * (C::kRows * 128) + r * 128 + (((c & 7) ^ (r & 7)) << 4)) = v;
        }
        fence_proxy_async_smem();
    }
    uint32_t tmem = 0;
    if (warp != C::kTmaWarp && warp != C::kTmaVWarp) {
        tc_fence_before();
        named_barrier_sync(2, C::kThreads - 64);  // every warp but the two TMA warps
        tc_fence_after();
        tmem = *tmem_slot;
    }
    if (threadIdx.x == 0) PX_STAMP(a, 2, global_ns());

    if (warp == C::kTmaWarp || warp == C::kTmaVWarp) {
        // ------------------------------------------------ TMA producers (K, V)
        // Step j: blocks 4j .. 4j+3 of the chunk, each in kHalves 64-column
        // boxes. A TMA instruction costs the issuing warp a few hundred cycles
        // almost whatever the number of lanes issuing it, so the copies go in
        // batches: lane group u (lanes 8u .. 8u + 7) takes step j + u, one box
        // per lane (block lane & 3, half (lane >> 2) & 1), for the run of free
        // stages from stage j on (at most 4, within one batch of table
        // entries); only when stage j itself is busy does the warp wait
        // (bounded) for it. A block past the chunk or with an invalid id is
        // loaded from row -16 (wholly out of range), which fills its box with
        // zeros.
        const bool is_k = warp == C::kTmaWarp;
        uint64_t* full = is_k ? k_full : v_full;
        uint64_t* empty = is_k ? k_empty : v_empty;
        const CUtensorMap* map = is_k ? &tmK : &tmV;
        const int nst = is_k ? C::kKStages : C::kVStages;
        uint8_t* ring = smem + (is_k ? C::kOffK : C::kOffV);
        const uint64_t policy = l2_evict_last_policy();
        const int32_t* trow = a.tables + static_cast<long long>(info[2]) * a.max_blocks + blk0;
        bool ok = true;
        int issued = 0;
#ifdef PKV_TRACE
        unsigned long long tr_tma = 0;
#endif
        // block-table entries, 32 (8 steps) at a time, the next 32 already in
        // flight: lane i holds entry 32 c + i of the current batch c
        int cur = lane < nblk ? __ldg(trow + lane) : 0;
        int nxt = 32 + lane < nblk ? __ldg(trow + 32 + lane) : 0;
        int batch = 0;
        const int grp = lane >> 3;                      // step offset within an issue
        const int bb = lane & (C::kBlk - 1);            // block of the step
        const int hf = (lane >> 2) & 1;                 // 64-column half
        const bool box_lane = hf < C::kHalves;          // head_dim 64: one half
        while (ok && issued < nsteps) {
            const int j = issued;
            if ((j >> 3) != batch) {
                batch = j >> 3;
                cur = nxt;
                const int ni = 32 * (batch + 1) + lane;
                nxt = ni < nblk ? __ldg(trow + ni) : 0;
            }
            const int maxn = min(4, min(nsteps - j, 8 - (j & 7)));
            bool free_stage = false;
            if ((lane & 7) == 0 && grp < maxn)
                free_stage = mbar_test_wait(&empty[(j + grp) % nst], static_cast<uint32_t>(((j + grp) / nst) & 1) ^ 1u);
            const unsigned int fmask = __ballot_sync(0xffffffffu, free_stage);
            int n = 0;
            while (n < maxn && ((fmask >> (8 * n)) & 1u)) ++n;
            if (n == 0) {
                int good = 1;
                if (lane == 0) {
                    PX_T(t0);
                    good = mbar_wait(&empty[j % nst], static_cast<uint32_t>((j / nst) & 1) ^ 1u, a.status, abort_flag,
                                     kWaitLimitNs, kAheadSleepNs)
                               ? 1 : 0;
                    PX_T(t1);
                    PX_ADD(tr_tma, t1 - t0);
                }
                if (!__shfl_sync(0xffffffffu, good, 0)) {
                    ok = false;
                    break;
                }
                n = 1;
            }
            const int jj = j + grp;
            const int bid = __shfl_sync(0xffffffffu, cur, (C::kBlk * jj + bb) & 31);
            if (grp < n) {
                const int st = jj % nst;
                if ((lane & 7) == 0) mbar_arrive_expect_tx(&full[st], C::kKBytes);
                if (box_lane) {
                    int y = -16;
                    if (C::kBlk * jj + bb < nblk) {
                        if (bid >= 0 && bid < a.num_blocks)
                            y = (bid * a.kv_heads + h) * 16;
                        else if (is_k && hf == 0)
                            atomicOr(a.status, PKV_DEVERR_RANGE);
                    }
                    tma_load_2d(ring + st * C::kKBytes + hf * C::kHalfBytes + bb * 2048, map, hf * 64, y, &full[st],
                                policy);
                }
            }
            issued += n;
        }
        if (!ok && lane == 0) {  // after an abort: wait (bounded) for the copies still in flight
            const int first = issued > nst ? issued - nst : 0;
            for (int u = first; u < issued; ++u)
                mbar_wait(&full[u % nst], static_cast<uint32_t>((u / nst) & 1), a.status, nullptr);
        }
        if (lane == 0 && is_k) PX_STAMP(a, 15, tr_tma);
    } else if (warp == C::kSWarp || warp == C::kSWarp1) {
        // ------------------------------------------------ score issuers (one thread each)
        // S_j = Q K_j^T into buffer j % kNumBufs, once the P.V product that
        // read P_{j - kNumBufs} out of it has completed and stage j of K has
        // landed. Both operands K-major; a K-step of 16 elements is 32 bytes
        // into the swizzled row.
        const int par = warp == C::kSWarp ? 0 : 1;  // even or odd steps
        if (lane == 0) {
            constexpr uint32_t idS = umma_idesc_bf16(C::kRows, C::kTok, false, false);
            const uint32_t q_base = smem_u32(smem + C::kOffQ);
#ifdef PKV_TRACE
            unsigned long long tr_kv = 0, tr_buf = 0;
#endif
            for (int j = par; j < nsteps; j += 2) {
                const int b = j % C::kNumBufs;
                PX_T(tb0);
                if (j >= C::kNumBufs && !mbar_wait(&o_done[b], static_cast<uint32_t>((j / C::kNumBufs - 1) & 1),
                                                   a.status, abort_flag, kWaitLimitNs, kAheadSleepNs))
                    break;
                PX_T(tb1);
                PX_ADD(tr_buf, tb1 - tb0);
                const int s = j % C::kKStages;
                PX_T(t0);
                if (!mbar_wait(&k_full[s], static_cast<uint32_t>((j / C::kKStages) & 1), a.status, abort_flag)) break;
                PX_T(t1);
                PX_ADD(tr_kv, t1 - t0);
                tc_fence_after();
                PX_STEP(j, 0);
                const uint32_t k_base = smem_u32(smem + C::kOffK + s * C::kKBytes);
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint64_t ad = umma_desc_sw128(q_base + (kk >> 2) * (C::kRows * 128) + (kk & 3) * 32, 16, 1024);
                    const uint64_t bd = umma_desc_sw128(k_base + (kk >> 2) * C::kHalfBytes + (kk & 3) * 32, 16, 1024);
                    umma_bf16(tmem + C::kColS + b * C::kTok, ad, bd, idS, kk > 0 ? 1u : 0u);
                }
                umma_commit(&k_empty[s]);  // the K stage is free once this product is done
                umma_commit(&s_full[b]);
                PX_STEP(j, 1);
            }
            // nothing may still run on the tensor cores when the memory is freed
            umma_commit(&final_s[par]);
            mbar_wait(&final_s[par], 0, a.status, nullptr);
            if (par == 0) {
                PX_STAMP(a, 14, tr_kv);
                PX_STAMP(a, 6, tr_buf);
            }
        }
        __syncwarp();
    } else if (warp == C::kMmaWarp || warp == C::kMmaWarp1) {
        // ------------------------------------------------ P.V issuers (one thread each, one token half each)
        const int th = warp == C::kMmaWarp ? 0 : 1;
        if (lane == 0) {
            constexpr uint32_t idO = umma_idesc_bf16(C::kRows, D, false, true);
            bool ok = true;
#ifdef PKV_TRACE
            unsigned long long tr_p = 0, tr_v = 0;
#endif
            // prefill: the step and stage row of the first slot past the
            // sequence's end, when that slot lies in a block this CTA streams
            int tail_step = -1, tail_row = 0;
            if constexpr (PF) {
                const int n_end = info[7];
                const int bl = n_end >> 4;
                if ((n_end & 15) != 0 && bl >= blk0 && bl < blk0 + nblk) {
                    tail_step = (bl - blk0) / C::kBlk;
                    tail_row = ((bl - blk0) % C::kBlk) * 16 + (n_end & 15);
                }
            }
            for (int j = 0; ok && j < nsteps; ++j) {
                PX_T(t0);
                const int b = j % C::kNumBufs;
                if (!mbar_wait(&p_full[th * C::kNumBufs + b], static_cast<uint32_t>((j / C::kNumBufs) & 1), a.status,
                               abort_flag)) {
                    ok = false;
                    break;
                }
                PX_T(t1);
                PX_ADD(tr_p, t1 - t0);
                // O_t += P_hi V + P_lo V over token half t (tokens 32t .. 32t+31)
                // into that half's accumulator. P is K-major (tokens along the
                // row); V is MN-major straight from the TMA layout: 64 columns
                // per 128-byte row, the two column halves kHalfBytes apart, 8
                // token rows per 1024-byte atom.
                const int s = j % C::kVStages;
                if (!mbar_wait(&v_full[s], static_cast<uint32_t>((j / C::kVStages) & 1), a.status, abort_flag)) {
                    ok = false;
                    break;
                }
                PX_T(tv1);
                PX_ADD(tr_v, tv1 - t1);
                tc_fence_after();
                if constexpr (PF) {
                    // The slots of the sequence's last block past its length may
                    // hold anything, NaN included. P is zero there, but 0 * NaN
                    // is not, so those V rows are zeroed before the product.
                    if (j == tail_step && tail_row / 32 == th) {  // the tail lies in this issuer's token half
                        uint8_t* vt = smem + C::kOffV + s * C::kKBytes;
                        for (int hf = 0; hf < C::kHalves; ++hf)
                            for (int row = tail_row; row < (tail_row | 15) + 1; ++row)
#pragma unroll
                                for (int c = 0; c < 8; ++c)
                                    *reinterpret_cast<uint4*>(vt + hf * C::kHalfBytes + row * 128 + c * 16) =
                                        make_uint4(0u, 0u, 0u, 0u);
                        fence_proxy_async_smem();
                    }
                }
                PX_STEP(j, 4);
                const uint32_t v_base = smem_u32(smem + C::kOffV + s * C::kKBytes);
                // token half th of P sits in columns 32 th .. 32 th + 31 of the
                // buffer: hi of tokens 32 th + 2c, + 1 in column 32 th + c, lo 16 further
                const uint32_t p_col = tmem + C::kColS + b * C::kTok;
#pragma unroll
                for (int part = 0; part < 2; ++part) {
#pragma unroll
                    for (int kt = 2 * th; kt < 2 * th + 2; ++kt) {
                        const uint64_t bd = umma_desc_sw128(v_base + kt * 2048, C::kHalfBytes, 1024);
                        umma_bf16_ts(tmem + C::kColO + th * D, p_col + 32 * th + 16 * part + 8 * (kt & 1), bd, idO,
                                     (j > 0 || part > 0 || kt > 2 * th) ? 1u : 0u);
                    }
                }
                umma_commit(&v_empty[s]);
                umma_commit(&o_done[b]);
                PX_STEP(j, 5);
            }
            // nothing may still run on the tensor cores when the memory is freed
            umma_commit(&final_bar[th]);
            mbar_wait(&final_bar[th], 0, a.status, nullptr);
            if (th == 0) {
                PX_STAMP(a, 13, tr_p);
                PX_STAMP(a, 4, tr_v);
            }
        }
        __syncwarp();
    }

    // ---------------------------------------------------- softmax warps
    // Thread (warp w < 8, lane i) keeps the online softmax of row 32 (w % 4) + i
    // over token half w / 4 of every step, with its own running max, sum and O
    // accumulator; the two halves of a row are combined once, at the end.
    float m = ninf(), l = 0.f;  // running max (base 2, scaled) and sum
    bool ok = true;
    const int q4 = warp & 3;
    const int th = (warp >> 2) & 1;  // token half of this softmax warp
    const uint32_t lane_base = static_cast<uint32_t>(q4 * 32) << 16;
    const uint32_t col_o = C::kColO + th * D;
    float* xfer = reinterpret_cast<float*>(smem + C::kOffX);  // [3][128]: half 1's max, sum, status
    // This chunk's partial of the tile's rows, in this CTA's shared memory over
    // the K/V rings (idle once the loop is done): O unnormalised [128][D + 4],
    // the running maxima, the sums. A CTA without the chunk, or one that gave
    // up, leaves empty rows (sum 0).
    constexpr int kPS = D + 4;
    float* part = reinterpret_cast<float*>(smem + C::kOffK);
    float* part_m = part + C::kRows * kPS;
    float* part_l = part_m + C::kRows;
    float* wts = part_l + C::kRows;  // [rows combined here][kMaxCluster + 1]
    int* rowoff = reinterpret_cast<int*>(wts + C::kRows * (kMaxCluster + 1));
    static_assert(C::kRows * (kPS + 2 + kMaxCluster + 2) * 4 <= C::kRingBytes, "partial fits the rings");
    if (warp < C::kSoftmaxWarps) {
        const int r = q4 * 32 + lane;
        const float scale_log2 = a.scale * kLog2e;
        // prefill: the last token position this row sees (-1 for a padding row)
        const int lim = PF ? (r < nrows ? info[7] - info[8] + (r0 + r) / G : -1) : 0;
#ifdef PKV_TRACE
        unsigned long long tr_s = 0, tr_ld = 0, tr_math = 0, tr_o = 0, tr_w = 0;
#endif
        for (int j = 0; j < nsteps; ++j) {
            PX_T(t0);
            const int bb = j % C::kNumBufs;
            if (!mbar_wait(&s_full[bb], static_cast<uint32_t>((j / C::kNumBufs) & 1), a.status, abort_flag)) {
                ok = false;
                break;
            }
            tc_fence_after();
            PX_T(t1);
            if (threadIdx.x == 0) PX_STEP(j, 2);
            uint32_t sv[32];
            tmem_ld32(tmem + lane_base + C::kColS + bb * C::kTok + th * 32, sv);
            tmem_ld_wait();
            PX_T(t2);
            int valid = min(C::kTok, (nblk - C::kBlk * j) * 16) - th * 32;
            if constexpr (PF) valid = min(valid, lim - ((blk0 + C::kBlk * j) * 16 + th * 32) + 1);
            // P = 2^(x - m) as bf16 hi + lo, both truncated: hi is the top half of
            // p, lo the top half of p - hi (together ~16 significant bits),
            // written over this thread's own S columns (already read): hi of
            // tokens 2c, 2c + 1 in column c, lo 16 columns further
            const uint32_t p_col = tmem + lane_base + C::kColS + bb * C::kTok + th * 32;
            uint32_t hi[16], lo[16];
            float psum;
            bool resc;
            float alpha = 1.f;
            {
                // The maximum of scale * s is the scale times the raw maximum (the
                // raw minimum for a negative scale), and 2^(scale * s - m) takes
                // one fused multiply-add per score (two scores per packed
                // instruction). A score past the valid range becomes an infinity
                // that the scale turns into -inf (weight 0). A zero scale is
                // replaced by 1e-30: every finite score then gives the same
                // weights in float32, and an infinity stays infinite.
                const bool pos = scale_log2 >= 0.f;
                const float sl = scale_log2 == 0.f ? 1e-30f : scale_log2;
                float x[32];
#pragma unroll
                for (int t = 0; t < 32; ++t) x[t] = __uint_as_float(sv[t]);
                if (valid < 32) {
                    const float kill = pos ? ninf() : -ninf();
#pragma unroll
                    for (int t = 0; t < 32; ++t)
                        if (t >= valid) x[t] = kill;
                }
                float ext;
                if (pos) {
                    float m1[11];
#pragma unroll
                    for (int k = 0; k < 10; ++k) m1[k] = fmax3(x[3 * k], x[3 * k + 1], x[3 * k + 2]);
                    m1[10] = fmaxf(x[30], x[31]);
                    ext = fmaxf(fmax3(fmax3(m1[0], m1[1], m1[2]), fmax3(m1[3], m1[4], m1[5]),
                                      fmax3(m1[6], m1[7], m1[8])),
                                fmaxf(m1[9], m1[10]));
                } else {
                    float m1[11];
#pragma unroll
                    for (int k = 0; k < 10; ++k) m1[k] = fmin3(x[3 * k], x[3 * k + 1], x[3 * k + 2]);
                    m1[10] = fminf(x[30], x[31]);
                    ext = fminf(fmin3(fmin3(m1[0], m1[1], m1[2]), fmin3(m1[3], m1[4], m1[5]),
                                      fmin3(m1[6], m1[7], m1[8])),
                                fminf(m1[9], m1[10]));
                }
                const float mx = valid > 0 ? ext * sl : ninf();
                // lazy rescale: the running max moves only when a score exceeds it by more than 8
                resc = mx > m + 8.f;
                if (resc) {
                    const float mn = fmaxf(m, mx);
                    alpha = m == ninf() ? 0.f : ex2(m - mn);
                    m = mn;
                }
                const float base = m == ninf() ? 0.f : m;  // a half with no valid token yet
                const uint64_t sc2 = f32x2_pack(sl, sl), nb2 = f32x2_pack(-base, -base);
                uint64_t acc0 = f32x2_pack(0.f, 0.f), acc1 = acc0;
                // two groups of 16 tokens: the first group's stores overlap the
                // second group's arithmetic
#pragma unroll
                for (int g = 0; g < 2; ++g) {
#pragma unroll
                    for (int t = 16 * g; t < 16 * g + 16; t += 2) {
                        float a0, a1;
                        f32x2_unpack(f32x2_fma(f32x2_pack(x[t], x[t + 1]), sc2, nb2), a0, a1);
                        const float p0 = ex2(a0), p1 = ex2(a1);
                        hi[t / 2] = pack_bf16x2_trunc(p0, p1);
                        const uint64_t pp = f32x2_pack(p0, p1);
                        float r0, r1;
                        f32x2_unpack(f32x2_sub(pp, f32x2_pack(bf16_trunc(p0), bf16_trunc(p1))), r0, r1);
                        lo[t / 2] = pack_bf16x2_trunc(r0, r1);
                        if ((t / 2) & 1)
                            acc1 = f32x2_add(acc1, pp);
                        else
                            acc0 = f32x2_add(acc0, pp);
                    }
                    tmem_st8(p_col + 8 * g, hi + 8 * g);
                    tmem_st8(p_col + 16 + 8 * g, lo + 8 * g);
                }
                float s0, s1, s2, s3;
                f32x2_unpack(acc0, s0, s1);
                f32x2_unpack(acc1, s2, s3);
                psum = (s0 + s1) + (s2 + s3);
            }
            l = l * alpha + psum;
            PX_T(t3);
            // rescale this half's O in tensor memory once the PV product of step j - 1 is in
            if (__any_sync(0xffffffffu, resc && j > 0)) {
                if (!mbar_wait(&o_done[(j - 1) % C::kNumBufs], static_cast<uint32_t>(((j - 1) / C::kNumBufs) & 1),
                               a.status, abort_flag)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
#pragma unroll
                for (int c = 0; c < D; c += 32) {
                    uint32_t ov[32];
                    tmem_ld32(tmem + lane_base + col_o + c, ov);
                    tmem_ld_wait();
#pragma unroll
                    for (int e = 0; e < 32; ++e) ov[e] = __float_as_uint(__uint_as_float(ov[e]) * alpha);
                    tmem_st32(tmem + lane_base + col_o + c, ov);
                }
                tmem_st_wait();
            }
            PX_T(t4);
            tmem_st_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&p_full[th * C::kNumBufs + bb]);
            if (threadIdx.x == 0) PX_STEP(j, 3);
            PX_T(t5);
            PX_ADD(tr_s, t1 - t0);
            PX_ADD(tr_ld, t2 - t1);
            PX_ADD(tr_math, t3 - t2);
            PX_ADD(tr_o, t4 - t3);
            PX_ADD(tr_w, t5 - t4);
        }
        if (threadIdx.x == 0) {
            PX_STAMP(a, 3, global_ns());
            PX_STAMP(a, 8, tr_s);
            PX_STAMP(a, 9, tr_ld);
            PX_STAMP(a, 10, tr_math);
            PX_STAMP(a, 11, tr_o);
            PX_STAMP(a, 12, tr_w);
        }
        // the last PV product must be in before O is read or the P buffers reused
        if (ok && nsteps > 0 &&
            !mbar_wait(&o_done[(nsteps - 1) % C::kNumBufs], static_cast<uint32_t>(((nsteps - 1) / C::kNumBufs) & 1), a.status,
                       abort_flag))
            ok = false;
        tc_fence_after();
        if (th == 1) {
            xfer[r] = m;
            xfer[C::kRows + r] = l;
            xfer[2 * C::kRows + r] = ok ? 1.f : 0.f;
        }
        named_barrier_sync(1, 32 * C::kSoftmaxWarps);
        if (th == 0) {
            // combine the row's two halves into the partial, 32 columns at a time
            const float m1 = xfer[r], l1 = xfer[C::kRows + r];
            const bool ok1 = xfer[2 * C::kRows + r] != 0.f;
            const bool has0 = ok && l > 0.f, has1 = ok1 && l1 > 0.f;
            const float M = fmaxf(has0 ? m : ninf(), has1 ? m1 : ninf());
            const float w0 = has0 ? ex2(m - M) : 0.f, w1 = has1 ? ex2(m1 - M) : 0.f;
            const float lc = (has0 ? w0 * l : 0.f) + (has1 ? w1 * l1 : 0.f);
            const bool live = !*abort_flag && lc > 0.f;
            if (PF && gridDim.y == 1) {
                // one chunk per tile: the row is final here, so it is normalised
                // and written at once (no partial, no cluster combine). The
                // tensor-memory loads are warp-wide, so every lane takes part;
                // only rows that exist are stored.
                const int Rg = r0 + r;
                const int t = Rg / G;
                __nv_bfloat16* orow = static_cast<__nv_bfloat16*>(a.out) +
                                      (static_cast<long long>(info[9] + t) * a.q_heads + h * G + (Rg - t * G)) * D;
                const float inv = live ? 1.f / lc : 0.f;
                const float v0 = w0 * inv, v1 = w1 * inv;
#pragma unroll
                for (int c = 0; c < D; c += 32) {
                    uint32_t o0[32], o1[32];
                    tmem_ld32(tmem + lane_base + C::kColO + c, o0);
                    tmem_ld32(tmem + lane_base + C::kColO + D + c, o1);
                    tmem_ld_wait();
                    if (r < nrows) {
#pragma unroll
                        for (int e = 0; e < 32; e += 8) {
                            uint32_t w[4];
#pragma unroll
                            for (int u = 0; u < 4; ++u) {
                                const float y0 = (has0 ? v0 * __uint_as_float(o0[e + 2 * u]) : 0.f) +
                                                 (has1 ? v1 * __uint_as_float(o1[e + 2 * u]) : 0.f);
                                const float y1 = (has0 ? v0 * __uint_as_float(o0[e + 2 * u + 1]) : 0.f) +
                                                 (has1 ? v1 * __uint_as_float(o1[e + 2 * u + 1]) : 0.f);
                                w[u] = pack_bf16x2(y0, y1);
                            }
                            *reinterpret_cast<uint4*>(orow + c + e) = make_uint4(w[0], w[1], w[2], w[3]);
                        }
                    }
                }
            } else {
            fence_proxy_async_smem();  // the rings were last written by TMA
#pragma unroll
            for (int c = 0; c < D; c += 32) {
                uint32_t o0[32], o1[32];
                tmem_ld32(tmem + lane_base + C::kColO + c, o0);
                tmem_ld32(tmem + lane_base + C::kColO + D + c, o1);
                tmem_ld_wait();
#pragma unroll
                for (int e = 0; e < 32; e += 4) {
                    float v[4];
#pragma unroll
                    for (int u = 0; u < 4; ++u)
                        v[u] = live ? (has0 ? w0 * __uint_as_float(o0[e + u]) : 0.f) +
                                          (has1 ? w1 * __uint_as_float(o1[e + u]) : 0.f)
                                    : 0.f;
                    *reinterpret_cast<float4*>(part + r * kPS + c + e) = make_float4(v[0], v[1], v[2], v[3]);
                }
            }
            part_m[r] = live ? M : ninf();
            part_l[r] = live ? lc : 0.f;
            }
        }
    }
    // ---- tensor memory is no longer read: free it
    tc_fence_before();
    __syncthreads();
    if (warp == C::kMmaWarp) {
        tc_fence_after();
        tmem_dealloc(tmem, C::kTmemCols);
    }
    if (PF && gridDim.y == 1) {  // the rows went out above
        if (threadIdx.x == 0) PX_STAMP(a, 5, global_ns());
        return;
    }

    cluster_sync();
    grid_dependency_wait();  // fold_o / fold_lse come from the decode kernel

    // ---- CTA k of the cluster combines rows [k R, (k + 1) R) of the tile: the
    // chunks' partials (distributed shared memory) and the own-token partial
    // (lse_s, normalised o_s), all weights in base 2
    const int cn = gridDim.y;  // CTAs of the cluster = chunks
    const int rank = static_cast<int>(cluster_ctarank());
    const int R = (C::kRows + cn - 1) / cn;
    const int rb = rank * R;
    const uint32_t part_addr = smem_u32(part);
    if (static_cast<int>(threadIdx.x) < R) {
        const int rr = threadIdx.x;
        const int r = rb + rr;
        int off = -1;
        if (r < nrows) {
            const int Rg = r0 + r;
            if constexpr (PF) {
                const int t = Rg / G;
                off = (info[9] + t) * a.q_heads + h * G + (Rg - t * G);
            } else {
                const int mm = Rg / G;
                off = members[mm - m0] * a.q_heads + h * G + (Rg - mm * G);
            }
            const float ls = PF ? ninf() : __ldcg(a.fold_lse + off);  // no own-token partial in prefill
            float mc[kMaxCluster], lc[kMaxCluster];
            float Mx = ls;
#pragma unroll
            for (int c = 0; c < kMaxCluster; ++c) {
                mc[c] = ninf();
                lc[c] = 0.f;
                if (c < cn) {
                    const uint32_t ad = mapa_shared(part_addr + (C::kRows * kPS + r) * 4, c);
                    mc[c] = ld_cluster_f32(ad);
                    lc[c] = ld_cluster_f32(ad + C::kRows * 4);
                }
            }
#pragma unroll
            for (int c = 0; c < kMaxCluster; ++c)
                if (lc[c] > 0.f) Mx = fmaxf(Mx, mc[c]);
            float den = 0.f, ws = 0.f;
            if (Mx != ninf()) {
                ws = ls == ninf() ? 0.f : ex2(ls - Mx);
                den = ws;
#pragma unroll
                for (int c = 0; c < kMaxCluster; ++c)
                    if (lc[c] > 0.f) den += lc[c] * ex2(mc[c] - Mx);
            }
            const float inv = den > 0.f ? 1.f / den : 0.f;
#pragma unroll
            for (int c = 0; c < kMaxCluster; ++c)
                wts[rr * (kMaxCluster + 1) + c] = lc[c] > 0.f ? ex2(mc[c] - Mx) * inv : 0.f;
            wts[rr * (kMaxCluster + 1) + kMaxCluster] = ws * inv;
        }
        rowoff[rr] = off;
    }
    __syncthreads();
    for (int u = threadIdx.x; u < R * (D / 4); u += blockDim.x) {
        const int rr = u / (D / 4);
        const int c4 = u - rr * (D / 4);
        const int off = rowoff[rr];
        if (off < 0) continue;
        const float* wr = wts + rr * (kMaxCluster + 1);
        const float wsr = wr[kMaxCluster];
        (void)wsr;
        float4 o4 = make_float4(0.f, 0.f, 0.f, 0.f);
        if constexpr (!PF) {
            const float4 f = __ldcg(reinterpret_cast<const float4*>(a.fold_o + static_cast<long long>(off) * D + 4 * c4));
            o4 = make_float4(wsr * f.x, wsr * f.y, wsr * f.z, wsr * f.w);
        }
        const uint32_t la = part_addr + ((rb + rr) * kPS + 4 * c4) * 4;
#pragma unroll
        for (int c = 0; c < kMaxCluster; ++c) {
            if (c < cn && wr[c] != 0.f) {
                const float4 v = ld_cluster_v4(mapa_shared(la, c));
                o4.x += wr[c] * v.x;
                o4.y += wr[c] * v.y;
                o4.z += wr[c] * v.z;
                o4.w += wr[c] * v.w;
            }
        }
        *reinterpret_cast<uint2*>(static_cast<__nv_bfloat16*>(a.out) + static_cast<long long>(off) * D + 4 * c4) =
            make_uint2(pack_bf16x2(o4.x, o4.y), pack_bf16x2(o4.z, o4.w));
    }
    cluster_sync();  // each CTA's partial stays in place until the whole cluster has read it
    if (threadIdx.x == 0) PX_STAMP(a, 5, global_ns());
}

// ------------------------------------------------------------------ checked mode
// One CTA per sequence: a member of a group must satisfy the membership rule
// and its first group_blocks[g] table entries must equal those of the
// group's first member.
__global__ void check_groups_kernel(const int32_t* tables, int32_t max_blocks, const int32_t* lens,
                                    const int32_t* prefix_group, const int32_t* group_blocks, int32_t num_groups,
                                    int32_t max_group_blocks, int32_t batch, unsigned int* verdict) {
    __shared__ int first;
    const int i = blockIdx.x;
    const int g = prefix_group[i];
    if (g < 0) return;
    if (threadIdx.x == 0) first = i;
    int n = lens[i];
    n = n < 0 ? 0 : (n > max_blocks * 16 ? max_blocks * 16 : n);
    const int nb = prefix_member_blocks(prefix_group, group_blocks, num_groups, max_group_blocks, n, i);
    if (nb < 0) {
        if (threadIdx.x == 0) atomicOr(verdict, kVerdictRange);
        return;
    }
    __syncthreads();
    for (int j = threadIdx.x; j < i; j += blockDim.x)
        if (prefix_group[j] == g) atomicMin(&first, j);
    __syncthreads();
    const int32_t* mine = tables + static_cast<long long>(i) * max_blocks;
    const int32_t* theirs = tables + static_cast<long long>(first) * max_blocks;
    for (int t = threadIdx.x; t < nb; t += blockDim.x)
        if (mine[t] != theirs[t]) atomicOr(verdict, kVerdictRange);
}

// Resident CTAs per SM of a kernel (cached per device); sets its dynamic
// shared-memory limit once.
template <typename K>
int kernel_occupancy(K kernel, int threads, size_t smem, int slot) {
    static std::mutex mu;
    static int cache[6][64] = {};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 0 || dev >= 64) dev = 0;
    std::lock_guard<std::mutex> lock(mu);
    if (cache[slot][dev] == 0) {
        cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
        int n = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kernel, threads, smem) != cudaSuccess || n < 1) n = 1;
        cache[slot][dev] = n;
    }
    return cache[slot][dev];
}

constexpr int kMmaStages = 4;

int occupancy_of(int kernel, int head_dim) {
    if (kernel == 1)
        return head_dim == 128
                   ? kernel_occupancy(prefix_mma_kernel<128, kMmaStages>, Px<128, kMmaStages>::kThreads,
                                      Px<128, kMmaStages>::kSmem, 0)
                   : kernel_occupancy(prefix_mma_kernel<64, kMmaStages>, Px<64, kMmaStages>::kThreads,
                                      Px<64, kMmaStages>::kSmem, 1);
    if (kernel == 3)  // the prefill mode of the tcgen05 kernel
        return head_dim == 128 ? kernel_occupancy(prefix_umma_kernel<128, true>, Ux<128>::kThreads, Ux<128>::kSmem, 4)
                               : kernel_occupancy(prefix_umma_kernel<64, true>, Ux<64>::kThreads, Ux<64>::kSmem, 5);
    return head_dim == 128 ? kernel_occupancy(prefix_umma_kernel<128, false>, Ux<128>::kThreads, Ux<128>::kSmem, 2)
                           : kernel_occupancy(prefix_umma_kernel<64, false>, Ux<64>::kThreads, Ux<64>::kSmem, 3);
}

// Clusters of `c` CTAs of the tcgen05 kernel (pf: its prefill mode) that fit
// on the device at once (cached per device and size).
int active_clusters(int head_dim, int c, bool pf = false) {
    static std::mutex mu;
    static int cache[2][2][kMaxCluster + 1][64] = {};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 0 || dev >= 64) dev = 0;
    const int hd = head_dim == 128 ? 1 : 0;
    std::lock_guard<std::mutex> lock(mu);
    int& slot = cache[pf ? 1 : 0][hd][c][dev];
    if (slot == 0) {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(1, c, 1);
        cfg.blockDim = dim3(hd ? Ux<128>::kThreads : Ux<64>::kThreads);
        cfg.dynamicSmemBytes = hd ? Ux<128>::kSmem : Ux<64>::kSmem;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = 1;
        attr[0].val.clusterDim.y = c;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        int n = 0;
        cudaError_t e;
        if (pf)
            e = hd ? cudaOccupancyMaxActiveClusters(&n, prefix_umma_kernel<128, true>, &cfg)
                   : cudaOccupancyMaxActiveClusters(&n, prefix_umma_kernel<64, true>, &cfg);
        else
            e = hd ? cudaOccupancyMaxActiveClusters(&n, prefix_umma_kernel<128, false>, &cfg)
                   : cudaOccupancyMaxActiveClusters(&n, prefix_umma_kernel<64, false>, &cfg);
        if (e != cudaSuccess || n < 1) {
            cudaGetLastError();
            n = -1;  // not launchable at this size
        }
        slot = n;
    }
    return slot;
}

template <int D>
cudaError_t run_prefix(const PrefixArgs& a, int kernel, cudaStream_t s) {
    CUtensorMap tmK, tmV;
    const int64_t rows = a.num_blocks * a.kv_heads * 16;
    if (!make_pool_map(&tmK, a.k_cache, rows, D) || !make_pool_map(&tmV, a.v_cache, rows, D))
        return cudaErrorInvalidValue;
    occupancy_of(kernel, D);  // sets the shared-memory limit once per device
    const dim3 grid(a.tiles, a.chunks, a.kv_heads);
    if (kernel == 1)
        return launch_pdl(prefix_mma_kernel<D, kMmaStages>, grid, dim3(Px<D, kMmaStages>::kThreads),
                          Px<D, kMmaStages>::kSmem, s, a, tmK, tmV);
    return launch_pdl_cluster(prefix_umma_kernel<D, false>, grid, dim3(Ux<D>::kThreads), dim3(1, a.chunks, 1),
                              Ux<D>::kSmem, s, a, tmK, tmV);
}

// Chunked prefill: tiles of 128 query rows (every sequence padded to whole
// tiles, at most max_query_len queries each); each (tile, KV head) is one
// cluster whose CTAs split the context into chunks of whole 64-token steps,
// as many as fill the device with one wave when the tiles are few.
template <int D>
cudaError_t run_prefill(PrefixArgs& a, cudaStream_t s) {
    CUtensorMap tmK, tmV;
    const int64_t rows = a.num_blocks * a.kv_heads * 16;
    if (!make_pool_map(&tmK, a.k_cache, rows, D) || !make_pool_map(&tmV, a.v_cache, rows, D))
        return cudaErrorInvalidValue;
    occupancy_of(3, D);  // sets the shared-memory limit once per device
    const int per_seq = (a.max_query_len * a.group + Ux<D>::kRows - 1) / Ux<D>::kRows;
    a.tiles = a.batch * per_seq;
    const int pairs = a.tiles * a.kv_heads;
    int c = device_sm_count() / (pairs > 0 ? pairs : 1);
    c = c < 1 ? 1 : (c > kMaxCluster ? kMaxCluster : c);
    while (c > 1 && active_clusters(D, c, true) < 1) --c;
    int cb = (a.max_blocks + c - 1) / c;
    cb = (cb + Ux<D>::kBlk - 1) / Ux<D>::kBlk * Ux<D>::kBlk;
    a.chunk_blocks = cb;
    a.chunks = (a.max_blocks + cb - 1) / cb;
    if (a.tiles == 0) return cudaSuccess;
    return launch_pdl_cluster(prefix_umma_kernel<D, true>, dim3(a.tiles, a.chunks, a.kv_heads), dim3(Ux<D>::kThreads),
                              dim3(1, a.chunks, 1), Ux<D>::kSmem, s, a, tmK, tmV);
}

size_t align256(size_t x) { return (x + 255) / 256 * 256; }

}  // namespace

PrefixPlan prefix_plan(int batch, int num_groups, int q_heads, int kv_heads, int head_dim, int max_group_blocks,
                       size_t base_offset, int kernel) {
    const int b = batch < 1 ? 1 : (batch < kMaxBatchPerLaunch ? batch : kMaxBatchPerLaunch);
    const int G = q_heads / kv_heads;
    PrefixPlan p;
    p.kernel = kernel == 1 ? 1 : 2;
    p.rows = p.kernel == 1 ? Px<128, kMmaStages>::kRows : Ux<128>::kRows;
    // blocks per chunk: a multiple of the tcgen05 kernel's 4-block step
    const int quantum = p.kernel == 1 ? 1 : Ux<128>::kBlk;
    const int full_tiles = (b * G + p.rows - 1) / p.rows;  // every sequence in one group
    p.tiles = full_tiles + (num_groups < b ? num_groups : b);  // one partly filled tile per group at most
    // Split the shared blocks so that a batch in one group fills the GPU with
    // one wave of resident CTAs (two for the mma.sync kernel, whose CTAs
    // are small).
    const int per_sm = occupancy_of(p.kernel, head_dim);
    const int want = (p.kernel == 1 ? 2 : 1) * per_sm * device_sm_count();
    const int pairs = full_tiles * kv_heads;
    int chunks = want / pairs;
    if (p.kernel == 2) {
        // one cluster of `chunks` CTAs per (tile, KV head): the largest
        // cluster size at which all of them fit on the device at once
        int c = chunks < kMaxCluster ? (chunks < 1 ? 1 : chunks) : kMaxCluster;
        while (c > 1 && active_clusters(head_dim, c) < pairs) --c;
        chunks = c;
    }
    const size_t slot_bytes = static_cast<size_t>(p.rows) * (head_dim + 2) * sizeof(float);
    const size_t cap_chunks = (static_cast<size_t>(256) << 20) / (static_cast<size_t>(p.tiles) * kv_heads * slot_bytes);
    if (chunks > (p.kernel == 1 ? kMaxChunks : kMaxCluster)) chunks = p.kernel == 1 ? kMaxChunks : kMaxCluster;
    if (static_cast<size_t>(chunks) > cap_chunks) chunks = static_cast<int>(cap_chunks);
    if (chunks < 1) chunks = 1;
    int cb = max_group_blocks > 0 ? (max_group_blocks + chunks - 1) / chunks : 1;
    cb = (cb + quantum - 1) / quantum * quantum;
    p.chunk_blocks = cb;
    p.chunks = max_group_blocks > 0 ? (max_group_blocks + cb - 1) / cb : 1;
    size_t off = align256(base_offset);
    p.counters_offset = off;
    off = align256(off + static_cast<size_t>(p.tiles) * kv_heads * 4 * sizeof(int));
    p.partials_offset = off;
    // the tcgen05 kernel combines its chunks through distributed shared memory
    if (p.chunks > 1 && p.kernel == 1)
        off = align256(off + static_cast<size_t>(p.tiles) * kv_heads * p.chunks * slot_bytes);
    p.fold_o_offset = off;
    off = align256(off + static_cast<size_t>(b) * q_heads * head_dim * sizeof(float));
    p.fold_lse_offset = off;
    off = align256(off + static_cast<size_t>(b) * q_heads * sizeof(float));
#ifdef PKV_TRACE
    p.trace_offset = off;
    off = align256(off + static_cast<size_t>(p.tiles) * p.chunks * kv_heads * 128);
#else
    p.trace_offset = 0;
#endif
    p.total = off;
    return p;
}

cudaError_t launch_prefix(const PrefixArgs& a, int kernel, cudaStream_t s) {
    return a.head_dim == 128 ? run_prefix<128>(a, kernel, s) : run_prefix<64>(a, kernel, s);
}

cudaError_t launch_prefill(PrefixArgs& a, cudaStream_t s) {
    return a.head_dim == 128 ? run_prefill<128>(a, s) : run_prefill<64>(a, s);
}

cudaError_t launch_check_groups(const int32_t* tables, int32_t max_blocks, const int32_t* lens,
                                const int32_t* prefix_group, const int32_t* group_blocks, int32_t num_groups,
                                int32_t max_group_blocks, int32_t batch, unsigned int* verdict, cudaStream_t s) {
    if (batch <= 0) return cudaSuccess;
    check_groups_kernel<<<batch, 128, 0, s>>>(tables, max_blocks, lens, prefix_group, group_blocks, num_groups,
                                              max_group_blocks, batch, verdict);
    return cudaGetLastError();
}

}  // namespace pkv

#ifdef PKV_TRACE
// Trace builds only: copies the prefill stamps (65536 CTAs x 16 words) to `host`.
extern "C" __attribute__((visibility("default"))) int pkv_trace_copy_prefill(void* host, size_t bytes) {
    return static_cast<int>(cudaMemcpyFromSymbol(host, pkv::g_px_trace, bytes));
}
#endif
