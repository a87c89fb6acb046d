// Chunk-first pass of the shared-prefix (two-phase) decode.
//
// A group is a set of sequences whose block tables begin with the same
// group_blocks[p] physical blocks (notebook section 5: share_prefix gives the
// target the source's leading blocks). The decode kernel, in prefixed mode,
// has already attended every member over its own tokens past those blocks
// and left the normalised result with its log2-sum-exp in fold_o / fold_lse.
// This kernel attends the queries of all members of a group together over
// the shared blocks -- each shared K/V block is read once per 64 query rows
// instead of once per sequence -- and combines the two partials by their
// log-sum-exp weights into the output rows (paper-search page, ChunkAttention
// abstract: "two-phase partition", shared chunks first, then each sequence).
//
// Work decomposition. The query rows of group p are (member m, query head g
// of KV head h) in member order, row r = m * G + g. CTA (x, y, z) takes
// 64-row tile x of the list of all groups' tiles (each group's rows padded to
// a whole tile), chunk y of the group's shared blocks and KV head z. A group
// whose shared blocks fit in one chunk is finished by its CTA directly;
// otherwise each chunk leaves an fp32 partial (unnormalised O, running max m,
// sum l) per row, and for each warp's 16 rows the last of the chunks' warps
// to finish (an atomic counter per tile, head and warp) merges them.
//
// Inside a CTA one producer warp streams the chunk's K and V blocks of head
// z through an NST-stage shared-memory ring with 2-D TMA loads (128-byte
// swizzle, L2 evict-last: the other tiles of the group read the same
// blocks). Four consumer warps own 16 query rows each and all consume every
// block:
//     S[16 rows][16 tokens] = Q[16][D] K^T           (mma m16n8k16, 2 n-tiles)
//     online softmax on the S fragments in fp32, base 2
//     O[16][D] += P[16][16] V[16][D]                  (mma m16n8k16)
// The S accumulator fragments are already laid out as the A operand of P;
// P is split into bf16 hi + lo as in the decode kernel.
#include <math.h>
#include <mutex>

#include "pkv_device.cuh"
#include "pkv_internal.h"

namespace pkv {
namespace {

constexpr float kLog2e = 1.4426950408889634f;
constexpr int kTileRows = 64;
constexpr int kMaxChunks = 32;
constexpr int kMaxGroups = kMaxBatchPerLaunch;
constexpr int kMemberSlots = 72;  // members of one tile: at most 64 / G + 2

__device__ __forceinline__ float ninf() { return __int_as_float(0xff800000); }

template <int D, int NST>
struct Px {
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
    static constexpr size_t kSmem = 1024 + kOffInts + (8 + kMemberSlots + kMaxGroups) * 4;
};

template <int D, int NST>
__global__ void __launch_bounds__(Px<D, NST>::kThreads)
    prefix_tc_kernel(const PrefixArgs a, const __grid_constant__ CUtensorMap tmK,
                     const __grid_constant__ CUtensorMap tmV) {
    using C = Px<D, NST>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::kOffBars);
    uint64_t* empty = full + C::kStages;
    int* stage_ok = reinterpret_cast<int*>(smem + C::kOffFlags);
    volatile int* abort_flag = stage_ok + C::kStages;
    int* info = reinterpret_cast<int*>(smem + C::kOffInts);  // [0] group, [1] tile in group, [2] first member
    int* members = info + 8;
    int* counts = members + kMemberSlots;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int G = a.group;
    const int h = blockIdx.z;
    const int chunk = blockIdx.y;
    const int cap = a.max_blocks * 16;

    if (threadIdx.x == 0) {
        for (int s = 0; s < C::kStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], C::kConsumers);
        }
        *abort_flag = 0;
        info[0] = -1;
        info[2] = 0;
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
    for (int g = threadIdx.x; g < a.num_groups; g += blockDim.x) counts[g] = 0;
    __syncthreads();
    auto member_blocks = [&](int i) {
        int n = a.lens[i];
        n = n < 0 ? 0 : (n > cap ? cap : n);
        return prefix_member_blocks(a.prefix_group, a.group_blocks, a.num_groups, a.max_group_blocks, n, i);
    };
    for (int i = threadIdx.x; i < a.batch; i += blockDim.x)
        if (member_blocks(i) >= 0) atomicAdd(&counts[a.prefix_group[i]], 1);
    __syncthreads();
    if (warp == 0) {
        // tile x -> (group, tile within the group): prefix sums of the groups' tile counts
        int carry = 0;
        for (int base = 0; base < a.num_groups; base += 32) {
            const int g = base + lane;
            const int t = g < a.num_groups ? (counts[g] * G + kTileRows - 1) / kTileRows : 0;
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
    // Every exit waits for the kernel before: this grid must not complete
    // (and release the next kernel in the stream) before that one has.
    if (p < 0) {
        grid_dependency_wait();
        return;
    }
    int nb = a.group_blocks[p];  // in [0, max_group_blocks]: p has members
    const int nch = nb > 0 ? (nb + a.chunk_blocks - 1) / a.chunk_blocks : 1;
    if (chunk >= nch) {
        grid_dependency_wait();
        return;
    }
    const int rows_total = counts[p] * G;
    const int r0 = info[1] * kTileRows;
    const int nrows = min(kTileRows, rows_total - r0);
    const int m0 = r0 / G;
    const int m1 = (r0 + nrows - 1) / G + 1;
    if (warp == 0) {
        int rank = 0;
        for (int base = 0; base < a.batch; base += 32) {
            const int i = base + lane;
            const bool is = i < a.batch && a.prefix_group[i] == p && member_blocks(i) >= 0;
            const unsigned int bal = __ballot_sync(0xffffffffu, is);
            const int r = rank + __popc(bal & ((1u << lane) - 1u));
            if (is) {
                if (r == 0) info[2] = i;
                if (r >= m0 && r < m1) members[r - m0] = i;
            }
            rank += __popc(bal);
        }
    }
    __syncthreads();
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

template <int D, int NST>
int prefix_occupancy() {
    static std::mutex mu;
    static int cache[64] = {0};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 0 || dev >= 64) dev = 0;
    std::lock_guard<std::mutex> lock(mu);
    if (cache[dev] == 0) {
        cudaFuncSetAttribute(prefix_tc_kernel<D, NST>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(Px<D, NST>::kSmem));
        int n = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, prefix_tc_kernel<D, NST>, Px<D, NST>::kThreads,
                                                          Px<D, NST>::kSmem) != cudaSuccess || n < 1)
            n = 1;
        cache[dev] = n;
    }
    return cache[dev];
}

constexpr int kPrefixStages = 4;

template <int D>
cudaError_t run_prefix(const PrefixArgs& a, cudaStream_t s) {
    using C = Px<D, kPrefixStages>;
    CUtensorMap tmK, tmV;
    const int64_t rows = a.num_blocks * a.kv_heads * 16;
    if (!make_pool_map(&tmK, a.k_cache, rows, D) || !make_pool_map(&tmV, a.v_cache, rows, D))
        return cudaErrorInvalidValue;
    prefix_occupancy<D, kPrefixStages>();  // sets the shared-memory attribute once per device
    return launch_pdl(prefix_tc_kernel<D, kPrefixStages>, dim3(a.tiles, a.chunks, a.kv_heads), dim3(C::kThreads),
                      C::kSmem, s, a, tmK, tmV);
}

size_t align256(size_t x) { return (x + 255) / 256 * 256; }

}  // namespace

PrefixPlan prefix_plan(int batch, int num_groups, int q_heads, int kv_heads, int head_dim, int max_group_blocks,
                       size_t base_offset) {
    const int b = batch < 1 ? 1 : (batch < kMaxBatchPerLaunch ? batch : kMaxBatchPerLaunch);
    const int G = q_heads / kv_heads;
    PrefixPlan p;
    const int full_tiles = (b * G + kTileRows - 1) / kTileRows;  // every sequence in one group
    p.tiles = full_tiles + (num_groups < b ? num_groups : b);    // one partly filled tile per group at most
    // Split the shared blocks so that a batch in one group fills the GPU:
    // about two waves of resident CTAs.
    const int per_sm = head_dim == 128 ? prefix_occupancy<128, kPrefixStages>() : prefix_occupancy<64, kPrefixStages>();
    const int want = 2 * per_sm * device_sm_count();
    const int pairs = full_tiles * kv_heads;
    int chunks = (want + pairs - 1) / pairs;
    const size_t slot_bytes = static_cast<size_t>(kTileRows) * (head_dim + 2) * sizeof(float);
    const size_t cap_chunks = (static_cast<size_t>(256) << 20) / (static_cast<size_t>(p.tiles) * kv_heads * slot_bytes);
    if (chunks > kMaxChunks) chunks = kMaxChunks;
    if (static_cast<size_t>(chunks) > cap_chunks) chunks = static_cast<int>(cap_chunks);
    if (chunks > max_group_blocks) chunks = max_group_blocks;
    if (chunks < 1) chunks = 1;
    p.chunk_blocks = max_group_blocks > 0 ? (max_group_blocks + chunks - 1) / chunks : 1;
    p.chunks = max_group_blocks > 0 ? (max_group_blocks + p.chunk_blocks - 1) / p.chunk_blocks : 1;
    size_t off = align256(base_offset);
    p.counters_offset = off;
    off = align256(off + static_cast<size_t>(p.tiles) * kv_heads * 4 * sizeof(int));
    p.partials_offset = off;
    if (p.chunks > 1) off = align256(off + static_cast<size_t>(p.tiles) * kv_heads * p.chunks * slot_bytes);
    p.fold_o_offset = off;
    off = align256(off + static_cast<size_t>(b) * q_heads * head_dim * sizeof(float));
    p.fold_lse_offset = off;
    off = align256(off + static_cast<size_t>(b) * q_heads * sizeof(float));
    p.total = off;
    return p;
}

cudaError_t launch_prefix(const PrefixArgs& a, cudaStream_t s) {
    return a.head_dim == 128 ? run_prefix<128>(a, s) : run_prefix<64>(a, s);
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
