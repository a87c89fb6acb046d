// Split-context decode attention over the paged KV cache, and the
// log-sum-exp merge of split pieces.
//
// Work decomposition. One unit of work is one (sequence i, KV head h, block
// b): 16 tokens of one head, 2 x 16 x head_dim elements of K and V. Units are
// ordered i-major, then h, then b; the units of one (i, h) form a segment. A
// launch of C CTAs gives each CTA a contiguous range of units placed by cost
// (CostSplit in pkv_schedule.cuh): a unit costs 1 and a short segment a few
// units more, so every CTA carries about the same work whatever the mix of
// context lengths. A segment that lies wholly inside one CTA's range is
// finished there and its output row written directly; a segment cut by a
// range boundary leaves one fp32 piece (unnormalised accumulator, running
// max, running sum) per CTA it touches; the CTA that finishes the last piece
// of such a segment (found with an atomic counter in the workspace) combines
// the pieces by log-sum-exp weights and writes the output row. One launch
// per call, no separate merge kernel.
//
// All query heads of a KV head (the GQA group, G <= 8) are computed from one
// read of each K/V byte.
//
// Tensor-core kernel (bf16): two producer warps stream the blocks of the
// CTA's range, one the K boxes and one the V boxes, through an NST-stage
// shared-memory ring with 2-D TMA loads (128-byte swizzle, so ldmatrix reads
// are bank-conflict free). Four consumer warps take the units round robin. Per unit a warp computes
//     S^T[16 tokens][8 heads] = K[16][D] * Q^T[D][8]        (mma m16n8k16)
// runs the online softmax in fp32 on the accumulator fragments, transposes
// P^T into the B-operand layout with movmatrix, and accumulates
//     O^T[D][8] += V^T[D][16] * P^T[16][8]                   (mma m16n8k16)
// with P split as hi + lo bf16 (P itself is fp32; the split keeps ~16
// significant bits, enough for the fp32-accumulation tolerance). At the end
// of a segment piece the four warps' (m, l, O) are combined through shared
// memory.
//
// CUDA-core kernel (fp32 or bf16, any G <= 16): four warps, direct loads,
// lanes split the head dimension; used for fp32 caches and as a second,
// independent implementation in the tests.
#include <math.h>
#include <mutex>
#include <type_traits>

#include "pkv_device.cuh"
#include "pkv_internal.h"
#include "pkv_schedule.cuh"

namespace pkv {
namespace {

constexpr float kLog2e = 1.4426950408889634f;

__device__ __forceinline__ float neg_inf() { return __int_as_float(0xff800000); }

// Build-time tracing (PKV_TRACE): each CTA of the tensor-core kernel records
// %globaltimer stamps in a per-CTA row of 8 words placed after the piece
// slots in the workspace: [0] entry, [1] prologue done, [2] first copy
// issued, [3] first block received, [4] last block consumed, [5] exit,
// [6] the SM the CTA ran on.
#ifdef PKV_TRACE
#define PKV_STAMP(a, cta, i) (reinterpret_cast<unsigned long long*>((a).trace))[(cta) * 8 + (i)] = global_ns()
#else
#define PKV_STAMP(a, cta, i) ((void)0)
#endif

// ------------------------------------------------------------------ schedule
// Cost a segment of nb blocks adds beyond its blocks in the CTA split, in
// blocks: kSegCost when nb < kSegCostBelow, plus max(kSegMinCost - nb, 0)
// (build knobs, passed to the kernels in DecodeArgs; all zero gives every CTA
// the same number of blocks). Swept on the 256-sequence mixed-length layer
// (decode call, 100 back to back): equal block counts 716 us; 4 for every
// segment 674 us but the 8K layer (one segment start per CTA range) 2.5 %
// slower; least cost 16 blocks 683 us; 4 below 256 blocks 674 us with the 8K
// and 128K layers unchanged (their segments are longer).
#ifndef PKV_SEG_COST
#define PKV_SEG_COST 4
#endif
#ifndef PKV_SEG_COST_BELOW
#define PKV_SEG_COST_BELOW 256
#endif
#ifndef PKV_SEG_MIN_COST
#define PKV_SEG_MIN_COST 1
#endif
constexpr int kSegCost = PKV_SEG_COST;
constexpr int kSegCostBelow = PKV_SEG_COST_BELOW;
constexpr int kSegMinCost = PKV_SEG_MIN_COST;

// s_pre[i] = sum_{i' <= i} ceil(len_i' / 16) over this launch's sequences,
// s_len[i] = len_i clamped to [0, max_blocks * 16], s_cost[i] = the sum over
// sequences 0 .. i with blocks of their cost in the CTA split (blocks plus
// seg_extra): the prefixes of the cost-weighted split.
//
// With shared-prefix groups (s_boff non-null) a member of a group (the rule
// of prefix_member_blocks) attends here only its tokens past the group's
// shared blocks: s_len[i] is that own-token count and s_boff[i] the block
// offset at which they start, -1 for a plain sequence. A sequence that names
// a group but fails the rule sets PKV_DEVERR_RANGE and is attended whole.
__device__ __forceinline__ int seg_extra(int nb, const DecodeArgs& a) {
    return (nb < a.seg_cost_below ? a.seg_cost : 0) + max(a.seg_min_cost - nb, 0);
}
__device__ __forceinline__ int seg_max_unit(const DecodeArgs& a) { return 1 + seg_extra(1, a); }

__device__ void build_prefix(int32_t* s_pre, int32_t* s_len, int32_t* s_cost, int32_t* s_boff, const DecodeArgs& a) {
    const int cap = a.max_blocks * 16;
    for (int i = threadIdx.x; i < a.batch; i += blockDim.x) {
        int n = a.lens[i];
        if (n < 0 || n > cap) {
            if (blockIdx.x == 0) atomicOr(a.status, PKV_DEVERR_RANGE);
            n = n < 0 ? 0 : cap;
        }
        if (s_boff != nullptr) {
            const int nb =
                prefix_member_blocks(a.prefix_group, a.group_blocks, a.num_groups, a.max_group_blocks, n, i);
            if (nb < 0 && a.prefix_group[i] >= 0 && blockIdx.x == 0) atomicOr(a.status, PKV_DEVERR_RANGE);
            s_boff[i] = nb;
            if (nb > 0) n -= nb * 16;
        }
        s_len[i] = n;
        s_pre[i] = (n + 15) >> 4;
        s_cost[i] = n > 0 ? ((n + 15) >> 4) + seg_extra((n + 15) >> 4, a) : 0;
    }
    __syncthreads();
    if (threadIdx.x < 32) {
        const int lane = threadIdx.x;
        int carry = 0, carry_c = 0;
        for (int base = 0; base < a.batch; base += 32) {
            const bool in = base + lane < a.batch;
            int x = in ? s_pre[base + lane] : 0;
            int xc = in ? s_cost[base + lane] : 0;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int y = __shfl_up_sync(0xffffffffu, x, o);
                const int yc = __shfl_up_sync(0xffffffffu, xc, o);
                if (lane >= o) {
                    x += y;
                    xc += yc;
                }
            }
            if (in) {
                s_pre[base + lane] = x + carry;
                s_cost[base + lane] = xc + carry_c;
            }
            carry += __shfl_sync(0xffffffffu, x, 31);
            carry_c += __shfl_sync(0xffffffffu, xc, 31);
        }
    }
    __syncthreads();
}

// Workspace slice of CTA `cta`, piece slot `slot` (0: the piece that opens
// the CTA's range, 1: the one that closes it), consumer warp `warp`:
// S accumulator values, then G maxima, then G sums.
__device__ __forceinline__ float* piece_slice(float* partials, long long cta, int slot, int warp, int S, int G) {
    return partials + ((cta * 2 + slot) * 4 + warp) * static_cast<long long>(S + 2 * G);
}

template <typename T>
__device__ __forceinline__ void store_out(T* p, float x);
template <>
__device__ __forceinline__ void store_out<float>(float* p, float x) {
    *p = x;
}
template <>
__device__ __forceinline__ void store_out<__nv_bfloat16>(__nv_bfloat16* p, float x) {
    *p = __float2bfloat16_rn(x);
}

template <typename T>
__device__ __forceinline__ float load_f32(const T* p);
template <>
__device__ __forceinline__ float load_f32<float>(const float* p) {
    return __ldg(p);
}
template <>
__device__ __forceinline__ float load_f32<__nv_bfloat16>(const __nv_bfloat16* p) {
    return __bfloat162float(*p);
}

// Finish one segment piece for the elements of warp `warp`'s slice.
//
// The four consumer warps of a CTA each own a fixed slice of the G x D output
// elements of the segment (S = G*D/4 elements; element e is head e / D, dim
// e % D). The per-warp online-softmax states (O, m, l) of the piece are in
// shared memory (sm_o[(w*gstride + g)*D + d], sm_m/sm_l[w*gstride + g]).
// A whole segment is normalised and written out directly. A cut segment's
// piece goes to this CTA's slot in the workspace; it is announced later by
// signal_pending. Returns true for a cut segment. With `fold` (a sequence of
// a shared-prefix group) a whole segment's rows go to fold_o / fold_lse
// instead of out.
template <typename T, int D>
__device__ bool write_piece(const float* sm_o, const float* sm_m, const float* sm_l, int gstride, int G,
                            const Piece& pc, const DecodeArgs& a, long long cta, int warp, int lane, bool fold) {
    const int S = G * D / 4;
    const int e0 = warp * S;
    const long long row0 = static_cast<long long>(pc.seq) * a.q_heads + pc.head * G;
    T* out_row = static_cast<T*>(a.out) + row0 * D;
    float* fold_row = fold ? a.fold_o + row0 * D : nullptr;
    float* slice = nullptr;
    if (!pc.complete) slice = piece_slice(a.partials, cta, pc.first ? 0 : 1, warp, S, G);
    for (int e = e0 + lane; e < e0 + S; e += 32) {
        const int g = e / D;
        const int d = e - g * D;
        float M = neg_inf();
        for (int w = 0; w < 4; ++w) M = fmaxf(M, sm_m[w * gstride + g]);
        const float base = (M == neg_inf()) ? 0.f : M;
        float o = 0.f, L = 0.f;
        for (int w = 0; w < 4; ++w) {
            const float mw = sm_m[w * gstride + g];
            const float wt = (mw == neg_inf()) ? 0.f : ex2(mw - base);
            o += wt * sm_o[(w * gstride + g) * D + d];
            L += wt * sm_l[w * gstride + g];
        }
        if (!pc.complete)
            slice[e - e0] = o;
        else if (fold)
            fold_row[e] = L > 0.f ? o / L : 0.f;
        else
            store_out<T>(out_row + e, L > 0.f ? o / L : 0.f);
    }
    if (pc.complete && !(fold && warp == 0)) return false;
    if (lane < G) {
        float M = neg_inf();
        for (int w = 0; w < 4; ++w) M = fmaxf(M, sm_m[w * gstride + lane]);
        const float base = (M == neg_inf()) ? 0.f : M;
        float L = 0.f;
        for (int w = 0; w < 4; ++w) {
            const float mw = sm_m[w * gstride + lane];
            L += (mw == neg_inf()) ? 0.f : ex2(mw - base) * sm_l[w * gstride + lane];
        }
        if (pc.complete) {
            a.fold_lse[row0 + lane] = L > 0.f ? M + log2f(L) : neg_inf();
        } else {
            slice[S + lane] = M;
            slice[S + G + lane] = L;
        }
    }
    return !pc.complete;
}

// Loads of one piece for one lane: the lane's NPER accumulator elements and
// the maxima / sums of the (at most NG) heads they belong to.
template <int NPER, int NG>
struct PieceVals {
    float m[NG], l[NG], o[NPER];
};

template <int NPER, int NG>
__device__ __forceinline__ void load_piece(PieceVals<NPER, NG>& v, const float* p, bool live, int S, int G,
                                           int g_first, int ng, int lane) {
#pragma unroll
    for (int k = 0; k < NG; ++k) {
        const bool ok = live && k < ng;
        v.m[k] = ok ? __ldcg(p + S + g_first + k) : neg_inf();
        v.l[k] = ok ? __ldcg(p + S + G + g_first + k) : 0.f;
    }
#pragma unroll
    for (int j = 0; j < NPER; ++j) {
        const int e = lane + 32 * j;
        v.o[j] = (live && e < S) ? __ldcg(p + e) : 0.f;
    }
}

// Merge every piece of this warp's slice of a cut segment and write the
// output row. This runs at the tail of the kernel while other CTAs still
// stream, when a load round trip costs microseconds, so the loop is
// software-pipelined: the loads of the next two pieces are in flight while
// the current two are combined (online log-sum-exp, per head).
template <typename T, int D, int NPER, int NG>
__device__ void merge_slice(const Piece& pc, int G, const DecodeArgs& a, const CostSplit& sp, int warp, int lane,
                            long long c0, int slot0, int npieces, bool fold) {
    const int S = G * D / 4;
    const int e0 = warp * S;
    const int g_first = e0 / D;
    const int ng = (e0 + S - 1) / D - g_first + 1;  // heads of the slice, <= NG
    int kj[NPER];                                   // head slot of each of the lane's elements
#pragma unroll
    for (int j = 0; j < NPER; ++j) kj[j] = (e0 + lane + 32 * j) / D - g_first;
    float M[NG], L[NG], O[NPER];
#pragma unroll
    for (int k = 0; k < NG; ++k) {
        M[k] = neg_inf();
        L[k] = 0.f;
    }
#pragma unroll
    for (int j = 0; j < NPER; ++j) O[j] = 0.f;
    auto ptr = [&](int p) {
        return piece_slice(a.partials, sp.piece_cta(c0, p), p == 0 ? slot0 : 0, warp, S, G);
    };
    PieceVals<NPER, NG> cur[2], nxt[2];
#pragma unroll
    for (int u = 0; u < 2; ++u) load_piece(cur[u], u < npieces ? ptr(u) : a.partials, u < npieces, S, G, g_first, ng, lane);
    for (int p0 = 0; p0 < npieces; p0 += 2) {
#pragma unroll
        for (int u = 0; u < 2; ++u) {
            const int p = p0 + 2 + u;
            load_piece(nxt[u], p < npieces ? ptr(p) : a.partials, p < npieces, S, G, g_first, ng, lane);
        }
#pragma unroll
        for (int u = 0; u < 2; ++u) {
            float sc[NG], w[NG];
#pragma unroll
            for (int k = 0; k < NG; ++k) {
                const float Mn = fmaxf(M[k], cur[u].m[k]);
                const float base = (Mn == neg_inf()) ? 0.f : Mn;
                sc[k] = (M[k] == neg_inf()) ? 0.f : ex2(M[k] - base);
                w[k] = (cur[u].m[k] == neg_inf()) ? 0.f : ex2(cur[u].m[k] - base);
                L[k] = L[k] * sc[k] + w[k] * cur[u].l[k];
                M[k] = Mn;
            }
#pragma unroll
            for (int j = 0; j < NPER; ++j) {
                float scj = 0.f, wj = 0.f;
#pragma unroll
                for (int k = 0; k < NG; ++k) {
                    scj = kj[j] == k ? sc[k] : scj;
                    wj = kj[j] == k ? w[k] : wj;
                }
                O[j] = O[j] * scj + wj * cur[u].o[j];
            }
        }
#pragma unroll
        for (int u = 0; u < 2; ++u) cur[u] = nxt[u];
    }
    const long long row0 = static_cast<long long>(pc.seq) * a.q_heads + pc.head * G;
    T* out_row = static_cast<T*>(a.out) + row0 * D;
#pragma unroll
    for (int j = 0; j < NPER; ++j) {
        const int e = lane + 32 * j;
        if (e >= S) continue;
        float Lj = 0.f;
#pragma unroll
        for (int k = 0; k < NG; ++k) Lj = kj[j] == k ? L[k] : Lj;
        if (fold)
            a.fold_o[row0 * D + e0 + e] = Lj > 0.f ? O[j] / Lj : 0.f;
        else
            store_out<T>(out_row + e0 + e, Lj > 0.f ? O[j] / Lj : 0.f);
    }
    if (fold && lane == 0) {
        // the log-sum-exp of each head whose first element is in this slice
#pragma unroll
        for (int k = 0; k < NG; ++k) {
            const int g = g_first + k;
            if (k < ng && g * D >= e0) a.fold_lse[row0 + g] = L[k] > 0.f ? M[k] + log2f(L[k]) : neg_inf();
        }
    }
}

// After the CTA's last piece: fence this warp's piece writes once, then
// announce the (at most two) cut pieces of the range -- the counter updates
// of both go out together. A warp whose update completes a segment's count
// merges that segment's slice and puts the counter back to zero for the
// next call.
template <typename T, int D, int NPER, int NG>
__device__ void signal_pending(const Piece* pending, int npending, int G, const DecodeArgs& a, const int32_t* s_pre,
                               const int32_t* s_cost, int warp, int lane, const int32_t* s_boff) {
    if (npending == 0) return;
    __threadfence();
    __syncwarp();
    CostSplit sp;  // rebuilt from shared memory: nothing of it stays live through the stream
    sp.init(s_pre, s_cost, a.batch, a.kv_heads, seg_max_unit(a), a.num_ctas);
    long long c0s[2];
    int nps[2];
    int* counters[2];
    int old[2] = {0, 0};
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        if (i >= npending) break;
        const Piece& pc = pending[i];
        c0s[i] = sp.cta_of(pc.seg_start);
        const long long c1 = sp.cta_of(pc.seg_start + pc.seg_len - 1);
        nps[i] = sp.pieces(c0s[i], c1);
        counters[i] = a.counters + (static_cast<long long>(pc.seq) * a.kv_heads + pc.head) * 4 + warp;
        if (lane == 0) old[i] = atomicAdd(counters[i], 1);
    }
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        if (i >= npending) break;
        const int last = __shfl_sync(0xffffffffu, old[i] == nps[i] - 1 ? 1 : 0, 0);
        if (!last) continue;
        __threadfence();
        const Piece& pc = pending[i];
        const int slot0 = (pc.seg_start == sp.start(c0s[i])) ? 0 : 1;
        merge_slice<T, D, NPER, NG>(pc, G, a, sp, warp, lane, c0s[i], slot0, nps[i],
                                    s_boff != nullptr && s_boff[pc.seq] >= 0);
        if (lane == 0) *counters[i] = 0;
    }
}

// Rows of sequences with no tokens are zero; CTA c writes those of the
// sequences i with i % num_ctas == c. A shared-prefix group member with no
// own tokens gets the empty partial instead (zero output, -inf log-sum-exp).
template <typename T>
__device__ void zero_empty_rows(const int32_t* s_len, const int32_t* s_boff, const DecodeArgs& a, int tid,
                                int nthreads) {
    const int row = a.q_heads * a.head_dim;
    for (int i = blockIdx.x; i < a.batch; i += a.num_ctas) {
        if (s_len[i] != 0) continue;
        if (s_boff != nullptr && s_boff[i] >= 0) {
            float* f = a.fold_o + static_cast<long long>(i) * row;
            for (int e = tid; e < row; e += nthreads) f[e] = 0.f;
            for (int e = tid; e < a.q_heads; e += nthreads)
                a.fold_lse[static_cast<long long>(i) * a.q_heads + e] = neg_inf();
            continue;
        }
        T* out = static_cast<T*>(a.out) + static_cast<long long>(i) * row;
        for (int e = tid; e < row; e += nthreads) store_out<T>(out + e, 0.f);
    }
}

// ------------------------------------------------------------------ tensor-core kernel
// Tensor-core kernel configuration. NST is the depth of the shared-memory ring
// (blocks in flight per CTA); the host picks the deepest ring that still fits
// two CTAs per SM.
// Most blocks the producer warp issues in one batch (one per lane).
#ifndef PKV_TC_ISSUE_LANES
#define PKV_TC_ISSUE_LANES 4
#endif
constexpr int kTcIssueLanes = PKV_TC_ISSUE_LANES;
#ifndef PKV_TC_PRODUCERS
#define PKV_TC_PRODUCERS 2
#endif
constexpr int kTcProducers = PKV_TC_PRODUCERS;

template <int D, int NST>
struct Tc {
    static constexpr int kStages = NST;
    static constexpr int kConsumers = 4;
    // Producer warps: 2 = one issues the K boxes of every block and the other
    // the V boxes, each on its own full barrier (consumers wait for the V side
    // just before the P.V product); 1 = one warp issues both on one barrier.
    static constexpr int kProducers = kTcProducers;
    static_assert(kProducers == 1 || kProducers == 2, "one or two producer warps");
    // Unit k goes to stage k % kStages and to consumer warp k % kConsumers. A
    // stage must always meet the same warp: otherwise a warp could wait on a
    // stage two phases ahead of its last use, and a parity wait cannot tell
    // those phases apart.
    static_assert(kStages % kConsumers == 0, "ring depth must be a multiple of the consumer warps");
    static_assert(kStages >= kTcIssueLanes && kTcIssueLanes < 32, "a batch of issued blocks must fit the ring");
    static constexpr int kThreads = (kConsumers + kProducers) * 32;
    static constexpr int kHalves = D / 64;                  // 64-column TMA boxes per row
    static constexpr int kPoolBytes = 16 * D * 2;           // one block, one head, one pool
    static constexpr int kStageBytes = 2 * kPoolBytes;      // K then V
    // shared memory layout (offsets from a 1024-byte aligned base): the ring,
    // then full[producers][NST], empty[NST], the merge barrier, stage flags and the abort
    // flag, then the combine scratch (two buffers of 4 warps x G x (D + 2)
    // floats, alternating between pieces) and the per-sequence prefix sums
    // and lengths.
    static constexpr int kOffBars = kStages * kStageBytes;
    static constexpr int kOffFlags = kOffBars + ((1 + kProducers) * kStages + 2) * 8;
    static constexpr int kOffScratch = ((kOffFlags + kStages * 4 + 4 + 15) / 16) * 16;
    static constexpr size_t scratch_floats(int G) { return 2 * static_cast<size_t>(kConsumers) * G * (D + 2); }
    static size_t smem_bytes(int G, int batch) {
        return 1024 + kOffScratch + scratch_floats(G) * 4 + 3 * static_cast<size_t>(batch) * 4;
    }
};

template <int D, int NST>
__global__ void __launch_bounds__(Tc<D, NST>::kThreads, 2)
    decode_tc_kernel(const DecodeArgs a, const __grid_constant__ CUtensorMap tmK,
                     const __grid_constant__ CUtensorMap tmV) {
    using C = Tc<D, NST>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::kOffBars);  // [producers][stages]: K side, V side
    uint64_t* empty = full + C::kProducers * C::kStages;
    uint64_t* merge_bar = empty + C::kStages;  // all four warps published their piece state
    int* stage_ok = reinterpret_cast<int*>(smem + C::kOffFlags);
    volatile int* abort_flag = stage_ok + C::kStages;
    const int G = a.group;
    float* scratch = reinterpret_cast<float*>(smem + C::kOffScratch);   // 2 x {[4][G][D], [4][G], [4][G]}
    const int buf_floats = C::kConsumers * G * (D + 2);
    int32_t* s_pre = reinterpret_cast<int32_t*>(scratch + 2 * buf_floats);
    int32_t* s_len = s_pre + a.batch;
    int32_t* s_cost = s_len + a.batch;
    int32_t* s_boff = a.prefix_group != nullptr ? s_cost + a.batch : nullptr;  // shared-prefix mode only

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    if (threadIdx.x == 0) PKV_STAMP(a, blockIdx.x, 0);
#ifdef PKV_TRACE
    if (threadIdx.x == 0) reinterpret_cast<unsigned long long*>(a.trace)[blockIdx.x * 8 + 6] = sm_id();
#endif

    if (threadIdx.x == 0) {
        for (int s = 0; s < C::kStages; ++s) {
            for (int p = 0; p < C::kProducers; ++p) mbar_init(&full[p * C::kStages + s], 1);
            mbar_init(&empty[s], 1);
        }
        mbar_init(merge_bar, C::kConsumers);
        *abort_flag = 0;
        fence_barrier_init();
    }
    if (threadIdx.x == 32) {
        tma_prefetch_desc(&tmK);
        tma_prefetch_desc(&tmV);
    }
    // Everything above touches no input; from here on the previous kernel in
    // the stream (typically the append) must be complete.
    grid_dependency_wait();
    allow_dependents();
    build_prefix(s_pre, s_len, s_cost, s_boff, a);  // contains __syncthreads
    if (threadIdx.x == 0) PKV_STAMP(a, blockIdx.x, 1);

    const long long cta = blockIdx.x;
    long long ua, ub;
    {
        CostSplit sp;
        sp.init(s_pre, s_cost, a.batch, a.kv_heads, seg_max_unit(a), a.num_ctas);
        ua = sp.start(cta);
        ub = sp.start(cta + 1);
    }

    if (warp >= C::kConsumers) {
        // ------------------------------------------------ producer warps
        // K/V blocks are read once per call: stream them with evict-first so
        // the block tables, q and the merge pieces stay in L2. With two
        // producers both walk the same blocks; side 0 issues K, side 1 V.
        const uint64_t kv_policy = l2_evict_first_policy();
        if (a.test_stall) return;  // test hook: nothing is ever issued, so every consumer wait runs out
        const int side = warp - C::kConsumers;
        uint64_t* fulls = full + side * C::kStages;
        constexpr int kTx = C::kProducers == 2 ? C::kPoolBytes : C::kStageBytes;
        Walker wk;
        wk.init(s_pre, a.batch, a.kv_heads, ua, ub);
        long long k = 0;
        Piece pc;
        bool ok = true;
        while (ok && wk.next(pc)) {
            const int boff = s_boff != nullptr ? max(s_boff[pc.seq], 0) : 0;
            const int32_t* trow = a.tables + static_cast<long long>(pc.seq) * a.max_blocks + boff + pc.blk_from;
            const int cnt_piece = pc.blk_to - pc.blk_from;
            int cur = lane < cnt_piece ? __ldg(trow + lane) : 0;
            for (int b0 = 0; ok && b0 < cnt_piece; b0 += 32) {
                const int nidx = b0 + 32 + lane;
                const int nxt = nidx < cnt_piece ? __ldg(trow + nidx) : 0;
                const int cnt = min(32, cnt_piece - b0);
                // In order, in batches: lane i probes (without blocking) the
                // stage of block e0 + i; the run of free stages from the first
                // is issued at once, one block per lane with the same
                // instructions (a TMA instruction costs the warp about the
                // same for one lane as for several). Only when the first
                // stage is busy does the warp wait (bounded), for that one.
                for (int e0 = 0; e0 < cnt;) {
                    const int e = e0 + lane;
                    const long long kk = k + lane;
                    const int s = static_cast<int>(kk % C::kStages);
                    const uint32_t par = static_cast<uint32_t>((kk / C::kStages) & 1) ^ 1u;
                    const bool probe = lane < kTcIssueLanes && e < cnt && mbar_test_wait(&empty[s], par);
                    int n = __ffs(~__ballot_sync(0xffffffffu, probe)) - 1;
                    if (n == 0) {
                        bool waited = true;
                        if (lane == 0) waited = mbar_wait(&empty[s], par, a.status, abort_flag);
                        if (!__shfl_sync(0xffffffffu, waited, 0)) {  // nothing of this batch was issued
                            ok = false;
                            break;
                        }
                        n = 1;
                    }
                    const int bid = __shfl_sync(0xffffffffu, cur, e & 31);
                    const bool mine = lane < n;
                    const bool load = mine && bid >= 0 && bid < a.num_blocks;
                    if (mine) {
                        stage_ok[s] = load ? 1 : 0;  // both sides write the same flag
                        if (load) {
                            mbar_arrive_expect_tx(&fulls[s], kTx);
                        } else {
                            if (side == 0) atomicOr(a.status, PKV_DEVERR_RANGE);
                            mbar_arrive(&fulls[s]);
                        }
                    }
                    if (load) {
                        uint8_t* st = smem + s * C::kStageBytes;
                        const int y = (bid * a.kv_heads + pc.head) * 16;
                        if (C::kProducers == 1 || side == 0) {
#pragma unroll
                            for (int hf = 0; hf < C::kHalves; ++hf)
                                tma_load_2d(st + hf * 2048, &tmK, hf * 64, y, &fulls[s], kv_policy);
                        }
                        if (C::kProducers == 1 || side == 1) {
#pragma unroll
                            for (int hf = 0; hf < C::kHalves; ++hf)
                                tma_load_2d(st + C::kPoolBytes + hf * 2048, &tmV, hf * 64, y, &fulls[s], kv_policy);
                        }
                        if (kk == 0 && side == 0) PKV_STAMP(a, blockIdx.x, 2);
                    }
                    k += n;
                    e0 += n;
                }
                cur = nxt;
            }
        }
        // After an abort, wait (bounded) for this warp's copies still in
        // flight into the ring before the CTA may exit.
        if (!ok && lane == 0) {
            const long long first = k > C::kStages ? k - C::kStages : 0;
            for (long long u = first; u < k; ++u)
                mbar_wait(&fulls[u % C::kStages], static_cast<uint32_t>((u / C::kStages) & 1), a.status, nullptr);
        }
        return;
    }

    // ---------------------------------------------------- consumer warps
    const int gid = lane >> 2;  // fragment row group
    const int tig = lane & 3;   // thread in group
    const float scale_log2 = a.scale * kLog2e;
    const __nv_bfloat16* q = static_cast<const __nv_bfloat16*>(a.q);

    // ldmatrix lane addressing (see the header comment): the 8x8 matrix a
    // lane addresses is q8 = lane / 8, its row r8 = lane % 8.
    const int q8 = lane >> 3, r8 = lane & 7;
    const int k_row = r8 + 8 * (q8 & 1);      // K: token row of this lane's address
    const int k_chunk = q8 >> 1;              // K: +0 / +1 16-byte chunk within a k-step
    const int v_row = r8 + 8 * (q8 >> 1);     // V: token row
    const int v_chunk = q8 & 1;               // V: +0 / +1 chunk within an m-tile

    zero_empty_rows<__nv_bfloat16>(s_len, s_boff, a, threadIdx.x, C::kConsumers * 32);
    Walker wk;
    wk.init(s_pre, a.batch, a.kv_heads, ua, ub);
    long long k = 0;
    int piece_idx = 0;
    Piece pc;
    Piece pending[2];  // cut pieces of this range: only its first and its last can be cut
    int npending = 0;
    while (wk.next(pc)) {
        // Q^T fragments: B operand of S^T = K Q^T; column n = query head gid.
        uint32_t qf[D / 16][2];
        {
            const bool live = gid < G;
            const __nv_bfloat16* qrow =
                q + (static_cast<long long>(pc.seq) * a.q_heads + pc.head * G + (live ? gid : 0)) * D;
            const uint32_t* q32 = reinterpret_cast<const uint32_t*>(qrow);
#pragma unroll
            for (int j = 0; j < D / 16; ++j) {
                qf[j][0] = live ? __ldg(q32 + (16 * j + 2 * tig) / 2) : 0u;
                qf[j][1] = live ? __ldg(q32 + (16 * j + 2 * tig + 8) / 2) : 0u;
            }
        }
        float m0 = neg_inf(), m1 = neg_inf(), l0 = 0.f, l1 = 0.f;
        float o[D / 16][4];
#pragma unroll
        for (int i = 0; i < D / 16; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
        const int n_ctx = s_len[pc.seq];

        for (int blk = pc.blk_from; blk < pc.blk_to; ++blk, ++k) {
            if (static_cast<int>(k & (C::kConsumers - 1)) != warp) continue;
            const int s = static_cast<int>(k % C::kStages);
            const uint32_t par = static_cast<uint32_t>((k / C::kStages) & 1);
            const unsigned long long wlim = a.test_stall ? kTestWaitLimitNs : kWaitLimitNs;
            if (!mbar_wait(&full[s], par, a.status, abort_flag, wlim)) return;
            if (k == 0 && lane == 0) PKV_STAMP(a, blockIdx.x, 3);
            const int valid = min(16, n_ctx - blk * 16);
            const bool use = stage_ok[s];
            if (use) {
                const uint32_t kbase = smem_u32(smem + s * C::kStageBytes);
                const uint32_t vbase = kbase + C::kPoolBytes;
                // ---- S^T = K Q^T, even and odd k-steps on two accumulators
                // (two independent MMA chains of D/32 instead of one of D/16)
                float sa[4] = {0.f, 0.f, 0.f, 0.f}, sb[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                for (int j = 0; j < D / 16; ++j) {
                    const int gc = 2 * j + k_chunk;
                    const uint32_t addr = kbase + (gc >> 3) * 2048 + k_row * 128 + (((gc & 7) ^ r8) << 4);
                    uint32_t a0, a1, a2, a3;
                    ldmatrix_x4(addr, a0, a1, a2, a3);
                    if (j & 1)
                        mma_bf16_16816(sb, a0, a1, a2, a3, qf[j][0], qf[j][1]);
                    else
                        mma_bf16_16816(sa, a0, a1, a2, a3, qf[j][0], qf[j][1]);
                }
                // sacc: [0] (t=gid, g=2tig) [1] (t=gid, g=2tig+1) [2] (t=gid+8, g=2tig) [3] (t=gid+8, g=2tig+1)
                const float x0 = gid < valid ? (sa[0] + sb[0]) * scale_log2 : neg_inf();
                const float x1 = gid < valid ? (sa[1] + sb[1]) * scale_log2 : neg_inf();
                const float x2 = gid + 8 < valid ? (sa[2] + sb[2]) * scale_log2 : neg_inf();
                const float x3 = gid + 8 < valid ? (sa[3] + sb[3]) * scale_log2 : neg_inf();
                // Lazy rescale: the running maximum m only has to bound the
                // scores closely enough that 2^(x - m) cannot overflow; the
                // output is exact for any m, since O and l use the same one.
                // So the cross-lane maximum and the rescale of O run only when
                // some score exceeds m by more than 8 (a factor 256); most
                // blocks after the first skip them.
                float mx0 = fmaxf(x0, x2), mx1 = fmaxf(x1, x3);
                if (__any_sync(0xffffffffu, mx0 > m0 + 8.f || mx1 > m1 + 8.f)) {
#pragma unroll
                    for (int off = 4; off < 32; off <<= 1) {
                        mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, off));
                        mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, off));
                    }
                    const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
                    const float nb0 = mn0 == neg_inf() ? 0.f : mn0;
                    const float nb1 = mn1 == neg_inf() ? 0.f : mn1;
                    const float al0 = ex2(m0 - nb0), al1 = ex2(m1 - nb1);
                    l0 *= al0;
                    l1 *= al1;
#pragma unroll
                    for (int i = 0; i < D / 16; ++i) {
                        o[i][0] *= al0;
                        o[i][1] *= al1;
                        o[i][2] *= al0;
                        o[i][3] *= al1;
                    }
                    m0 = mn0;
                    m1 = mn1;
                }
                const float b0 = m0 == neg_inf() ? 0.f : m0;
                const float b1 = m1 == neg_inf() ? 0.f : m1;
                const float p0 = ex2(x0 - b0), p1 = ex2(x1 - b1), p2 = ex2(x2 - b0), p3 = ex2(x3 - b1);
                l0 += p0 + p2;
                l1 += p1 + p3;
                // ---- P^T as bf16 hi + lo, moved into the B-operand layout
                const uint32_t h01 = pack_bf16x2(p0, p1), h23 = pack_bf16x2(p2, p3);
                const uint32_t l01 = pack_bf16x2(p0 - bf16lo_to_f32(h01), p1 - bf16hi_to_f32(h01));
                const uint32_t l23 = pack_bf16x2(p2 - bf16lo_to_f32(h23), p3 - bf16hi_to_f32(h23));
                const uint32_t bh0 = movmatrix_trans(h01), bh1 = movmatrix_trans(h23);
                const uint32_t bl0 = movmatrix_trans(l01), bl1 = movmatrix_trans(l23);
                // ---- O^T += V^T P^T; rows past the context are zeroed (they may hold anything)
                if (C::kProducers == 2 && !mbar_wait(&full[C::kStages + s], par, a.status, abort_flag, wlim)) return;
                uint32_t mlo = 0xffffffffu, mhi = 0xffffffffu;
                if (valid < 16) {
                    mlo = (2 * tig < valid ? 0x0000ffffu : 0u) | (2 * tig + 1 < valid ? 0xffff0000u : 0u);
                    mhi = (2 * tig + 8 < valid ? 0x0000ffffu : 0u) | (2 * tig + 9 < valid ? 0xffff0000u : 0u);
                }
#pragma unroll
                for (int i = 0; i < D / 16; ++i) {
                    const int gc = 2 * i + v_chunk;
                    const uint32_t addr = vbase + (gc >> 3) * 2048 + v_row * 128 + (((gc & 7) ^ r8) << 4);
                    uint32_t a0, a1, a2, a3;
                    ldmatrix_x4_trans(addr, a0, a1, a2, a3);
                    a0 &= mlo;
                    a1 &= mlo;
                    a2 &= mhi;
                    a3 &= mhi;
                    mma_bf16_16816(o[i], a0, a1, a2, a3, bh0, bh1);
                    mma_bf16_16816(o[i], a0, a1, a2, a3, bl0, bl1);
                }
            }
            // a stage is handed back only after both of its sides have landed
            if (C::kProducers == 2 && !use && !mbar_wait(&full[C::kStages + s], par, a.status, abort_flag, wlim))
                return;
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[s]);
        }

        if (warp == 0 && lane == 0 && wk.u >= wk.end) PKV_STAMP(a, blockIdx.x, 4);
        // ---- combine the four warps' states for this piece
#pragma unroll
        for (int off = 4; off < 32; off <<= 1) {
            l0 += __shfl_xor_sync(0xffffffffu, l0, off);
            l1 += __shfl_xor_sync(0xffffffffu, l1, off);
        }
        // Alternate two scratch buffers: a warp can only be one piece ahead of
        // the others (the merge barrier below), so it never overwrites a
        // buffer that another warp still reads.
        float* sm_o = scratch + (piece_idx & 1) * buf_floats;   // [4][G][D]
        float* sm_m = sm_o + C::kConsumers * G * D;             // [4][G]
        float* sm_l = sm_m + C::kConsumers * G;                 // [4][G]
        const int g0 = 2 * tig, g1 = 2 * tig + 1;
#pragma unroll
        for (int i = 0; i < D / 16; ++i) {
            const int d = 16 * i + gid;
            if (g0 < G) {
                sm_o[(warp * G + g0) * D + d] = o[i][0];
                sm_o[(warp * G + g0) * D + d + 8] = o[i][2];
            }
            if (g1 < G) {
                sm_o[(warp * G + g1) * D + d] = o[i][1];
                sm_o[(warp * G + g1) * D + d + 8] = o[i][3];
            }
        }
        if (gid == 0) {
            if (g0 < G) {
                sm_m[warp * G + g0] = m0;
                sm_l[warp * G + g0] = l0;
            }
            if (g1 < G) {
                sm_m[warp * G + g1] = m1;
                sm_l[warp * G + g1] = l1;
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(merge_bar);
        if (!mbar_wait(merge_bar, static_cast<uint32_t>(piece_idx & 1), a.status, abort_flag)) return;
        if (write_piece<__nv_bfloat16, D>(sm_o, sm_m, sm_l, G, G, pc, a, cta, warp, lane,
                                          s_boff != nullptr && s_boff[pc.seq] >= 0))
            pending[npending++] = pc;
        ++piece_idx;
    }
    // G <= 8: a warp's slice is G*D/4 <= 2*D elements, at most D/16 per lane
    // and at most three heads
    signal_pending<__nv_bfloat16, D, D / 16, 3>(pending, npending, G, a, s_pre, s_cost, warp, lane, s_boff);
    if (warp == 0 && lane == 0) PKV_STAMP(a, blockIdx.x, 5);
}

// ------------------------------------------------------------------ CUDA-core kernel
template <typename T, int D, int GMAX>
struct Cc {
    static constexpr int kWarps = 4;
    static constexpr int kThreads = kWarps * 32;
    static constexpr int kPer = D / 32;  // head-dim elements per lane
};

template <typename T, int D, int GMAX>
__global__ void __launch_bounds__(128) decode_cc_kernel(const DecodeArgs a) {
    using C = Cc<T, D, GMAX>;
    extern __shared__ float smem_f[];
    float* sm_o = smem_f;                                        // [warps][GMAX][D]
    float* sm_m = sm_o + C::kWarps * GMAX * D;                   // [warps][GMAX]
    float* sm_l = sm_m + C::kWarps * GMAX;
    int32_t* s_pre = reinterpret_cast<int32_t*>(sm_l + C::kWarps * GMAX);
    int32_t* s_len = s_pre + a.batch;
    int32_t* s_cost = s_len + a.batch;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    grid_dependency_wait();
    allow_dependents();
    build_prefix(s_pre, s_len, s_cost, nullptr, a);

    const long long cta = blockIdx.x;
    long long ua, ub;
    {
        CostSplit sp;
        sp.init(s_pre, s_cost, a.batch, a.kv_heads, seg_max_unit(a), a.num_ctas);
        ua = sp.start(cta);
        ub = sp.start(cta + 1);
    }
    const int G = a.group;
    const float scale_log2 = a.scale * kLog2e;
    const T* q = static_cast<const T*>(a.q);
    const T* kc = static_cast<const T*>(a.k_cache);
    const T* vc = static_cast<const T*>(a.v_cache);

    zero_empty_rows<T>(s_len, nullptr, a, threadIdx.x, C::kThreads);
    Walker wk;
    wk.init(s_pre, a.batch, a.kv_heads, ua, ub);
    long long k = 0;
    Piece pc;
    Piece pending[2];
    int npending = 0;
    while (wk.next(pc)) {
        float qr[GMAX][C::kPer];
#pragma unroll
        for (int g = 0; g < GMAX; ++g)
#pragma unroll
            for (int e = 0; e < C::kPer; ++e)
                qr[g][e] = g < G ? load_f32<T>(q + (static_cast<long long>(pc.seq) * a.q_heads + pc.head * G + g) * D +
                                               lane + 32 * e)
                                 : 0.f;
        float m[GMAX], l[GMAX], o[GMAX][C::kPer];
#pragma unroll
        for (int g = 0; g < GMAX; ++g) {
            m[g] = neg_inf();
            l[g] = 0.f;
#pragma unroll
            for (int e = 0; e < C::kPer; ++e) o[g][e] = 0.f;
        }
        const int n_ctx = s_len[pc.seq];
        const int32_t* trow = a.tables + static_cast<long long>(pc.seq) * a.max_blocks;
        for (int blk = pc.blk_from; blk < pc.blk_to; ++blk, ++k) {
            if (static_cast<int>(k & (C::kWarps - 1)) != warp) continue;
            const int bid = __ldg(trow + blk);
            if (bid < 0 || bid >= a.num_blocks) {
                if (lane == 0) atomicOr(a.status, PKV_DEVERR_RANGE);
                continue;
            }
            const int valid = min(16, n_ctx - blk * 16);
            const long long row0 = (static_cast<long long>(bid) * a.kv_heads + pc.head) * 16;
            for (int t = 0; t < valid; ++t) {
                const T* krow = kc + (row0 + t) * D;
                const T* vrow = vc + (row0 + t) * D;
                float kv[C::kPer], vv[C::kPer];
#pragma unroll
                for (int e = 0; e < C::kPer; ++e) {
                    kv[e] = load_f32<T>(krow + lane + 32 * e);
                    vv[e] = load_f32<T>(vrow + lane + 32 * e);
                }
#pragma unroll
                for (int g = 0; g < GMAX; ++g) {
                    if (g >= G) break;
                    float dot = 0.f;
#pragma unroll
                    for (int e = 0; e < C::kPer; ++e) dot = fmaf(qr[g][e], kv[e], dot);
#pragma unroll
                    for (int off = 16; off > 0; off >>= 1) dot += __shfl_xor_sync(0xffffffffu, dot, off);
                    const float x = dot * scale_log2;
                    const float mn = fmaxf(m[g], x);
                    const float al = ex2(m[g] - mn);
                    const float p = ex2(x - mn);
                    l[g] = l[g] * al + p;
#pragma unroll
                    for (int e = 0; e < C::kPer; ++e) o[g][e] = fmaf(o[g][e], al, p * vv[e]);
                    m[g] = mn;
                }
            }
        }
        // publish each warp's state, then finish the piece slice by slice
        __syncthreads();
#pragma unroll
        for (int g = 0; g < GMAX; ++g) {
            if (g >= G) break;
#pragma unroll
            for (int e = 0; e < C::kPer; ++e) sm_o[(warp * GMAX + g) * D + lane + 32 * e] = o[g][e];
            if (lane == 0) {
                sm_m[warp * GMAX + g] = m[g];
                sm_l[warp * GMAX + g] = l[g];
            }
        }
        __syncthreads();
        if (write_piece<T, D>(sm_o, sm_m, sm_l, GMAX, G, pc, a, cta, warp, lane, false)) pending[npending++] = pc;
        __syncthreads();
    }
    signal_pending<T, D, GMAX * D / 128, GMAX / 4 + 1>(pending, npending, G, a, s_pre, s_cost, warp, lane, nullptr);
}

// ------------------------------------------------------------------ host side
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

// 2-D view of a pool: rows of head_dim bf16 (one token of one head), boxes of
// 16 rows x 64 columns with the 128-byte swizzle.
bool encode_pool_map(CUtensorMap* map, const void* pool, int64_t rows, int head_dim) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(head_dim), static_cast<cuuint64_t>(rows)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(head_dim) * 2};
    const cuuint32_t box[2] = {64, 16};
    const cuuint32_t estr[2] = {1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(pool), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <typename K>
int occupancy(K kernel, int threads, size_t smem) {
    int dev = 0;
    cudaGetDevice(&dev);
    if (smem > 48 * 1024) cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kernel, threads, smem) != cudaSuccess) n = 0;
    return n;
}

struct OccKey {
    int dev, kernel, variant;
    size_t smem;
};

int cached_occupancy(int kernel_id, int variant, size_t smem, int threads, const void* fnptr,
                     int (*query)(const void*, int, size_t)) {
    static std::mutex mu;
    static OccKey keys[64];
    static int vals[64];
    static int used = 0;
    int dev = 0;
    cudaGetDevice(&dev);
    std::lock_guard<std::mutex> lock(mu);
    for (int i = 0; i < used; ++i)
        if (keys[i].dev == dev && keys[i].kernel == kernel_id && keys[i].variant == variant && keys[i].smem == smem)
            return vals[i];
    const int n = query(fnptr, threads, smem);
    if (used < 64) {
        keys[used] = OccKey{dev, kernel_id, variant, smem};
        vals[used] = n;
        ++used;
    }
    return n;
}

template <int D, int NST>
int tc_query(const void*, int threads, size_t smem) {
    return occupancy(decode_tc_kernel<D, NST>, threads, smem);
}
template <typename T, int D, int GMAX>
int cc_query(const void*, int threads, size_t smem) {
    return occupancy(decode_cc_kernel<T, D, GMAX>, threads, smem);
}

template <typename T, int D, int GMAX>
size_t cc_smem(int batch) {
    return static_cast<size_t>(4) * GMAX * D * 4 + 2 * 4 * GMAX * 4 + 3 * static_cast<size_t>(batch) * 4;
}

int variant_of(int dtype, int D, int gmax) { return (dtype == PKV_BF16 ? 4 : 0) + (D == 128 ? 2 : 0) + (gmax == 16 ? 1 : 0); }

template <typename T, int D, int GMAX>
cudaError_t run_cc(const DecodeArgs& a, int grid, size_t smem, cudaStream_t s) {
    if (smem > 48 * 1024)
        cudaFuncSetAttribute(decode_cc_kernel<T, D, GMAX>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(smem));
    return launch_pdl(decode_cc_kernel<T, D, GMAX>, dim3(grid), dim3(128), smem, s, a);
}

template <int D, int NST>
cudaError_t run_tc(const DecodeArgs& a, int grid, size_t smem, cudaStream_t s) {
    CUtensorMap tmK, tmV;
    const int64_t rows = a.num_blocks * a.kv_heads * 16;
    if (!encode_pool_map(&tmK, a.k_cache, rows, D) || !encode_pool_map(&tmV, a.v_cache, rows, D))
        return cudaErrorInvalidValue;
    cudaFuncSetAttribute(decode_tc_kernel<D, NST>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         static_cast<int>(smem));
    return launch_pdl(decode_tc_kernel<D, NST>, dim3(grid), dim3(Tc<D, NST>::kThreads), smem, s, a, tmK, tmV);
}

}  // namespace

bool make_pool_map(CUtensorMap* map, const void* pool, int64_t rows, int head_dim) {
    return encode_pool_map(map, pool, rows, head_dim);
}

bool make_map_2d(CUtensorMap* map, int dtype, const void* base, uint64_t inner, uint64_t rows, uint64_t row_bytes,
                 uint32_t box_inner, uint32_t box_rows, bool swizzle128, bool l2_promote) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[2] = {inner, rows};
    const cuuint64_t strides[1] = {row_bytes};
    const cuuint32_t box[2] = {box_inner, box_rows};
    const cuuint32_t estr[2] = {1, 1};
    const CUtensorMapDataType t = dtype == PKV_INT8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
    return fn(map, t, 2, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
              swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
              l2_promote ? CU_TENSOR_MAP_L2_PROMOTION_L2_256B : CU_TENSOR_MAP_L2_PROMOTION_NONE,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

WorkspaceLayout decode_workspace_layout(int batch, int kv_heads, int num_ctas, int group, int head_dim) {
    const int chunk = batch < kMaxBatchPerLaunch ? batch : kMaxBatchPerLaunch;
    WorkspaceLayout w;
    w.counters_offset = 256;
    const size_t counters = static_cast<size_t>(chunk) * kv_heads * 4 * sizeof(int);
    w.partials_offset = w.counters_offset + ((counters + 255) / 256) * 256;
    // per CTA: 2 piece slots x 4 warp slices x (G*D/4 values + G maxima + G sums)
    const size_t per_cta = 2 * 4 * (static_cast<size_t>(group) * head_dim / 4 + 2 * group) * sizeof(float);
    w.total = w.partials_offset + static_cast<size_t>(num_ctas) * per_cta;
#ifdef PKV_TRACE
    w.trace_offset = (w.total + 255) / 256 * 256;
    w.total = w.trace_offset + static_cast<size_t>(num_ctas) * 64;
#else
    w.trace_offset = 0;
#endif
    return w;
}

int decode_plan(const pkv_cache_desc& d, int32_t batch, int32_t q_heads, int32_t max_blocks,
                const pkv_decode_opts* opts, DecodePlan* plan, bool prefixed) {
    (void)max_blocks;
    const int G = q_heads / d.num_kv_heads;
    const int want = opts ? opts->kernel : 0;
    const bool tc_ok = d.dtype == PKV_BF16 && G <= 8 && (d.head_dim == 64 || d.head_dim == 128);
    int kernel = want;
    if (kernel == 0) kernel = tc_ok ? 2 : 1;
    if (kernel == 2 && !tc_ok) return PKV_ERR_UNSUPPORTED;
    if (kernel == 1 && G > 16) return PKV_ERR_UNSUPPORTED;
    if (kernel != 1 && kernel != 2) return PKV_ERR_UNSUPPORTED;
    const int chunk = batch < kMaxBatchPerLaunch ? (batch < 1 ? 1 : batch) : kMaxBatchPerLaunch;
    int per_sm = 0;
    size_t smem = 0;
    int stages = 0;
    if (kernel == 2) {
        // 8 stages by default (measured faster than 12 at two CTAs per SM on
        // every workload); 12 on request
        const int want_st = opts ? opts->stages : 0;
        for (int st : {8, 12}) {
            if (want_st && want_st != st) continue;
            size_t sm = prefixed ? static_cast<size_t>(chunk) * 4 : 0;  // per-sequence block offsets
            int n = 0;
            if (d.head_dim == 128) {
                sm += st == 12 ? Tc<128, 12>::smem_bytes(G, chunk) : Tc<128, 8>::smem_bytes(G, chunk);
                n = st == 12 ? cached_occupancy(2, 128 * 100 + st, sm, Tc<128, 12>::kThreads, nullptr, tc_query<128, 12>)
                             : cached_occupancy(2, 128 * 100 + st, sm, Tc<128, 8>::kThreads, nullptr, tc_query<128, 8>);
            } else {
                sm += st == 12 ? Tc<64, 12>::smem_bytes(G, chunk) : Tc<64, 8>::smem_bytes(G, chunk);
                n = st == 12 ? cached_occupancy(2, 64 * 100 + st, sm, Tc<64, 12>::kThreads, nullptr, tc_query<64, 12>)
                             : cached_occupancy(2, 64 * 100 + st, sm, Tc<64, 8>::kThreads, nullptr, tc_query<64, 8>);
            }
            if (want_st == st || (want_st == 0 && st == 8)) {
                stages = st;
                smem = sm;
                per_sm = n;
                break;
            }
        }
        if (stages == 0) return PKV_ERR_UNSUPPORTED;
    } else {
        const int gmax = G <= 8 ? 8 : 16;
        const int v = variant_of(d.dtype, d.head_dim, gmax);
#define PKV_CC_CASE(T, DD, GM)                                                      \
    if (v == variant_of(std::is_same<T, float>::value ? PKV_F32 : PKV_BF16, DD, GM)) { \
        smem = cc_smem<T, DD, GM>(chunk);                                           \
        per_sm = cached_occupancy(1, v, smem, 128, nullptr, cc_query<T, DD, GM>);   \
    }
        PKV_CC_CASE(float, 64, 8)
        PKV_CC_CASE(float, 64, 16)
        PKV_CC_CASE(float, 128, 8)
        PKV_CC_CASE(float, 128, 16)
        PKV_CC_CASE(__nv_bfloat16, 64, 8)
        PKV_CC_CASE(__nv_bfloat16, 64, 16)
        PKV_CC_CASE(__nv_bfloat16, 128, 8)
        PKV_CC_CASE(__nv_bfloat16, 128, 16)
#undef PKV_CC_CASE
    }
    if (per_sm < 1) per_sm = 1;
    plan->kernel = kernel;
    plan->stages = stages;
    plan->smem = smem;
    plan->num_ctas = (opts && opts->num_ctas > 0) ? opts->num_ctas : device_sm_count() * per_sm;
    return PKV_OK;
}

cudaError_t launch_decode(const DecodeArgs& args, const DecodePlan& plan, cudaStream_t s) {
    DecodeArgs a = args;
    a.seg_cost = kSegCost;
    a.seg_cost_below = kSegCostBelow;
    a.seg_min_cost = kSegMinCost;
    cudaError_t err = cudaSuccess;
    const int D = a.head_dim;
    if (plan.kernel == 2) {
        if (D == 128)
            err = plan.stages == 12 ? run_tc<128, 12>(a, plan.num_ctas, plan.smem, s)
                                    : run_tc<128, 8>(a, plan.num_ctas, plan.smem, s);
        else
            err = plan.stages == 12 ? run_tc<64, 12>(a, plan.num_ctas, plan.smem, s)
                                    : run_tc<64, 8>(a, plan.num_ctas, plan.smem, s);
    } else {
        const bool g16 = a.group > 8;
        if (a.dtype == PKV_F32) {
            if (D == 128)
                err = g16 ? run_cc<float, 128, 16>(a, plan.num_ctas, plan.smem, s)
                          : run_cc<float, 128, 8>(a, plan.num_ctas, plan.smem, s);
            else
                err = g16 ? run_cc<float, 64, 16>(a, plan.num_ctas, plan.smem, s)
                          : run_cc<float, 64, 8>(a, plan.num_ctas, plan.smem, s);
        } else {
            if (D == 128)
                err = g16 ? run_cc<__nv_bfloat16, 128, 16>(a, plan.num_ctas, plan.smem, s)
                          : run_cc<__nv_bfloat16, 128, 8>(a, plan.num_ctas, plan.smem, s);
            else
                err = g16 ? run_cc<__nv_bfloat16, 64, 16>(a, plan.num_ctas, plan.smem, s)
                          : run_cc<__nv_bfloat16, 64, 8>(a, plan.num_ctas, plan.smem, s);
        }
    }
    return err;
}

}  // namespace pkv
