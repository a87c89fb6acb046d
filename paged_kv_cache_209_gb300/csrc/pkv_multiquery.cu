// Multi-query paged attention: several causal queries per sequence (the K
// draft tokens a speculative step verifies in one pass, or a short prefill
// chunk) against the sequence's paged context.
//
// Sequence i holds n = context_lens[i] tokens, the last nq of which are this
// step's new tokens; its queries are rows query_start[i] .. query_start[i+1]-1
// of q, and query t attends to tokens 0 .. n - nq + t (release page
// "NeuralOps v1.3.4", Architectural Breakdown 2, single-pass verification of
// the K candidates; notebook section 7: a suffix attends to every cached
// position, causally within itself).
//
// This kernel takes calls with up to 32 query rows per (sequence, KV head)
// (max_query_len * G); more rows (a chunked prefill) run on the tcgen05 tile
// kernel's prefill mode in pkv_prefix.cu.
//
// Work decomposition: the stream-K split of the decode kernel over (sequence,
// KV head, block) units, so K/V is read once per call for all query rows.
// The query rows of one (sequence, KV head) are (query t, query head g),
// row r = t G + g, at most 32, split into row groups of 8. With W = 1, 2 or 4
// row groups (from max_query_len * G), the four consumer warps form 4 / W
// unit lanes of W warps: warp w serves row group w % W and takes the blocks
// k of its CTA's range with k % (4 / W) == w / W, so up to four blocks are in
// flight per CTA whatever the row count:
//     S^T[16 tokens][8 rows] = K[16][D] * Q^T[D][8]        (mma m16n8k16)
//     causal mask per row, base-2 online softmax (lazy rescale)
//     O^T[D][8] += V^T[D][16] * P^T[16][8]                  (P as bf16 hi + lo)
// At the end of a segment piece the unit lanes' states of a row group are
// combined through shared memory by the row group's first warp. A segment cut
// by a CTA range boundary leaves one fp32 piece per CTA and row group; the
// warp that completes a (segment, row group) counter merges them by
// log-sum-exp.
#include <math.h>
#include <mutex>

#include "pkv_device.cuh"
#include "pkv_internal.h"
#include "pkv_schedule.cuh"

namespace pkv {
namespace {

constexpr float kLog2e = 1.4426950408889634f;
constexpr int kMqRows = 32;  // query rows per (sequence, KV head): 4 warps x 8

__device__ __forceinline__ float ninf() { return __int_as_float(0xff800000); }

// Most blocks whose copies the producer warp issues together (one per lane),
// a build-time knob per cache type. A TMA instruction costs the issuing warp
// about a hundred cycles whether one lane or eight issue it, so a producer
// that issued one block at a time could not keep up with 4 KB int8 blocks.
#ifndef PKV_MQ_ISSUE_LANES
#define PKV_MQ_ISSUE_LANES 4
#endif
#ifndef PKV_MQ8_ISSUE_LANES
#define PKV_MQ8_ISSUE_LANES 6
#endif

template <int D, int NST, bool Q8 = false>
struct Mq {
    static constexpr int kIssueLanes = Q8 ? PKV_MQ8_ISSUE_LANES : PKV_MQ_ISSUE_LANES;
    static constexpr int kStages = NST;
    static constexpr int kConsumers = 4;
    // two producer warps: one issues the K side of every block (K rows, or K
    // codes and K scales), the other the V side, each on its own barrier
    static constexpr int kThreads = (kConsumers + 2) * 32;
    static constexpr int kHalves = D / 64;
    static constexpr int kPoolBytes = 16 * D * 2;
    // bf16: K then V (16 rows x D each). int8: K codes [16][D] at 0, V codes
    // [D][16] at 16 D; the (block, head) scale record (16 K scales, then 16 V
    // scales at byte 64) of the stage sits in a ring of its own after the
    // stages, 128 bytes per stage, and comes with the K side. Every TMA
    // destination is 128-byte aligned (a smaller alignment faults); stages
    // are 1024-byte aligned (the K swizzle).
    static constexpr int kStageBytes = Q8 ? 2 * 16 * D : 2 * kPoolBytes;
    static constexpr int kScaleBytes = Q8 ? 128 : 0;
    static constexpr int kVScaleOff = 64;
    static constexpr int kSideBytes = kStageBytes / 2;  // K or V of one stage
    // bytes one side's copies deliver: the K side carries the scale record
    static constexpr int kTxK = Q8 ? kSideBytes + kScaleBytes : kSideBytes;
    static constexpr int kTxV = kSideBytes;
    static constexpr int kOffScales = kStages * kStageBytes;
    static_assert(kStages >= kIssueLanes && kIssueLanes < 32, "a batch of issued blocks must fit the ring");
    static_assert(kOffScales % 1024 == 0 && kScaleBytes % 128 == 0, "TMA destinations must stay 128-byte aligned");
    // shared memory (offsets from a 1024-byte aligned base): the ring,
    // full[2][NST] (K side, V side), empty[NST] and the piece barrier, stage flags and the abort
    // flag, the combine scratch (two buffers of 4 warps x 8 rows x (D + 2)
    // floats, alternating between pieces), then per sequence: block prefix
    // sums and context lengths.
    static constexpr int kOffBars = kOffScales + kStages * kScaleBytes;
    static constexpr int kOffFlags = kOffBars + (3 * kStages + 1) * 8;
    static constexpr int kOffScratch = ((kOffFlags + kStages * 4 + 4 + 15) / 16) * 16;
    static constexpr int kScratchFloats = 2 * kConsumers * 8 * (D + 2);
    static constexpr int kOffSeq = kOffScratch + kScratchFloats * 4;
    static size_t smem_bytes(int batch) { return 1024 + kOffSeq + 2 * static_cast<size_t>(batch) * 4; }
};

// Workspace slice of one piece: CTA `cta`, slot (0: the piece that opens the
// range, 1: the one that closes it), warp: 8 rows x D accumulators, 8 maxima,
// 8 sums.
__device__ __forceinline__ float* mq_slice(float* partials, long long cta, int slot, int warp, int D) {
    return partials + ((cta * 2 + slot) * 4 + warp) * static_cast<long long>(8 * (D + 2));
}

// Merge every piece of warp `warp`'s rows of a cut segment and write the
// output rows. Lane = 4 * row + quarter: row lane / 4 of the warp's 8, head-dim
// quarter lane % 4.
template <int D>
__device__ void mq_merge(const Piece& pc, const MqArgs& a, long long U, int warp, int lane, long long c0, int slot0,
                         int npieces, int rows, int q0) {
    const long long C = a.num_ctas;
    const int r8 = lane >> 2;
    const int rr = warp * 8 + r8;
    const int d0 = (lane & 3) * (D / 4);
    float M = ninf(), L = 0.f;
    float O[D / 4];
#pragma unroll
    for (int k = 0; k < D / 4; ++k) O[k] = 0.f;
    for (int p = 0; p < npieces; ++p) {
        const float* sl = mq_slice(a.partials, piece_cta(pc.seg_start, c0, p, U, C), p == 0 ? slot0 : 0, warp, D);
        const float mp = __ldcg(sl + 8 * D + r8);
        const float lp = __ldcg(sl + 8 * D + 8 + r8);
        const float Mn = fmaxf(M, mp);
        const float base = Mn == ninf() ? 0.f : Mn;
        const float sc = M == ninf() ? 0.f : ex2(M - base);
        const float w = mp == ninf() ? 0.f : ex2(mp - base);
        L = L * sc + w * lp;
        M = Mn;
#pragma unroll
        for (int k = 0; k < D / 4; k += 4) {
            const float4 v = __ldcg(reinterpret_cast<const float4*>(sl + r8 * D + d0 + k));
            O[k] = O[k] * sc + w * v.x;
            O[k + 1] = O[k + 1] * sc + w * v.y;
            O[k + 2] = O[k + 2] * sc + w * v.z;
            O[k + 3] = O[k + 3] * sc + w * v.w;
        }
    }
    if (rr >= rows) return;
    const int G = a.group;
    const int t = rr / G;
    __nv_bfloat16* orow = static_cast<__nv_bfloat16*>(a.out) +
                          (static_cast<long long>(q0 + t) * a.q_heads + pc.head * G + (rr - t * G)) * D;
    const float inv = L > 0.f ? 1.f / L : 0.f;
#pragma unroll
    for (int k = 0; k < D / 4; k += 2)
        *reinterpret_cast<uint32_t*>(orow + d0 + k) = pack_bf16x2(O[k] * inv, O[k + 1] * inv);
}

// Token order of the int8 path: row m of S^T = K Q^T holds token sigma(m), so
// that the four codes a lane reads from a V coordinate row (tokens 4 tig ..
// 4 tig + 3) are the P^T k-slots 2 tig, 2 tig + 1, 2 tig + 8, 2 tig + 9 it
// meets in the PV product.
__device__ __forceinline__ int sigma(int m) {
    return m < 8 ? 4 * (m >> 1) + (m & 1) : 4 * ((m - 8) >> 1) + 2 + (m & 1);
}

// Four int8 codes c (one 32-bit word, lowest byte first) -> two f16x2 pairs
// (bytes 0, 1) and (bytes 2, 3) holding c + 1152 exactly: the code offset by
// 128 becomes the low mantissa byte of the f16 1024 + u. Used for K, whose
// scores are formed afresh for every block: S = S' - 1152 * (query sum), one
// subtraction per score instead of one per code; the rounding of S' stays
// within a few fp32 steps of 1152 * sum |q|, below 2^-16 of the largest
// score the row could reach.
constexpr float kCodeBias = 1152.f;
// Largest V scale for which P' = P * s_v (P <= 2^8 under the lazy rescale)
// stays below the f16 maximum 65504 (255 * 256 = 65280).
constexpr float kVScaleF16Safe = 255.f;

// Smallest k >= 0 with v * 2^-k <= kVScaleF16Safe, for a finite v above it:
// with v = m 2^e (m in [1, 2)), v 2^-(e-7) = 128 m lies in [128, 256), so k is
// e - 7, or e - 6 when 128 m exceeds 255. Halvings of a float are exact.
__device__ __forceinline__ int pow2_shift_to_fit(float v) {
    const uint32_t b = __float_as_uint(v);
    const int e = static_cast<int>((b >> 23) & 0xffu) - 127;
    const float m128 = __uint_as_float((b & 0x007fffffu) | (134u << 23));
    return e - 7 + (m128 > kVScaleF16Safe ? 1 : 0);
}
__device__ __forceinline__ void codes_to_f16x2_biased(uint32_t w, uint32_t& p01, uint32_t& p23) {
    const uint32_t u = w ^ 0x80808080u;
    p01 = __byte_perm(u, 0x64646464u, 0x5140);
    p23 = __byte_perm(u, 0x64646464u, 0x5342);
}

// The same, exact codes c (the bias subtracted in f16). Used for V: the
// output accumulates over the whole context, so a bias there would let the
// accumulator's rounding grow with the context length times 1152.
__device__ __forceinline__ void codes_to_f16x2(uint32_t w, uint32_t& p01, uint32_t& p23) {
    uint32_t h01, h23;
    codes_to_f16x2_biased(w, h01, h23);
    const __half2 bias = __halves2half2(__ushort_as_half(0x6480), __ushort_as_half(0x6480));
    const __half2 r01 = __hsub2(*reinterpret_cast<const __half2*>(&h01), bias);
    const __half2 r23 = __hsub2(*reinterpret_cast<const __half2*>(&h23), bias);
    p01 = *reinterpret_cast<const uint32_t*>(&r01);
    p23 = *reinterpret_cast<const uint32_t*>(&r23);
}

__device__ __forceinline__ float f16x2_sum(uint32_t h) {
    const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&h));
    return f.x + f.y;
}

__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
    const __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<const uint32_t*>(&h);
}

template <int D, int NST, bool Q8>
__global__ void __launch_bounds__(Mq<D, NST, Q8>::kThreads, 2)
    mq_tc_kernel(const MqArgs a, const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                 const __grid_constant__ CUtensorMap tmS) {
    using C = Mq<D, NST, Q8>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::kOffBars);  // K side; full + kStages: V side
    uint64_t* empty = full + 2 * C::kStages;
    uint64_t* piece_bar = empty + C::kStages;  // every consumer warp published its piece state
    int* stage_ok = reinterpret_cast<int*>(smem + C::kOffFlags);
    volatile int* abort_flag = stage_ok + C::kStages;
    float* scratch = reinterpret_cast<float*>(smem + C::kOffScratch);
    int32_t* s_pre = reinterpret_cast<int32_t*>(smem + C::kOffSeq);
    int32_t* s_len = s_pre + a.batch;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int G = a.group;

    if (threadIdx.x == 0) {
        for (int s = 0; s < C::kStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&full[C::kStages + s], 1);
            mbar_init(&empty[s], a.wpu);  // the warps of one unit lane consume a stage
        }
        mbar_init(piece_bar, C::kConsumers);
        *abort_flag = 0;
        fence_barrier_init();
    }
    if (threadIdx.x == 32) {
        tma_prefetch_desc(&tmK);
        tma_prefetch_desc(&tmV);
        if (Q8) tma_prefetch_desc(&tmS);
    }
    grid_dependency_wait();
    allow_dependents();
    // per sequence: context (clamped to the table), query count (clamped to
    // [0, min(n, max_query_len)]), first query row, and block prefix sums
    const int cap = a.max_blocks * 16;
    for (int i = threadIdx.x; i < a.batch; i += blockDim.x) {
        int n = a.lens[i];
        bool bad = n < 0 || n > cap;
        n = n < 0 ? 0 : (n > cap ? cap : n);
        // without query offsets: one query per sequence (row i), none for an empty context
        const int q0 = a.qstart != nullptr ? a.qstart[i] : i;
        int nq = a.qstart != nullptr ? a.qstart[i + 1] - q0 : (n > 0 ? 1 : 0);
        if (q0 < 0 || nq < 0 || nq > n || nq > a.max_query_len) {
            bad = true;
            nq = 0;
        }
        if (bad && blockIdx.x == 0) atomicOr(a.status, PKV_DEVERR_RANGE);
        s_len[i] = n;
        s_pre[i] = nq > 0 ? (n + 15) >> 4 : 0;  // a sequence without queries streams nothing
    }
    __syncthreads();
    if (threadIdx.x < 32) {
        int carry = 0;
        for (int base = 0; base < a.batch; base += 32) {
            int x = base + lane < a.batch ? s_pre[base + lane] : 0;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int y = __shfl_up_sync(0xffffffffu, x, o);
                if (lane >= o) x += y;
            }
            if (base + lane < a.batch) s_pre[base + lane] = x + carry;
            carry += __shfl_sync(0xffffffffu, x, 31);
        }
    }
    __syncthreads();

    if (a.qstart == nullptr) {
        // one query per sequence: an empty context gives a zero row
        const int row = a.q_heads * D;
        for (int i = blockIdx.x; i < a.batch; i += a.num_ctas) {
            if (s_len[i] != 0) continue;
            __nv_bfloat16* o = static_cast<__nv_bfloat16*>(a.out) + static_cast<long long>(i) * row;
            for (int e = threadIdx.x; e < row; e += blockDim.x) o[e] = __float2bfloat16_rn(0.f);
        }
    }
    const long long U = static_cast<long long>(a.kv_heads) * s_pre[a.batch - 1];
    const long long cta = blockIdx.x;
    const long long ua = range_start(cta, U, a.num_ctas);
    const long long ub = range_start(cta + 1, U, a.num_ctas);

    if (warp >= C::kConsumers) {
        // ------------------------------------------------ producer warps (as in the decode kernel)
        // Both walk the same blocks in the same order; warp kConsumers issues
        // the K side and warp kConsumers + 1 the V side, each arriving on its
        // own full barrier. One warp issuing all the copies of an int8 block
        // (codes and scale rows) was the pace-setter: the int8 call took
        // 107 us with one producer, 95 us without the scale copies.
        if (a.test_stall) return;  // test hook: nothing is ever issued, so every consumer wait runs out
        const int side = warp - C::kConsumers;
        uint64_t* fulls = full + side * C::kStages;
        const uint64_t kv_policy = l2_evict_first_policy();
        Walker wk;
        wk.init(s_pre, a.batch, a.kv_heads, ua, ub);
        long long k = 0;
        Piece pc;
        bool ok = true;
        while (ok && wk.next(pc)) {
            const int32_t* trow = a.tables + static_cast<long long>(pc.seq) * a.max_blocks + pc.blk_from;
            const int cnt_piece = pc.blk_to - pc.blk_from;
            int cur = lane < cnt_piece ? __ldg(trow + lane) : 0;
            for (int b0 = 0; ok && b0 < cnt_piece; b0 += 32) {
                const int nidx = b0 + 32 + lane;
                const int nxt = nidx < cnt_piece ? __ldg(trow + nidx) : 0;
                const int cnt = min(32, cnt_piece - b0);
                // In order, but in batches: each lane probes (without
                // blocking) the stage of one of the next kIssueLanes blocks,
                // and the longest run of free stages from the first is issued
                // at once, one block per lane with the same instructions (a
                // TMA instruction costs the warp about the same whether one
                // lane issues it or eight). Only when the first stage is busy
                // does the warp wait (bounded), for that one.
                for (int e0 = 0; e0 < cnt;) {
                    const int e = e0 + lane;
                    const long long kk = k + lane;
                    const int s = static_cast<int>(kk % C::kStages);
                    const uint32_t par = static_cast<uint32_t>((kk / C::kStages) & 1) ^ 1u;
                    const bool probe = lane < C::kIssueLanes && e < cnt && mbar_test_wait(&empty[s], par);
                    int n = __ffs(~__ballot_sync(0xffffffffu, probe)) - 1;  // free stages from the first on
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
                            mbar_arrive_expect_tx(&fulls[s], side == 0 ? C::kTxK : C::kTxV);
                        } else {
                            if (side == 0) atomicOr(a.status, PKV_DEVERR_RANGE);
                            mbar_arrive(&fulls[s]);
                        }
                    }
                    if (load) {
                        uint8_t* st = smem + s * C::kStageBytes + side * C::kSideBytes;
                        const int hb = bid * a.kv_heads + pc.head;
                        if (Q8) {
                            if (side == 0) {
                                tma_load_2d(st, &tmK, 0, hb * 16, &fulls[s], kv_policy);
                                tma_load_2d(smem + C::kOffScales + s * C::kScaleBytes, &tmS, 0, hb, &fulls[s],
                                            kv_policy);
                            } else {
                                tma_load_2d(st, &tmV, 0, hb * 16, &fulls[s], kv_policy);
                            }
                        } else {
                            const int y = hb * 16;
                            if (side == 0) {
#pragma unroll
                                for (int hf = 0; hf < C::kHalves; ++hf)
                                    tma_load_2d(st + hf * 2048, &tmK, hf * 64, y, &fulls[s], kv_policy);
                            } else {
#pragma unroll
                                for (int hf = 0; hf < C::kHalves; ++hf)
                                    tma_load_2d(st + hf * 2048, &tmV, hf * 64, y, &fulls[s], kv_policy);
                            }
                        }
                    }
                    k += n;
                    e0 += n;
                }
                cur = nxt;
            }
        }
        if (!ok && lane == 0) {  // after an abort: wait (bounded) for this side's copies still in flight
            const long long first = k > C::kStages ? k - C::kStages : 0;
            for (long long u = first; u < k; ++u)
                mbar_wait(&fulls[u % C::kStages], static_cast<uint32_t>((u / C::kStages) & 1), a.status, nullptr);
        }
        return;
    }

    // ---------------------------------------------------- consumer warps
    const int W = a.wpu;      // warps per unit (row groups)
    const int UG = 4 / W;     // unit lanes
    const int rg = warp % W;  // this warp's row group: rows 8 rg .. 8 rg + 7
    const int ul = warp / W;  // this warp's unit lane
    const int gid = lane >> 2;  // fragment row group
    const int tig = lane & 3;   // thread in group
    const float scale_log2 = a.scale * kLog2e;
    const __nv_bfloat16* q = static_cast<const __nv_bfloat16*>(a.q);
    const int q8 = lane >> 3, r8 = lane & 7;
    const int k_row = r8 + 8 * (q8 & 1);
    const int k_chunk = q8 >> 1;
    const int v_row = r8 + 8 * (q8 >> 1);
    const int v_chunk = q8 & 1;

    Walker wk;
    wk.init(s_pre, a.batch, a.kv_heads, ua, ub);
    long long k = 0;
    int piece_idx = 0;
    Piece pc;
    Piece pending[2];
    int npending = 0;
    while (wk.next(pc)) {
        const int n_ctx = s_len[pc.seq];
        const int q0 = a.qstart != nullptr ? a.qstart[pc.seq] : pc.seq;
        const int nq = a.qstart != nullptr ? a.qstart[pc.seq + 1] - q0 : 1;  // valid: the sequence has units
        const int rows = nq * G;
        const bool active = rg * 8 < rows;
        // Q^T fragments: column n = row 8 rg + gid of the row group
        uint32_t qf[D / 16][2];
        float cf0 = scale_log2, cf1 = scale_log2;  // int8 path: per-column score factors
        float kb0 = 0.f, kb1 = 0.f;                // int8 path: the code bias times the column's query sum
        {
            const int rr = rg * 8 + gid;
            const bool live = rr < rows;
            const int t = live ? rr / G : 0;
            const __nv_bfloat16* qrow =
                q + (static_cast<long long>(q0 + t) * a.q_heads + pc.head * G + (live ? rr - t * G : 0)) * D;
            if (!Q8) {
                const uint32_t* q32 = reinterpret_cast<const uint32_t*>(qrow);
#pragma unroll
                for (int j = 0; j < D / 16; ++j) {
                    qf[j][0] = live ? __ldg(q32 + (16 * j + 2 * tig) / 2) : 0u;
                    qf[j][1] = live ? __ldg(q32 + (16 * j + 2 * tig + 8) / 2) : 0u;
                }
            } else {
                // f16 operands: coordinates 4 tig .. 4 tig + 3 of each 16 (the
                // contraction order of the int8 K fragments), the row scaled by
                // 2^-e so that its largest magnitude stays below 2^15
                float qv[D / 16][4];
                float qmax = 0.f;
#pragma unroll
                for (int j = 0; j < D / 16; ++j) {
                    const uint2 w = live ? __ldg(reinterpret_cast<const uint2*>(qrow + 16 * j + 4 * tig)) : make_uint2(0u, 0u);
                    qv[j][0] = bf16lo_to_f32(w.x);
                    qv[j][1] = bf16hi_to_f32(w.x);
                    qv[j][2] = bf16lo_to_f32(w.y);
                    qv[j][3] = bf16hi_to_f32(w.y);
                    qmax = fmaxf(qmax, fmaxf(fmaxf(fabsf(qv[j][0]), fabsf(qv[j][1])), fmaxf(fabsf(qv[j][2]), fabsf(qv[j][3]))));
                }
                qmax = fmaxf(qmax, __shfl_xor_sync(0xffffffffu, qmax, 1));
                qmax = fmaxf(qmax, __shfl_xor_sync(0xffffffffu, qmax, 2));
                const int ex = static_cast<int>((__float_as_uint(qmax) >> 23) & 0xffu) - 127;
                const int e = ex > 14 ? ex - 14 : 0;
                const float down = __uint_as_float(static_cast<uint32_t>(127 - e) << 23);
                const float up = __uint_as_float(static_cast<uint32_t>(127 + e) << 23);
                float qsum = 0.f;  // of the f16 operands as rounded
#pragma unroll
                for (int j = 0; j < D / 16; ++j) {
                    qf[j][0] = pack_f16x2(qv[j][0] * down, qv[j][1] * down);
                    qf[j][1] = pack_f16x2(qv[j][2] * down, qv[j][3] * down);
                    qsum += f16x2_sum(qf[j][0]) + f16x2_sum(qf[j][1]);
                }
                qsum += __shfl_xor_sync(0xffffffffu, qsum, 1);
                qsum += __shfl_xor_sync(0xffffffffu, qsum, 2);
                // S^T columns 2 tig, 2 tig + 1 are the rows held by lanes 8 tig and 8 tig + 4
                cf0 = __shfl_sync(0xffffffffu, up, 8 * tig) * scale_log2;
                cf1 = __shfl_sync(0xffffffffu, up, 8 * tig + 4) * scale_log2;
                kb0 = kCodeBias * __shfl_sync(0xffffffffu, qsum, 8 * tig);
                kb1 = kCodeBias * __shfl_sync(0xffffffffu, qsum, 8 * tig + 4);
            }
        }
        const int tokA = sigma(gid), tokB = sigma(gid + 8);  // int8 path: tokens of S^T rows gid, gid + 8
        const int kq_tok = sigma(r8 + 8 * (q8 & 1));         // int8 path: K token row of this lane's address
        // last visible position of the lane's two columns (rows 2 tig, 2 tig + 1 of the group)
        const int rc0 = rg * 8 + 2 * tig, rc1 = rc0 + 1;
        const int lim0 = rc0 < rows ? n_ctx - nq + rc0 / G : -1;
        const int lim1 = rc1 < rows ? n_ctx - nq + rc1 / G : -1;
        float m0 = ninf(), m1 = ninf(), l0 = 0.f, l1 = 0.f;
        float o[D / 16][4];
#pragma unroll
        for (int i = 0; i < D / 16; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;

        // this unit lane's blocks of the piece: running block index k = ul (mod UG)
        const long long k_end = k + (pc.blk_to - pc.blk_from);
        const int skip = (ul - static_cast<int>(k & (UG - 1))) & (UG - 1);
        k += skip;
        for (int blk = pc.blk_from + skip; blk < pc.blk_to; blk += UG, k += UG) {
            const int s = static_cast<int>(k % C::kStages);
            // K side first; the V side is waited for just before the PV product
            const uint32_t par = static_cast<uint32_t>((k / C::kStages) & 1);
            const unsigned long long wlim = a.test_stall ? kTestWaitLimitNs : kWaitLimitNs;
            if (!mbar_wait(&full[s], par, a.status, abort_flag, wlim)) return;
            const int valid = min(16, n_ctx - blk * 16);
            const bool use = stage_ok[s] && active;
            if (!Q8 && use) {
                const uint32_t kbase = smem_u32(smem + s * C::kStageBytes);
                const uint32_t vbase = kbase + C::kPoolBytes;
                // four independent accumulator chains over the k-steps
                float sc4[4][4] = {};
#pragma unroll
                for (int j = 0; j < D / 16; ++j) {
                    const int gc = 2 * j + k_chunk;
                    const uint32_t addr = kbase + (gc >> 3) * 2048 + k_row * 128 + (((gc & 7) ^ r8) << 4);
                    uint32_t a0, a1, a2, a3;
                    ldmatrix_x4(addr, a0, a1, a2, a3);
                    mma_bf16_16816(sc4[j & 3], a0, a1, a2, a3, qf[j][0], qf[j][1]);
                }
                float sa[4], sb[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    sa[e] = sc4[0][e] + sc4[2][e];
                    sb[e] = sc4[1][e] + sc4[3][e];
                }
                // [0] (token gid, row 2tig) [1] (gid, 2tig+1) [2] (gid+8, 2tig) [3] (gid+8, 2tig+1)
                const int p0 = blk * 16 + gid, p1 = p0 + 8;
                const float x0 = p0 <= lim0 ? (sa[0] + sb[0]) * scale_log2 : ninf();
                const float x1 = p0 <= lim1 ? (sa[1] + sb[1]) * scale_log2 : ninf();
                const float x2 = p1 <= lim0 ? (sa[2] + sb[2]) * scale_log2 : ninf();
                const float x3 = p1 <= lim1 ? (sa[3] + sb[3]) * scale_log2 : ninf();
                float mx0 = fmaxf(x0, x2), mx1 = fmaxf(x1, x3);
                if (__any_sync(0xffffffffu, mx0 > m0 + 8.f || mx1 > m1 + 8.f)) {
#pragma unroll
                    for (int off = 4; off < 32; off <<= 1) {
                        mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, off));
                        mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, off));
                    }
                    const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
                    const float nb0 = mn0 == ninf() ? 0.f : mn0;
                    const float nb1 = mn1 == ninf() ? 0.f : mn1;
                    const float al0 = m0 == ninf() ? 0.f : ex2(m0 - nb0);
                    const float al1 = m1 == ninf() ? 0.f : ex2(m1 - nb1);
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
                const float b0 = m0 == ninf() ? 0.f : m0;
                const float b1 = m1 == ninf() ? 0.f : m1;
                const float e0 = ex2(x0 - b0), e1 = ex2(x1 - b1), e2 = ex2(x2 - b0), e3 = ex2(x3 - b1);
                l0 += e0 + e2;
                l1 += e1 + e3;
                const uint32_t h01 = pack_bf16x2(e0, e1), h23 = pack_bf16x2(e2, e3);
                const uint32_t lo01 = pack_bf16x2(e0 - bf16lo_to_f32(h01), e1 - bf16hi_to_f32(h01));
                const uint32_t lo23 = pack_bf16x2(e2 - bf16lo_to_f32(h23), e3 - bf16hi_to_f32(h23));
                const uint32_t bh0 = movmatrix_trans(h01), bh1 = movmatrix_trans(h23);
                const uint32_t bl0 = movmatrix_trans(lo01), bl1 = movmatrix_trans(lo23);
                if (!mbar_wait(&full[C::kStages + s], par, a.status, abort_flag, wlim)) return;
                // rows past the context may hold anything: zero them in V
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
            if (Q8 && use) {
                const uint32_t kb = smem_u32(smem + s * C::kStageBytes);
                const uint32_t vb = kb + 16 * D;
                const float* ksc = reinterpret_cast<const float*>(smem + C::kOffScales + s * C::kScaleBytes);
                const float* vsc = ksc + C::kVScaleOff / 4;
                // ---- S^T = K Q^T on f16 codes: one ldmatrix gives two k-steps
                // four independent accumulator chains over the k-steps
                float sc4[4][4] = {};
#pragma unroll
                for (int jj = 0; jj < D / 32; ++jj) {
                    const int gc = 2 * jj + (q8 >> 1);
                    const uint32_t addr = kb + kq_tok * 128 + (((gc & 7) ^ (kq_tok & 7)) << 4);
                    uint32_t w0, w1, w2, w3;
                    ldmatrix_x4(addr, w0, w1, w2, w3);
                    uint32_t a0, a1, a2, a3;
                    codes_to_f16x2_biased(w0, a0, a2);
                    codes_to_f16x2_biased(w1, a1, a3);
                    mma_f16_16816(sc4[(2 * jj) & 3], a0, a1, a2, a3, qf[2 * jj][0], qf[2 * jj][1]);
                    codes_to_f16x2_biased(w2, a0, a2);
                    codes_to_f16x2_biased(w3, a1, a3);
                    mma_f16_16816(sc4[(2 * jj + 1) & 3], a0, a1, a2, a3, qf[2 * jj + 1][0], qf[2 * jj + 1][1]);
                }
                float sa[4], sb[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    sa[e] = sc4[0][e] + sc4[2][e];
                    sb[e] = sc4[1][e] + sc4[3][e];
                }
                // [0] (token tokA, row 2tig) [1] (tokA, 2tig+1) [2] (tokB, 2tig) [3] (tokB, 2tig+1)
                const int pA = blk * 16 + tokA, pB = blk * 16 + tokB;
                const float kA = ksc[tokA], kB = ksc[tokB];
                const float x0 = pA <= lim0 ? (sa[0] + sb[0] - kb0) * kA * cf0 : ninf();
                const float x1 = pA <= lim1 ? (sa[1] + sb[1] - kb1) * kA * cf1 : ninf();
                const float x2 = pB <= lim0 ? (sa[2] + sb[2] - kb0) * kB * cf0 : ninf();
                const float x3 = pB <= lim1 ? (sa[3] + sb[3] - kb1) * kB * cf1 : ninf();
                if (!mbar_wait(&full[C::kStages + s], par, a.status, abort_flag, wlim)) return;
                // P' = P times the V scale of its token (zero past the context), as f16
                float vA = pA < n_ctx ? vsc[tokA] : 0.f, vB = pB < n_ctx ? vsc[tokB] : 0.f;
                // P <= 2^8 under the lazy rescale, so P' stays below the f16
                // maximum while every V scale is at most kVScaleF16Safe. A block
                // with a larger scale (rows with max |v| above ~32 000) runs its
                // product on P' 2^-k and O 2^-k, and O is scaled back by 2^k
                // afterwards: powers of two, exact in fp32. One vote covers both
                // rare cases (a new running maximum, a large V scale): a second
                // vote and branch per block cost 1.6 % of the call.
                float mx0 = fmaxf(x0, x2), mx1 = fmaxf(x1, x3);
                float o_back = 1.f;
                if (__any_sync(0xffffffffu, mx0 > m0 + 8.f || mx1 > m1 + 8.f || fmaxf(vA, vB) > kVScaleF16Safe)) {
#pragma unroll
                    for (int off = 4; off < 32; off <<= 1) {
                        mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, off));
                        mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, off));
                    }
                    // a rescale to the running maximum (exact whether or not it moved)
                    const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
                    const float nb0 = mn0 == ninf() ? 0.f : mn0;
                    const float nb1 = mn1 == ninf() ? 0.f : mn1;
                    float al0 = m0 == ninf() ? 0.f : ex2(m0 - nb0);
                    float al1 = m1 == ninf() ? 0.f : ex2(m1 - nb1);
                    l0 *= al0;
                    l1 *= al1;
                    m0 = mn0;
                    m1 = mn1;
                    // and the block's V-scale shift, folded into the same pass over O
                    float vm = fmaxf(vA, vB);
#pragma unroll
                    for (int off = 1; off < 32; off <<= 1) vm = fmaxf(vm, __shfl_xor_sync(0xffffffffu, vm, off));
                    if (vm > kVScaleF16Safe && vm <= 3.0e38f) {
                        const int k2 = pow2_shift_to_fit(vm);
                        const float down = __uint_as_float(static_cast<uint32_t>(127 - k2) << 23);
                        o_back = __uint_as_float(static_cast<uint32_t>(127 + k2) << 23);
                        vA *= down;
                        vB *= down;
                        al0 *= down;
                        al1 *= down;
                    }
#pragma unroll
                    for (int i = 0; i < D / 16; ++i) {
                        o[i][0] *= al0;
                        o[i][1] *= al1;
                        o[i][2] *= al0;
                        o[i][3] *= al1;
                    }
                }
                const float b0 = m0 == ninf() ? 0.f : m0;
                const float b1 = m1 == ninf() ? 0.f : m1;
                const float e0 = ex2(x0 - b0), e1 = ex2(x1 - b1), e2 = ex2(x2 - b0), e3 = ex2(x3 - b1);
                l0 += e0 + e2;
                l1 += e1 + e3;
                const uint32_t bh0 = movmatrix_trans(pack_f16x2(e0 * vA, e1 * vA));
                const uint32_t bh1 = movmatrix_trans(pack_f16x2(e2 * vB, e3 * vB));
                // ---- O^T += V^T P'^T: V coordinate rows of 16 token codes
#pragma unroll
                for (int ii = 0; ii < D / 32; ++ii) {
                    uint32_t w0, w1, w2, w3;
                    ldmatrix_x4(vb + (32 * ii + 8 * q8 + r8) * 16, w0, w1, w2, w3);
                    uint32_t a0, a1, a2, a3;
                    codes_to_f16x2(w0, a0, a2);
                    codes_to_f16x2(w1, a1, a3);
                    mma_f16_16816(o[2 * ii], a0, a1, a2, a3, bh0, bh1);
                    codes_to_f16x2(w2, a0, a2);
                    codes_to_f16x2(w3, a1, a3);
                    mma_f16_16816(o[2 * ii + 1], a0, a1, a2, a3, bh0, bh1);
                }
                if (o_back != 1.f) {
#pragma unroll
                    for (int i = 0; i < D / 16; ++i) {
                        o[i][0] *= o_back;
                        o[i][1] *= o_back;
                        o[i][2] *= o_back;
                        o[i][3] *= o_back;
                    }
                }
            }
            // a stage is handed back only after both of its sides have landed
            if (!use && !mbar_wait(&full[C::kStages + s], par, a.status, abort_flag, wlim)) return;
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[s]);
        }
        k = k_end;
        // ---- end of the piece: sums across the token rows of the fragments
#pragma unroll
        for (int off = 4; off < 32; off <<= 1) {
            l0 += __shfl_xor_sync(0xffffffffu, l0, off);
            l1 += __shfl_xor_sync(0xffffffffu, l1, off);
        }
        const int c0 = 2 * tig, c1 = c0 + 1;  // the group's rows of the lane's columns
        // The row group's state: the warp's own registers (one unit lane), or
        // the combination of the unit lanes' states through shared memory.
        float* buf = scratch + (piece_idx & 1) * (C::kConsumers * 8 * (D + 2));
        if (UG > 1) {
            float* so = buf + warp * 8 * (D + 2);  // [8 rows][D], then 8 maxima, 8 sums
#pragma unroll
            for (int i = 0; i < D / 16; ++i) {
                so[c0 * D + 16 * i + gid] = o[i][0];
                so[c1 * D + 16 * i + gid] = o[i][1];
                so[c0 * D + 16 * i + gid + 8] = o[i][2];
                so[c1 * D + 16 * i + gid + 8] = o[i][3];
            }
            if (gid == 0) {
                so[8 * D + c0] = active ? m0 : ninf();
                so[8 * D + c1] = active ? m1 : ninf();
                so[8 * D + 8 + c0] = active ? l0 : 0.f;
                so[8 * D + 8 + c1] = active ? l1 : 0.f;
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(piece_bar);
            if (!mbar_wait(piece_bar, static_cast<uint32_t>(piece_idx & 1), a.status, abort_flag)) return;
            ++piece_idx;
            if (ul != 0 || !active) continue;
            // combine the unit lanes of this row group: lane = 4 row + quarter
            const int rw = lane >> 2;
            const int d0 = (lane & 3) * (D / 4);
            float M = ninf();
            for (int u = 0; u < UG; ++u) M = fmaxf(M, buf[(u * W + rg) * 8 * (D + 2) + 8 * D + rw]);
            const float base = M == ninf() ? 0.f : M;
            float L = 0.f;
            float O[D / 4];
#pragma unroll
            for (int e = 0; e < D / 4; ++e) O[e] = 0.f;
            for (int u = 0; u < UG; ++u) {
                const float* su = buf + (u * W + rg) * 8 * (D + 2);
                const float mu = su[8 * D + rw];
                const float wu = mu == ninf() ? 0.f : ex2(mu - base);
                L += wu * su[8 * D + 8 + rw];
#pragma unroll
                for (int e = 0; e < D / 4; ++e) O[e] += wu * su[rw * D + d0 + e];
            }
            const int rr = rg * 8 + rw;
            if (pc.complete) {
                if (rr < rows) {
                    const int t = rr / G;
                    __nv_bfloat16* orow = static_cast<__nv_bfloat16*>(a.out) +
                                          (static_cast<long long>(q0 + t) * a.q_heads + pc.head * G + (rr - t * G)) * D;
                    const float inv = L > 0.f ? 1.f / L : 0.f;
#pragma unroll
                    for (int e = 0; e < D / 4; e += 2)
                        *reinterpret_cast<uint32_t*>(orow + d0 + e) = pack_bf16x2(O[e] * inv, O[e + 1] * inv);
                }
            } else {
                float* sl = mq_slice(a.partials, cta, pc.first ? 0 : 1, rg, D);
#pragma unroll
                for (int e = 0; e < D / 4; ++e) sl[rw * D + d0 + e] = O[e];
                if ((lane & 3) == 0) {
                    sl[8 * D + rw] = M;
                    sl[8 * D + 8 + rw] = L;
                }
                pending[npending++] = pc;
            }
            continue;
        }
        if (!active) continue;
        if (pc.complete) {
            const float i0 = l0 > 0.f ? 1.f / l0 : 0.f, i1 = l1 > 0.f ? 1.f / l1 : 0.f;
#pragma unroll
            for (int c = 0; c < 2; ++c) {
                const int rr = rg * 8 + (c ? c1 : c0);
                if (rr >= rows) continue;
                const int t = rr / G;
                __nv_bfloat16* orow = static_cast<__nv_bfloat16*>(a.out) +
                                      (static_cast<long long>(q0 + t) * a.q_heads + pc.head * G + (rr - t * G)) * D;
                const float inv = c ? i1 : i0;
#pragma unroll
                for (int i = 0; i < D / 16; ++i) {
                    orow[16 * i + gid] = __float2bfloat16_rn(o[i][c] * inv);
                    orow[16 * i + gid + 8] = __float2bfloat16_rn(o[i][2 + c] * inv);
                }
            }
        } else {
            float* sl = mq_slice(a.partials, cta, pc.first ? 0 : 1, rg, D);
#pragma unroll
            for (int i = 0; i < D / 16; ++i) {
                sl[c0 * D + 16 * i + gid] = o[i][0];
                sl[c1 * D + 16 * i + gid] = o[i][1];
                sl[c0 * D + 16 * i + gid + 8] = o[i][2];
                sl[c1 * D + 16 * i + gid + 8] = o[i][3];
            }
            if (gid == 0) {
                sl[8 * D + c0] = m0;
                sl[8 * D + c1] = m1;
                sl[8 * D + 8 + c0] = l0;
                sl[8 * D + 8 + c1] = l1;
            }
            pending[npending++] = pc;
        }
    }
    // announce this row group's cut pieces; the warp completing a count merges
    if (npending == 0) return;
    __threadfence();
    __syncwarp();
    const long long Cn = a.num_ctas;
    for (int i = 0; i < npending; ++i) {
        const Piece& pp = pending[i];
        const long long c0s = cta_of(pp.seg_start, U, Cn);
        const long long c1s = cta_of(pp.seg_start + pp.seg_len - 1, U, Cn);
        const int np = pieces_of_segment(c0s, c1s, U, Cn);
        int* counter = a.counters + (static_cast<long long>(pp.seq) * a.kv_heads + pp.head) * 4 + rg;
        int old = 0;
        if (lane == 0) old = atomicAdd(counter, 1);
        old = __shfl_sync(0xffffffffu, old, 0);
        if (old != np - 1) continue;
        __threadfence();
        const int slot0 = (pp.seg_start == range_start(c0s, U, Cn)) ? 0 : 1;
        // without query offsets: sequence i has its one query in row i
        const int qq0 = a.qstart != nullptr ? a.qstart[pp.seq] : pp.seq;
        const int nqq = a.qstart != nullptr ? a.qstart[pp.seq + 1] - qq0 : 1;
        mq_merge<D>(pp, a, U, rg, lane, c0s, slot0, np, nqq * G, qq0);
        if (lane == 0) *counter = 0;
    }
}

template <typename K>
int mq_occupancy(K kernel, int threads, size_t smem) {
    int n = 0;
    cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kernel, threads, smem) != cudaSuccess || n < 1) n = 1;
    return n;
}

// Ring depth (a build-time knob): stages of 2 * 16 * D bytes (bf16) or 16 * D
// bytes (int8 codes) per CTA.
#ifndef PKV_MQ_STAGES
#define PKV_MQ_STAGES 8
#endif
#ifndef PKV_MQ8_STAGES
#define PKV_MQ8_STAGES 16
#endif
constexpr int kMqStages = PKV_MQ_STAGES;
constexpr int kMq8Stages = PKV_MQ8_STAGES;
template <bool Q8>
constexpr int mq_stages() { return Q8 ? kMq8Stages : kMqStages; }

template <int D, bool Q8>
cudaError_t run_mq(const MqArgs& a, int grid, cudaStream_t s) {
    using C = Mq<D, mq_stages<Q8>(), Q8>;
    CUtensorMap tmK, tmV, tmS;
    if (Q8) {
        const uint64_t hb = static_cast<uint64_t>(a.num_blocks) * a.kv_heads;
        if (!make_map_2d(&tmK, PKV_INT8, a.k_cache, D, hb * 16, D, D, 16, true, true) ||
            // the V codes of one (block, head) are D x 16 contiguous bytes: described as 16 rows of D
            // bytes, one TMA box moves them with 16 row requests instead of D requests of 16 bytes
            !make_map_2d(&tmV, PKV_INT8, a.v_cache, D, hb * 16, D, D, 16, false, true) ||
            // one 128-byte scale record (K row, V row) per (block, head), fetched
            // without L2 promotion: a 256-byte fetch would bring a record of
            // another head along, which this CTA does not read
            !make_map_2d(&tmS, PKV_F32, a.scales, 32, hb, 128, 32, 1, false, false))
            return cudaErrorInvalidValue;
    } else {
        const int64_t rows = a.num_blocks * a.kv_heads * 16;
        if (!make_pool_map(&tmK, a.k_cache, rows, D) || !make_pool_map(&tmV, a.v_cache, rows, D))
            return cudaErrorInvalidValue;
        tmS = tmK;  // unused by the bf16 path
    }
    const size_t smem = C::smem_bytes(a.batch);
    cudaFuncSetAttribute(mq_tc_kernel<D, mq_stages<Q8>(), Q8>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         static_cast<int>(smem));
    return launch_pdl(mq_tc_kernel<D, mq_stages<Q8>(), Q8>, dim3(grid), dim3(C::kThreads), smem, s, a, tmK, tmV, tmS);
}

}  // namespace

int mq_num_ctas(int head_dim, int batch, const pkv_decode_opts* opts, bool q8) {
    if (opts && opts->num_ctas > 0) return opts->num_ctas;
    static std::mutex mu;
    static int cache[3][64] = {};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 0 || dev >= 64) dev = 0;
    (void)batch;
    std::lock_guard<std::mutex> lock(mu);
    const int which = q8 ? 2 : (head_dim == 128 ? 1 : 0);
    int& slot = cache[which][dev];
    if (slot == 0) {
        // occupancy at the largest launch (the per-sequence arrays grow with the batch)
        if (q8)
            slot = mq_occupancy(mq_tc_kernel<128, kMq8Stages, true>, Mq<128, kMq8Stages, true>::kThreads,
                                Mq<128, kMq8Stages, true>::smem_bytes(kMaxBatchPerLaunch));
        else if (head_dim == 128)
            slot = mq_occupancy(mq_tc_kernel<128, kMqStages, false>, Mq<128, kMqStages>::kThreads,
                                Mq<128, kMqStages>::smem_bytes(kMaxBatchPerLaunch));
        else
            slot = mq_occupancy(mq_tc_kernel<64, kMqStages, false>, Mq<64, kMqStages>::kThreads,
                                Mq<64, kMqStages>::smem_bytes(kMaxBatchPerLaunch));
    }
    return slot * device_sm_count();
}

size_t mq_workspace_bytes(int batch, int kv_heads, int head_dim, int num_ctas, size_t* counters_offset,
                          size_t* partials_offset) {
    const int chunk = batch < kMaxBatchPerLaunch ? (batch < 1 ? 1 : batch) : kMaxBatchPerLaunch;
    const size_t counters = static_cast<size_t>(chunk) * kv_heads * 4 * sizeof(int);
    *counters_offset = 256;
    *partials_offset = 256 + (counters + 255) / 256 * 256;
    return *partials_offset + static_cast<size_t>(num_ctas) * 2 * 4 * 8 * (head_dim + 2) * sizeof(float);
}

namespace {
// Checked mode: query counts must lie in [0, min(context, max_query_len)]
// and the first query rows must be non-negative.
__global__ void check_queries_kernel(const int32_t* lens, const int32_t* qstart, int32_t batch,
                                     int32_t max_query_len, unsigned int* verdict) {
    for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < batch; i += gridDim.x * blockDim.x) {
        const int n = lens[i], q0 = qstart[i], nq = qstart[i + 1] - q0;
        if (q0 < 0 || nq < 0 || nq > n || nq > max_query_len) atomicOr(verdict, kVerdictRange);
    }
}
}  // namespace

cudaError_t launch_check_queries(const int32_t* lens, const int32_t* qstart, int32_t batch, int32_t max_query_len,
                                 unsigned int* verdict, cudaStream_t s) {
    if (batch <= 0) return cudaSuccess;
    check_queries_kernel<<<(batch + 255) / 256, 256, 0, s>>>(lens, qstart, batch, max_query_len, verdict);
    return cudaGetLastError();
}

cudaError_t launch_multiquery(const MqArgs& a, cudaStream_t s) {
    if (a.q8) return run_mq<128, true>(a, a.num_ctas, s);
    return a.head_dim == 128 ? run_mq<128, false>(a, a.num_ctas, s) : run_mq<64, false>(a, a.num_ctas, s);
}

}  // namespace pkv
