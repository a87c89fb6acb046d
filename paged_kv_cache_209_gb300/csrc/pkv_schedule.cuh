// Stream-K schedule shared by the split decode kernels: one unit of work is
// one (sequence i, KV head h, block b), units ordered i-major, then h, then
// b; the units of one (i, h) form a segment. A launch of C CTAs gives CTA c
// the contiguous units [c U / C, (c + 1) U / C), so every CTA streams the same
// number of blocks (to within one) whatever the mix of context lengths; a
// segment cut by a range boundary leaves one piece per CTA it touches.
#pragma once

#include <stdint.h>

namespace pkv {
namespace {

struct Piece {
    int seq, head;
    int blk_from, blk_to;  // blocks [from, to) of the sequence
    bool complete;         // the piece is the whole segment
    bool first;            // the piece opens this CTA's range
    long long seg_start;   // first unit of the segment
    int seg_len;           // units (blocks) of the segment
};

// Walks the segment pieces of the unit range [start, end).
struct Walker {
    const int32_t* pre;
    int kv_heads;
    long long start, u, end;
    int i, h, nb;
    long long seg_base;

    __device__ void init(const int32_t* pre_, int batch, int kvh, long long a, long long b) {
        pre = pre_;
        kv_heads = kvh;
        start = u = a;
        end = b;
        if (u >= end) return;
        int lo = 0, hi = batch - 1;
        while (lo < hi) {
            const int mid = (lo + hi) >> 1;
            if (static_cast<long long>(pre[mid]) * kvh > u)
                hi = mid;
            else
                lo = mid + 1;
        }
        i = lo;
        const int excl = i ? pre[i - 1] : 0;
        nb = pre[i] - excl;
        seg_base = static_cast<long long>(kvh) * excl;
        h = static_cast<int>((u - seg_base) / nb);
    }

    __device__ bool next(Piece& p) {
        if (u >= end) return false;
        const long long s0 = seg_base + static_cast<long long>(h) * nb;
        const long long s1 = s0 + nb;
        const long long pe = s1 < end ? s1 : end;
        p.seq = i;
        p.head = h;
        p.blk_from = static_cast<int>(u - s0);
        p.blk_to = static_cast<int>(pe - s0);
        p.complete = (u == s0) && (pe == s1);
        p.first = (u == start);
        p.seg_start = s0;
        p.seg_len = nb;
        u = pe;
        if (u < end) {
            if (++h == kv_heads) {
                h = 0;
                do {
                    ++i;
                } while (pre[i] == pre[i - 1]);
                const int excl = pre[i - 1];
                nb = pre[i] - excl;
                seg_base = static_cast<long long>(kv_heads) * excl;
            }
        }
        return true;
    }
};

__device__ __forceinline__ long long range_start(long long c, long long U, long long C) { return c * U / C; }

// The CTA whose range holds unit u: max c with range_start(c) <= u.
__device__ __forceinline__ long long cta_of(long long u, long long U, long long C) { return ((u + 1) * C - 1) / U; }

// Pieces of one segment: every CTA whose unit range meets [S0, S1).
__device__ __forceinline__ int pieces_of_segment(long long c0, long long c1, long long U, long long C) {
    if (U >= C) return static_cast<int>(c1 - c0 + 1);  // no CTA range is empty
    int n = 0;
    for (long long c = c0; c <= c1; ++c) n += range_start(c, U, C) < range_start(c + 1, U, C);
    return n;
}

// CTA holding piece p (0-based) of the segment that starts at unit S0 and
// whose first piece is in CTA c0. With at least one unit per CTA every range
// is non-empty, so pieces sit in consecutive CTAs; with fewer units than CTAs
// every non-empty range holds one unit, so piece p is unit S0 + p's CTA.
__device__ __forceinline__ long long piece_cta(long long S0, long long c0, int p, long long U, long long C) {
    return U >= C ? c0 + p : cta_of(S0 + p, U, C);
}

}  // namespace
}  // namespace pkv
