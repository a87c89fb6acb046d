// Stream-K schedule shared by the split decode kernels: one unit of work is
// one (sequence i, KV head h, block b), units ordered i-major, then h, then
// b; the units of one (i, h) form a segment. A launch of C CTAs gives CTA c
// a contiguous range of units: [c U / C, (c + 1) U / C) in the multi-query
// kernels, so every CTA streams the same number of blocks (to within one)
// whatever the mix of context lengths; in the decode kernels the ranges are
// placed by cost (CostSplit below), so a CTA whose range holds many short
// segments streams fewer blocks. A segment cut by a range boundary leaves
// one piece per CTA it touches.
#pragma once

#include <stdint.h>

// The schedule is plain integer arithmetic, compiled for the host as well so
// that tests can check it against brute force without a GPU.
#define PKV_HD __host__ __device__

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

    PKV_HD void init(const int32_t* pre_, int batch, int kvh, long long a, long long b) {
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

    PKV_HD bool next(Piece& p) {
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

PKV_HD __forceinline__ long long range_start(long long c, long long U, long long C) { return c * U / C; }

// The same split weighted by cost: a segment of nb blocks costs nb + e(nb),
// e >= 0 being the work of a segment outside its blocks (loading q,
// combining the consumer warps' states, writing the row) that the ring of
// staged blocks does not hide; its first unit carries e, every unit costs 1.
// With K(u) the cost of the units before u and T = K(U), CTA c gets
// [start(c), start(c + 1)), start(c) being the first unit with
// K(u) >= floor(c T / C). e = 0 is the plain split. The block prefix sums
// pre[] and the cost prefix sums cost[] (per sequence, one KV head) locate a
// unit or a cost in O(log batch); max_unit bounds the cost of one unit.
struct CostSplit {
    const int32_t* pre;
    const int32_t* cost;
    int batch, kvh, max_unit;
    long long U, T, C;

    PKV_HD void init(const int32_t* pre_, const int32_t* cost_, int batch_, int kvh_, int max_unit_,
                     long long C_) {
        pre = pre_;
        cost = cost_;
        batch = batch_;
        kvh = kvh_;
        max_unit = max_unit_ > 1 ? max_unit_ : 1;
        C = C_;
        U = static_cast<long long>(kvh) * pre[batch - 1];
        T = static_cast<long long>(kvh) * cost[batch - 1];
    }
    // smallest i with kvh * arr[i] > x (arr non-decreasing, x < kvh * arr[batch - 1])
    PKV_HD int seq_of(const int32_t* arr, long long x) const {
        int lo = 0, hi = batch - 1;
        while (lo < hi) {
            const int mid = (lo + hi) >> 1;
            if (static_cast<long long>(kvh) * arr[mid] > x)
                hi = mid;
            else
                lo = mid + 1;
        }
        return lo;
    }
    // K(u) for 0 <= u <= U
    PKV_HD long long cost_before(long long u) const {
        if (T == U) return u;
        if (u >= U) return T;
        const int i = seq_of(pre, u);
        const int p0 = i ? pre[i - 1] : 0, q0 = i ? cost[i - 1] : 0;
        const int nb = pre[i] - p0, e = cost[i] - q0 - nb;
        const long long u0 = static_cast<long long>(kvh) * p0;
        const long long h = (u - u0) / nb, b = u - u0 - h * nb;
        return static_cast<long long>(kvh) * q0 + h * (nb + e) + (b > 0 ? e + b : 0);
    }
    PKV_HD long long start(long long c) const {
        const long long t = c * T / C;
        if (T == U) return t;
        if (t >= T) return U;
        const int i = seq_of(cost, t);
        const int p0 = i ? pre[i - 1] : 0, q0 = i ? cost[i - 1] : 0;
        const int nb = pre[i] - p0, e = cost[i] - q0 - nb;
        const long long k0 = static_cast<long long>(kvh) * q0;
        const long long h = (t - k0) / (nb + e), rr = t - k0 - h * (nb + e);
        const long long s0 = static_cast<long long>(kvh) * p0 + h * nb;
        return rr == 0 ? s0 : s0 + (rr - e > 1 ? rr - e : 1);
    }
    // the CTA whose range holds unit u: max c with start(c) <= u
    PKV_HD long long cta_of(long long u) const { return ((cost_before(u) + 1) * C - 1) / T; }
    // every range is non-empty when a range's cost share covers the dearest unit
    PKV_HD bool dense() const { return T >= C * max_unit; }
    // pieces of a segment whose units lie in CTAs c0 .. c1 (the non-empty ranges among them)
    PKV_HD int pieces(long long c0, long long c1) const {
        if (dense()) return static_cast<int>(c1 - c0 + 1);
        int n = 0;
        for (long long c = c0; c <= c1; ++c) n += start(c) < start(c + 1);
        return n;
    }
    // CTA of piece p of a segment whose first piece is in CTA c0
    PKV_HD long long piece_cta(long long c0, int p) const {
        if (dense()) return c0 + p;
        for (long long c = c0; c < C; ++c)
            if (start(c) < start(c + 1) && p-- == 0) return c;
        return C - 1;  // not reached for a valid piece index
    }
};

// The CTA whose range holds unit u: max c with range_start(c) <= u.
PKV_HD __forceinline__ long long cta_of(long long u, long long U, long long C) { return ((u + 1) * C - 1) / U; }

// Pieces of one segment: every CTA whose unit range meets [S0, S1).
PKV_HD __forceinline__ int pieces_of_segment(long long c0, long long c1, long long U, long long C) {
    if (U >= C) return static_cast<int>(c1 - c0 + 1);  // no CTA range is empty
    int n = 0;
    for (long long c = c0; c <= c1; ++c) n += range_start(c, U, C) < range_start(c + 1, U, C);
    return n;
}

// CTA holding piece p (0-based) of the segment that starts at unit S0 and
// whose first piece is in CTA c0. With at least one unit per CTA every range
// is non-empty, so pieces sit in consecutive CTAs; with fewer units than CTAs
// every non-empty range holds one unit, so piece p is unit S0 + p's CTA.
PKV_HD __forceinline__ long long piece_cta(long long S0, long long c0, int p, long long U, long long C) {
    return U >= C ? c0 + p : cta_of(S0 + p, U, C);
}

}  // namespace
}  // namespace pkv
