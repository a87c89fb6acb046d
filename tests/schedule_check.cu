// Host-side check of the split schedule in pkv_schedule.cuh (the code the
// kernels run, compiled for the host) against brute force over random length
// mixes: the cost-weighted split (CostSplit), the equal split (range_start and
// the helpers of the multi-query kernels) and the piece walker. Prints
// "ok <cases>" or the first mismatch, and exits non-zero on a mismatch.
#include <cstdio>
#include <cstdlib>
#include <vector>

#include "pkv_schedule.cuh"

using namespace pkv;

namespace {

unsigned long long g_state = 0x9e3779b97f4a7c15ull;
int rnd(int n) {  // splitmix64, then reduced to [0, n)
    g_state += 0x9e3779b97f4a7c15ull;
    unsigned long long z = g_state;
    z = (z ^ (z >> 30)) * 0xbf58476d1ce4e5b9ull;
    z = (z ^ (z >> 27)) * 0x94d049bb133111ebull;
    z ^= z >> 31;
    return static_cast<int>(z % static_cast<unsigned long long>(n));
}

int g_fail = 0;
#define CHECK(cond, ...)                                  \
    do {                                                  \
        if (!(cond)) {                                    \
            if (g_fail++ < 5) {                           \
                std::printf("mismatch: " __VA_ARGS__);    \
                std::printf("\n");                        \
            }                                             \
        }                                                 \
    } while (0)

// A length mix with empty sequences, one-block sequences and long ones.
std::vector<int> random_blocks(int batch) {
    std::vector<int> nb(batch);
    for (int i = 0; i < batch; ++i) {
        const int kind = rnd(6);
        nb[i] = kind == 0 ? 0 : kind == 1 ? 1 : kind == 2 ? 2 + rnd(6) : kind == 3 ? 20 + rnd(60) : 1 + rnd(300);
    }
    nb[rnd(batch)] = 1 + rnd(40);  // at least one sequence with blocks
    return nb;
}

// The pieces of every CTA's range, concatenated in CTA order, must cover
// every segment exactly once and in order, with the fields the kernels use.
template <class StartFn>
void check_walk(const std::vector<int32_t>& pre, const std::vector<int>& nb, int kvh, long long C, StartFn start) {
    const int batch = static_cast<int>(pre.size());
    long long next_unit = 0;
    for (long long c = 0; c < C; ++c) {
        const long long a = start(c), b = start(c + 1);
        Walker wk;
        wk.init(pre.data(), batch, kvh, a, b);
        Piece pc;
        bool first = true;
        long long u = a;
        while (wk.next(pc)) {
            const long long units_before_seq = static_cast<long long>(kvh) * (pc.seq ? pre[pc.seq - 1] : 0);
            CHECK(pc.seg_len == nb[pc.seq] && pc.seg_len > 0, "walker segment length (seq %d)", pc.seq);
            CHECK(pc.seg_start == units_before_seq + static_cast<long long>(pc.head) * pc.seg_len,
                  "walker segment start (seq %d head %d)", pc.seq, pc.head);
            CHECK(pc.seg_start + pc.blk_from == u, "walker piece start (cta %lld)", c);
            CHECK(pc.blk_from < pc.blk_to && pc.blk_to <= pc.seg_len, "walker piece bounds (cta %lld)", c);
            CHECK(pc.complete == (pc.blk_from == 0 && pc.blk_to == pc.seg_len), "walker complete flag");
            CHECK(pc.first == first, "walker first flag");
            first = false;
            u = pc.seg_start + pc.blk_to;
        }
        CHECK(u == b, "walker stops at the range end (cta %lld: %lld vs %lld)", c, u, b);
        next_unit = b;
    }
    CHECK(next_unit == static_cast<long long>(kvh) * pre.back(), "ranges cover every unit");
}

void one_case(int kvh, int batch, long long C, int cost_add, int cost_below, int min_cost) {
    const std::vector<int> nb = random_blocks(batch);
    std::vector<int32_t> pre(batch), cost(batch);
    int extra_max = 0;
    for (int i = 0, p = 0, q = 0; i < batch; ++i) {
        const int e = nb[i] == 0 ? 0 : (nb[i] < cost_below ? cost_add : 0) + (min_cost > nb[i] ? min_cost - nb[i] : 0);
        extra_max = e > extra_max ? e : extra_max;
        p += nb[i];
        q += nb[i] ? nb[i] + e : 0;
        pre[i] = p;
        cost[i] = q;
    }
    // ---- the cost-weighted split against brute force
    CostSplit sp;
    sp.init(pre.data(), cost.data(), batch, kvh, 1 + (cost_add > 0 ? cost_add : 0) + (min_cost > 1 ? min_cost - 1 : 0), C);
    std::vector<long long> K(1, 0);  // K[u]: cost of the units before u
    for (int i = 0; i < batch; ++i)
        for (int h = 0; h < kvh; ++h)
            for (int j = 0; j < nb[i]; ++j) {
                const int e = j == 0 ? (cost[i] - (i ? cost[i - 1] : 0)) - nb[i] : 0;
                K.push_back(K.back() + 1 + e);
            }
    const long long U = static_cast<long long>(K.size()) - 1;
    CHECK(U == sp.U && K.back() == sp.T, "totals");
    for (long long u = 0; u <= U; ++u) CHECK(sp.cost_before(u) == K[u], "cost_before(%lld)", u);
    std::vector<long long> st(C + 1);
    for (long long c = 0; c <= C; ++c) {
        const long long t = c * sp.T / C;
        long long want = 0;
        while (want < U && K[want] < t) ++want;
        st[c] = sp.start(c);
        CHECK(st[c] == want, "start(%lld) = %lld, want %lld", c, st[c], want);
    }
    for (long long u = 0; u < U; ++u) {
        long long want = 0;
        for (long long c = 0; c < C; ++c)
            if (st[c] <= u) want = c;
        CHECK(sp.cta_of(u) == want, "cta_of(%lld)", u);
    }
    if (sp.dense())
        for (long long c = 0; c < C; ++c) CHECK(st[c] < st[c + 1], "dense split with an empty range %lld", c);
    // pieces of every segment: the non-empty ranges that meet it, in order
    for (int i = 0; i < batch; ++i)
        for (int h = 0; h < kvh && nb[i] > 0; ++h) {
            const long long s0 = static_cast<long long>(kvh) * (i ? pre[i - 1] : 0) + static_cast<long long>(h) * nb[i];
            const long long s1 = s0 + nb[i];
            const long long c0 = sp.cta_of(s0), c1 = sp.cta_of(s1 - 1);
            std::vector<long long> ctas;
            for (long long c = 0; c < C; ++c)
                if (st[c] < st[c + 1] && st[c] < s1 && st[c + 1] > s0) ctas.push_back(c);
            CHECK(sp.pieces(c0, c1) == static_cast<int>(ctas.size()), "pieces of segment at %lld", s0);
            for (int p = 0; p < static_cast<int>(ctas.size()); ++p)
                CHECK(sp.piece_cta(c0, p) == ctas[p], "piece_cta(%lld, %d)", c0, p);
        }
    check_walk(pre, nb, kvh, C, [&](long long c) { return sp.start(c); });
    // ---- the equal split of the multi-query kernels against brute force
    for (long long u = 0; u < U; ++u) {
        long long want = 0;
        for (long long c = 0; c < C; ++c)
            if (range_start(c, U, C) <= u) want = c;
        CHECK(cta_of(u, U, C) == want, "equal split cta_of(%lld)", u);
    }
    for (int i = 0; i < batch; ++i)
        for (int h = 0; h < kvh && nb[i] > 0; ++h) {
            const long long s0 = static_cast<long long>(kvh) * (i ? pre[i - 1] : 0) + static_cast<long long>(h) * nb[i];
            const long long s1 = s0 + nb[i];
            const long long c0 = cta_of(s0, U, C), c1 = cta_of(s1 - 1, U, C);
            std::vector<long long> ctas;
            for (long long c = 0; c < C; ++c) {
                const long long a = range_start(c, U, C), b = range_start(c + 1, U, C);
                if (a < b && a < s1 && b > s0) ctas.push_back(c);
            }
            CHECK(pieces_of_segment(c0, c1, U, C) == static_cast<int>(ctas.size()), "equal split pieces at %lld", s0);
            for (int p = 0; p < static_cast<int>(ctas.size()); ++p)
                CHECK(piece_cta(s0, c0, p, U, C) == ctas[p], "equal split piece_cta(%lld, %d)", s0, p);
        }
    check_walk(pre, nb, kvh, C, [&](long long c) { return range_start(c, U, C); });
}

}  // namespace

int main() {
    const int kvhs[] = {1, 2, 8};
    const long long ctas[] = {1, 2, 3, 7, 19, 64, 304, 700};
    int cases = 0;
    for (int trial = 0; trial < 400; ++trial) {
        const int kvh = kvhs[rnd(3)];
        const int batch = 1 + rnd(12);
        const long long C = ctas[rnd(8)];
        const int mode = rnd(4);  // equal split, the decode kernels' model, a least cost, both
        const int cost_add = mode == 1 || mode == 3 ? 1 + rnd(8) : 0;
        const int cost_below = mode == 1 || mode == 3 ? 1 + rnd(300) : 0;
        const int min_cost = mode >= 2 ? 1 + rnd(20) : 1;
        one_case(kvh, batch, C, cost_add, cost_below, min_cost);
        ++cases;
    }
    if (g_fail) {
        std::printf("FAILED: %d mismatches\n", g_fail);
        return 1;
    }
    std::printf("ok %d\n", cases);
    return 0;
}
