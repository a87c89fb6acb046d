// Host-side block pool (page table) of the paged KV cache.
//
// Behaviour follows "Notebook 10. KV cache and serving: bytes, pages, and
// ceilings", section 5 ("Page pool: prefix sharing and copy-on-write"):
// reference-counted physical blocks on a last-in-first-out free stack,
// allocation preflighted so a failed append changes nothing, copy-on-write of
// a shared partial final block, release returning unreferenced blocks. Where
// the notebook's simulator recomputes per-block fills after every change,
// this pool keeps only what the hot path needs (lengths, tables, reference
// counts, the free stack) and derives fills when statistics or a validation
// are asked for.
#include <algorithm>
#include <new>
#include <unordered_map>
#include <vector>

#include "pkv.h"

struct pkv_pool {
    int64_t total_blocks = 0;
    int32_t block_size = 16;
    std::vector<int32_t> refs;          // references per physical block
    std::vector<int32_t> free_stack;    // pops from the back
    std::vector<uint8_t> is_free;       // membership of free_stack
    struct Seq {
        int64_t length = 0;
        std::vector<int32_t> blocks;
    };
    std::unordered_map<int64_t, Seq> seqs;
};

namespace {

int32_t pop_block(pkv_pool* p) {
    const int32_t b = p->free_stack.back();
    p->free_stack.pop_back();
    p->is_free[b] = 0;
    p->refs[b] = 1;
    return b;
}

void push_block(pkv_pool* p, int32_t b) {
    p->free_stack.push_back(b);
    p->is_free[b] = 1;
}

// Blocks an append of `count` tokens to `s` takes from the free stack.
int64_t blocks_needed(const pkv_pool* p, const pkv_pool::Seq& s, int64_t count) {
    if (count == 0) return 0;
    const int64_t B = p->block_size;
    const int64_t used = s.length % B;
    int64_t room = 0, need = 0;
    if (!s.blocks.empty() && used) {
        room = B - used;
        if (p->refs[s.blocks.back()] > 1) need += 1;  // private replacement of the shared partial block
    }
    const int64_t overflow = count > room ? count - room : 0;
    return need + (overflow + B - 1) / B;
}

pkv_status do_append(pkv_pool* p, int64_t seq, int64_t count, int64_t* slots_out, int64_t* pair_out,
                     int32_t* num_pairs) {
    if (num_pairs) *num_pairs = 0;
    if (count < 0) return PKV_ERR_SHAPE;
    auto it = p->seqs.find(seq);
    if (it == p->seqs.end()) return PKV_ERR_UNKNOWN_SEQUENCE;
    pkv_pool::Seq& s = it->second;
    if (blocks_needed(p, s, count) > static_cast<int64_t>(p->free_stack.size())) return PKV_ERR_OUT_OF_BLOCKS;
    if (count == 0) return PKV_OK;
    const int64_t B = p->block_size;
    const int64_t start = s.length;
    const int64_t used = s.length % B;
    if (!s.blocks.empty() && used) {
        int32_t last = s.blocks.back();
        if (p->refs[last] > 1) {
            p->refs[last] -= 1;
            const int32_t fresh = pop_block(p);
            s.blocks.back() = fresh;
            if (pair_out) {
                pair_out[0] = last;
                pair_out[1] = fresh;
            }
            if (num_pairs) *num_pairs = 1;
        }
    }
    // the new tokens fill the last block's room, then whole new blocks
    int64_t left = count;
    const int64_t room = (!s.blocks.empty() && used) ? B - used : 0;
    int64_t take = std::min(left, room);
    s.length += take;
    left -= take;
    while (left > 0) {
        take = std::min(left, B);
        s.blocks.push_back(pop_block(p));
        s.length += take;
        left -= take;
    }
    if (slots_out)
        for (int64_t t = start; t < start + count; ++t) slots_out[t - start] = s.blocks[t / B] * B + t % B;
    return PKV_OK;
}

// Per-block fill: the most slots any sharer still covers.
std::vector<int64_t> fills(const pkv_pool* p) {
    std::vector<int64_t> f(p->total_blocks, 0);
    const int64_t B = p->block_size;
    for (const auto& kv : p->seqs) {
        const auto& s = kv.second;
        for (size_t j = 0; j < s.blocks.size(); ++j) {
            const int64_t covered = std::min<int64_t>(B, s.length - static_cast<int64_t>(j) * B);
            f[s.blocks[j]] = std::max(f[s.blocks[j]], covered);
        }
    }
    return f;
}

}  // namespace

extern "C" {

pkv_status pkv_pool_create(int64_t total_blocks, int32_t block_size, const int64_t* pop_order, pkv_pool** out) {
    if (out == nullptr) return PKV_ERR_NULL;
    *out = nullptr;
    if (total_blocks < 1 || total_blocks >= (int64_t(1) << 31) || block_size < 1) return PKV_ERR_SHAPE;
    pkv_pool* p = new (std::nothrow) pkv_pool;
    if (p == nullptr) return PKV_ERR_OUT_OF_BLOCKS;
    p->total_blocks = total_blocks;
    p->block_size = block_size;
    p->refs.assign(total_blocks, 0);
    p->is_free.assign(total_blocks, 0);
    p->free_stack.reserve(total_blocks);
    if (pop_order) {
        std::vector<uint8_t> seen(total_blocks, 0);
        for (int64_t i = 0; i < total_blocks; ++i) {
            const int64_t b = pop_order[i];
            if (b < 0 || b >= total_blocks || seen[b]) {
                delete p;
                return PKV_ERR_RANGE;
            }
            seen[b] = 1;
        }
        for (int64_t i = total_blocks - 1; i >= 0; --i) push_block(p, static_cast<int32_t>(pop_order[i]));
    } else {
        for (int64_t i = total_blocks - 1; i >= 0; --i) push_block(p, static_cast<int32_t>(i));
    }
    *out = p;
    return PKV_OK;
}

void pkv_pool_destroy(pkv_pool* pool) { delete pool; }

pkv_status pkv_pool_add_sequence(pkv_pool* pool, int64_t seq) {
    if (pool == nullptr) return PKV_ERR_NULL;
    if (pool->seqs.count(seq)) return PKV_ERR_EXISTS;
    pool->seqs.emplace(seq, pkv_pool::Seq{});
    return PKV_OK;
}

pkv_status pkv_pool_append(pkv_pool* pool, int64_t seq, int64_t tokens, int64_t* slots_out, int64_t* copy_pair_out,
                           int32_t* num_pairs_out) {
    if (pool == nullptr) return PKV_ERR_NULL;
    return do_append(pool, seq, tokens, slots_out, copy_pair_out, num_pairs_out);
}

pkv_status pkv_pool_append_batch(pkv_pool* pool, const int64_t* seqs, const int64_t* tokens, int64_t n,
                                 int64_t* slots_out, int64_t* pairs_out, int64_t* num_pairs_out,
                                 int64_t* num_done_out) {
    if (num_pairs_out) *num_pairs_out = 0;
    if (num_done_out) *num_done_out = 0;
    if (pool == nullptr) return PKV_ERR_NULL;
    if (n < 0) return PKV_ERR_SHAPE;
    if (n > 0 && (seqs == nullptr || tokens == nullptr)) return PKV_ERR_NULL;
    int64_t slot_pos = 0, npairs = 0;
    for (int64_t i = 0; i < n; ++i) {
        int64_t pair[2];
        int32_t got = 0;
        const pkv_status st = do_append(pool, seqs[i], tokens[i], slots_out ? slots_out + slot_pos : nullptr, pair,
                                        &got);
        if (st != PKV_OK) return st;
        if (got && pairs_out) {
            pairs_out[2 * npairs] = pair[0];
            pairs_out[2 * npairs + 1] = pair[1];
        }
        npairs += got;
        slot_pos += tokens[i];
        if (num_pairs_out) *num_pairs_out = npairs;
        if (num_done_out) *num_done_out = i + 1;
    }
    return PKV_OK;
}

pkv_status pkv_pool_share_prefix(pkv_pool* pool, int64_t source, int64_t target, int64_t prefix_tokens) {
    if (pool == nullptr) return PKV_ERR_NULL;
    auto it = pool->seqs.find(source);
    if (it == pool->seqs.end()) return PKV_ERR_UNKNOWN_SEQUENCE;
    if (prefix_tokens < 0 || prefix_tokens > it->second.length) return PKV_ERR_SHAPE;
    if (pool->seqs.count(target)) return PKV_ERR_EXISTS;
    const int64_t nb = (prefix_tokens + pool->block_size - 1) / pool->block_size;
    pkv_pool::Seq t;
    t.length = prefix_tokens;
    t.blocks.assign(it->second.blocks.begin(), it->second.blocks.begin() + nb);
    for (int32_t b : t.blocks) pool->refs[b] += 1;
    pool->seqs.emplace(target, std::move(t));
    return PKV_OK;
}

pkv_status pkv_pool_release(pkv_pool* pool, int64_t seq) {
    if (pool == nullptr) return PKV_ERR_NULL;
    auto it = pool->seqs.find(seq);
    if (it == pool->seqs.end()) return PKV_ERR_UNKNOWN_SEQUENCE;
    for (int32_t b : it->second.blocks)
        if (--pool->refs[b] == 0) push_block(pool, b);
    pool->seqs.erase(it);
    return PKV_OK;
}

pkv_status pkv_pool_sequence_length(const pkv_pool* pool, int64_t seq, int64_t* length_out) {
    if (pool == nullptr || length_out == nullptr) return PKV_ERR_NULL;
    auto it = pool->seqs.find(seq);
    if (it == pool->seqs.end()) return PKV_ERR_UNKNOWN_SEQUENCE;
    *length_out = it->second.length;
    return PKV_OK;
}

pkv_status pkv_pool_page_table(const pkv_pool* pool, int64_t seq, int32_t* table_out, int64_t capacity,
                               int64_t* num_blocks_out) {
    if (pool == nullptr || num_blocks_out == nullptr) return PKV_ERR_NULL;
    auto it = pool->seqs.find(seq);
    if (it == pool->seqs.end()) return PKV_ERR_UNKNOWN_SEQUENCE;
    const auto& b = it->second.blocks;
    *num_blocks_out = static_cast<int64_t>(b.size());
    if (static_cast<int64_t>(b.size()) > capacity) return PKV_ERR_SHAPE;
    if (!b.empty() && table_out == nullptr) return PKV_ERR_NULL;
    std::copy(b.begin(), b.end(), table_out);
    return PKV_OK;
}

pkv_status pkv_pool_block_tables(const pkv_pool* pool, const int64_t* seqs, int64_t n, int32_t* tables_out,
                                 int64_t width, int32_t* lens_out) {
    if (pool == nullptr) return PKV_ERR_NULL;
    if (n < 0 || width < 1) return PKV_ERR_SHAPE;
    if (n > 0 && (seqs == nullptr || tables_out == nullptr || lens_out == nullptr)) return PKV_ERR_NULL;
    for (int64_t i = 0; i < n; ++i) {  // check everything before writing
        auto it = pool->seqs.find(seqs[i]);
        if (it == pool->seqs.end()) return PKV_ERR_UNKNOWN_SEQUENCE;
        if (static_cast<int64_t>(it->second.blocks.size()) > width || it->second.length >= (int64_t(1) << 31))
            return PKV_ERR_SHAPE;
    }
    for (int64_t i = 0; i < n; ++i) {
        const auto& s = pool->seqs.find(seqs[i])->second;
        int32_t* row = tables_out + i * width;
        std::fill(row, row + width, -1);
        std::copy(s.blocks.begin(), s.blocks.end(), row);
        lens_out[i] = static_cast<int32_t>(s.length);
    }
    return PKV_OK;
}

pkv_status pkv_pool_get_stats(const pkv_pool* pool, pkv_pool_stats* out) {
    if (pool == nullptr || out == nullptr) return PKV_ERR_NULL;
    const std::vector<int64_t> f = fills(pool);
    int64_t payload = 0, logical = 0;
    for (int64_t b = 0; b < pool->total_blocks; ++b)
        if (pool->refs[b]) payload += f[b];
    for (const auto& kv : pool->seqs) logical += kv.second.length;
    out->total_blocks = pool->total_blocks;
    out->free_blocks = static_cast<int64_t>(pool->free_stack.size());
    out->allocated_blocks = pool->total_blocks - out->free_blocks;
    out->physical_capacity_tokens = out->allocated_blocks * pool->block_size;
    out->physical_payload_tokens = payload;
    out->logical_tokens = logical;
    out->internal_waste_tokens = out->physical_capacity_tokens - payload;
    out->sharing_savings_tokens = logical - payload;
    out->sequences = static_cast<int64_t>(pool->seqs.size());
    return PKV_OK;
}

pkv_status pkv_pool_validate(const pkv_pool* pool) {
    if (pool == nullptr) return PKV_ERR_NULL;
    const int64_t N = pool->total_blocks, B = pool->block_size;
    std::vector<uint8_t> on_stack(N, 0);
    for (int32_t b : pool->free_stack) {
        if (b < 0 || b >= N || on_stack[b]) return PKV_ERR_INVARIANT;
        on_stack[b] = 1;
    }
    std::vector<int32_t> refs(N, 0);
    for (const auto& kv : pool->seqs) {
        const auto& s = kv.second;
        if (s.length < 0) return PKV_ERR_INVARIANT;
        if (static_cast<int64_t>(s.blocks.size()) != (s.length + B - 1) / B) return PKV_ERR_INVARIANT;
        std::vector<int32_t> sorted(s.blocks);
        std::sort(sorted.begin(), sorted.end());
        if (std::adjacent_find(sorted.begin(), sorted.end()) != sorted.end()) return PKV_ERR_INVARIANT;
        for (int32_t b : s.blocks) {
            if (b < 0 || b >= N) return PKV_ERR_INVARIANT;
            ++refs[b];
        }
    }
    const std::vector<int64_t> f = fills(pool);
    int64_t payload = 0, logical = 0;
    for (int64_t b = 0; b < N; ++b) {
        if (refs[b] != pool->refs[b] || on_stack[b] != pool->is_free[b]) return PKV_ERR_INVARIANT;
        if (refs[b] == 0) {
            if (!on_stack[b]) return PKV_ERR_INVARIANT;
        } else {
            if (on_stack[b] || f[b] < 1 || f[b] > B) return PKV_ERR_INVARIANT;
            payload += f[b];
        }
    }
    for (const auto& kv : pool->seqs) logical += kv.second.length;
    if (logical < payload) return PKV_ERR_INVARIANT;
    return PKV_OK;
}

}  // extern "C"
