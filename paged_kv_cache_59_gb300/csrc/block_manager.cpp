// Host block manager: free list, refcounts, fork aliasing and copy-on-write.
// It only builds tables, slots and copy pairs; no device work happens here.
//
// Rules (page title, section):
//  - "PagedAttention vs Traditional KV Cache", Section 4 "PagedAttention: How
//    It Works": a free list of block ids; appending a token takes a new block
//    only when the sequence's last block is full; an empty free list is the
//    caller's signal to preempt.
//  - "Inference serving: the KV-cache machine", section "Paged KV: virtual
//    memory for tokens": refcounted blocks freed at zero; a forked child's
//    table aliases the parent's blocks; the first divergent token gets a
//    private block.
//  - "Modern AI Infrastructure and Agentic System Design", 9.1, copy-on-write
//    figure: a write into a shared block copies it into a fresh one first.
//  - "KV Cache Explained Like You're an LLM Engineer", section "Sliding Window
//    Attention": with a window the cache a sequence needs stays O(W); blocks
//    wholly before the window are released (table entry -1, a hole) and
//    return to the free list when no table references them.
//  - "Modern AI Infrastructure and Agentic System Design", 9.1, part
//    "Batching and the scheduler", and "Inference serving: the KV-cache
//    machine", section "Paged KV: virtual memory for tokens" (and its Lab B
//    simulator): a preempted sequence's private blocks are swapped to host
//    memory and reloaded later into any free blocks. The private tail is the
//    longest run of trailing blocks only this table holds.
//  - "Modular LLM Inference Engine from Scratch", section "Prefix caching -
//    skip recomputing the same prompt": a hash-based LRU cache of prompt
//    prefixes; lookup returns the longest cached prefix of whole blocks and
//    refreshes it. An entry is one full block, identified by all the tokens
//    from position 0 through its last one; the cache holds one reference per
//    entry; an allocation that finds the free list empty evicts entries from
//    the least-recently-used end, skipping blocks a table still holds.
//
// A prefix is identified by a 128-bit hash chained over its tokens (two
// independent 64-bit chains, each token absorbed with the splitmix64
// finalizer of Steele, Lea and Flood); distinct prefixes collide with
// probability about 2^-128 per pair.
#include <cstdint>
#include <list>
#include <new>
#include <unordered_map>
#include <vector>

#include "../../include/pagedkv.h"

namespace {

uint64_t mix64(uint64_t z) {  // splitmix64 finalizer
    z = (z ^ (z >> 30)) * 0xbf58476d1ce4e5b9ull;
    z = (z ^ (z >> 27)) * 0x94d049bb133111ebull;
    return z ^ (z >> 31);
}

struct PrefixKey {
    uint64_t a, b;
    bool operator==(const PrefixKey& o) const { return a == o.a && b == o.b; }
};
struct PrefixKeyHash {
    size_t operator()(const PrefixKey& k) const { return (size_t)(k.a ^ (k.b * 0x9e3779b97f4a7c15ull)); }
};

// Extends the hash of a prefix by the tokens [t, t + n).
PrefixKey extend(PrefixKey h, const int32_t* t, int64_t n) {
    for (int64_t i = 0; i < n; ++i) {
        const uint64_t v = (uint64_t)(uint32_t)t[i];
        h.a = mix64(h.a ^ (v + 0x632be59bd9b4e019ull));
        h.b = mix64(h.b + v * 0xd6e8feb86659fd93ull + 0x8cb92ba72f3d8dd7ull);
    }
    return h;
}
constexpr PrefixKey kEmptyPrefix = {0x243f6a8885a308d3ull, 0x13198a2e03707344ull};

}  // namespace

struct pa_bm {
    int block_size = 16;
    std::vector<int32_t> free_list;  // LIFO: back() is the next allocation
    std::vector<int32_t> ref;        // table references + cache entries
    std::vector<uint8_t> cached;     // block has a cache entry
    int64_t evictable = 0;           // cache entries whose block only the cache holds
    struct Seq {
        std::vector<int32_t> table;
        int64_t len = 0;
        int64_t swapped = -1;  // >= 0: that many trailing blocks are in host memory
    };
    std::unordered_map<int64_t, Seq> seqs;
    struct Entry {
        PrefixKey key;
        int32_t block;
    };
    std::list<Entry> lru;  // front = least recently used
    std::unordered_map<PrefixKey, std::list<Entry>::iterator, PrefixKeyHash> index;

    void inc(int32_t b) {
        if (cached[b] && ref[b] == 1) --evictable;
        ++ref[b];
    }
    void put(int32_t b) {
        --ref[b];
        if (cached[b] && ref[b] == 1) ++evictable;
        if (ref[b] == 0) free_list.push_back(b);
    }
    int64_t available() const { return (int64_t)free_list.size() + evictable; }
    // Drops the least recently used entry whose block only the cache holds.
    bool evict_one() {
        for (auto it = lru.begin(); it != lru.end(); ++it) {
            const int32_t b = it->block;
            if (ref[b] != 1) continue;
            index.erase(it->key);
            lru.erase(it);
            cached[b] = 0;
            --evictable;
            put(b);  // 1 -> 0: back to the free list
            return true;
        }
        return false;
    }
    int32_t alloc() {  // callers check available() first
        if (free_list.empty()) evict_one();
        int32_t b = free_list.back();
        free_list.pop_back();
        ref[b] = 1;
        return b;
    }
};

extern "C" {

pa_bm* pa_bm_create(int num_blocks, int block_size) {
    if (num_blocks < 0 || block_size <= 0) return nullptr;
    pa_bm* bm = new (std::nothrow) pa_bm();
    if (!bm) return nullptr;
    try {
        bm->block_size = block_size;
        bm->ref.assign(num_blocks, 0);
        bm->cached.assign(num_blocks, 0);
        bm->free_list.resize(num_blocks);
        for (int i = 0; i < num_blocks; ++i) bm->free_list[i] = i;
    } catch (...) {
        delete bm;
        return nullptr;
    }
    return bm;
}

void pa_bm_destroy(pa_bm* bm) { delete bm; }

int pa_bm_add_seq(pa_bm* bm, int64_t seq_id) {
    if (!bm) return PA_ERR_INVALID_ARG;
    if (bm->seqs.count(seq_id)) return PA_ERR_REFCOUNT;
    bm->seqs.emplace(seq_id, pa_bm::Seq());
    return PA_OK;
}

int pa_bm_append_tokens(pa_bm* bm, int64_t seq_id, int n, int64_t* slots_out,
                        int64_t* cow_pairs_out, int cow_cap, int* n_cow_out) {
    if (!bm || n < 0 || (n > 0 && !slots_out)) return PA_ERR_INVALID_ARG;
    auto it = bm->seqs.find(seq_id);
    if (it == bm->seqs.end()) return PA_ERR_REFCOUNT;
    pa_bm::Seq& s = it->second;
    if (s.swapped >= 0) return PA_ERR_INVALID_ARG;  // swapped out
    const int64_t bs = bm->block_size;
    if (n_cow_out) *n_cow_out = 0;
    // blocks this append needs: a copy of a shared, partially filled tail
    // plus enough fresh blocks for the tokens that do not fit
    bool tail_cow = n > 0 && (s.len % bs) != 0 && bm->ref[s.table.back()] > 1;
    int64_t have = (int64_t)s.table.size() * bs - s.len;
    int64_t extra = n - have;
    int64_t need = (tail_cow ? 1 : 0) + (extra > 0 ? (extra + bs - 1) / bs : 0);
    if (need > bm->available()) return PA_ERR_OOM;
    if (tail_cow && (cow_cap < 1 || !cow_pairs_out || !n_cow_out)) return PA_ERR_CAPACITY;
    for (int i = 0; i < n; ++i) {
        int64_t L = s.len;
        if (L % bs == 0) {
            s.table.push_back(bm->alloc());
        } else {
            int32_t last = s.table[L / bs];
            if (bm->ref[last] > 1) {
                int32_t fresh = bm->alloc();
                cow_pairs_out[0] = last;
                cow_pairs_out[1] = fresh;
                *n_cow_out = 1;
                bm->put(last);
                s.table[L / bs] = fresh;
            }
        }
        slots_out[i] = (int64_t)s.table[L / bs] * bs + L % bs;
        s.len = L + 1;
    }
    return PA_OK;
}

int pa_bm_make_private(pa_bm* bm, int64_t seq_id, int logical_block, int64_t* pair_out,
                       int* n_out) {
    if (!bm || !pair_out || !n_out) return PA_ERR_INVALID_ARG;
    auto it = bm->seqs.find(seq_id);
    if (it == bm->seqs.end()) return PA_ERR_REFCOUNT;
    pa_bm::Seq& s = it->second;
    if (s.swapped >= 0) return PA_ERR_INVALID_ARG;
    if (logical_block < 0 || logical_block >= (int)s.table.size()) return PA_ERR_INVALID_ARG;
    *n_out = 0;
    int32_t b = s.table[logical_block];
    if (b < 0) return PA_ERR_INVALID_ARG;  // released by the window
    if (bm->ref[b] <= 1) return PA_OK;
    if (bm->available() < 1) return PA_ERR_OOM;
    int32_t fresh = bm->alloc();
    bm->put(b);
    s.table[logical_block] = fresh;
    pair_out[0] = b;
    pair_out[1] = fresh;
    *n_out = 1;
    return PA_OK;
}

int pa_bm_fork(pa_bm* bm, int64_t parent, int64_t child) {
    if (!bm) return PA_ERR_INVALID_ARG;
    auto it = bm->seqs.find(parent);
    if (it == bm->seqs.end() || bm->seqs.count(child)) return PA_ERR_REFCOUNT;
    if (it->second.swapped >= 0) return PA_ERR_INVALID_ARG;
    pa_bm::Seq c = it->second;  // copy before emplace may rehash
    for (int32_t b : c.table)
        if (b >= 0) bm->inc(b);
    bm->seqs.emplace(child, std::move(c));
    return PA_OK;
}

int pa_bm_free_seq(pa_bm* bm, int64_t seq_id) {
    if (!bm) return PA_ERR_INVALID_ARG;
    auto it = bm->seqs.find(seq_id);
    if (it == bm->seqs.end()) return PA_ERR_REFCOUNT;
    for (int32_t b : it->second.table) {
        if (b >= 0 && bm->ref[b] <= 0) return PA_ERR_REFCOUNT;  // cannot happen if state is consistent
    }
    for (int32_t b : it->second.table)
        if (b >= 0) bm->put(b);
    bm->seqs.erase(it);
    return PA_OK;
}

int pa_bm_release_before(pa_bm* bm, int64_t seq_id, int64_t first_pos, int* n_released_out) {
    if (!bm || !n_released_out) return PA_ERR_INVALID_ARG;
    auto it = bm->seqs.find(seq_id);
    if (it == bm->seqs.end()) return PA_ERR_REFCOUNT;
    pa_bm::Seq& s = it->second;
    if (s.swapped >= 0) return PA_ERR_INVALID_ARG;
    if (first_pos < 0) first_pos = 0;
    if (first_pos > s.len) first_pos = s.len;
    const int64_t whole = first_pos / bm->block_size;  // blocks wholly before first_pos
    int n = 0;
    for (int64_t j = 0; j < whole && j < (int64_t)s.table.size(); ++j) {
        if (s.table[j] >= 0) {
            bm->put(s.table[j]);
            s.table[j] = -1;
            ++n;
        }
    }
    *n_released_out = n;
    return PA_OK;
}

int pa_bm_swap_out(pa_bm* bm, int64_t seq_id, int32_t* blocks_out, int cap, int* n_out) {
    if (!bm || !n_out || cap < 0 || (cap > 0 && !blocks_out)) return PA_ERR_INVALID_ARG;
    auto it = bm->seqs.find(seq_id);
    if (it == bm->seqs.end()) return PA_ERR_REFCOUNT;
    pa_bm::Seq& s = it->second;
    if (s.swapped >= 0) return PA_ERR_INVALID_ARG;
    size_t k = s.table.size();
    while (k > 0 && s.table[k - 1] >= 0 && bm->ref[s.table[k - 1]] == 1) --k;
    const int n = (int)(s.table.size() - k);
    *n_out = n;
    if (n > cap) return PA_ERR_CAPACITY;  // nothing changed
    for (int i = 0; i < n; ++i) {
        blocks_out[i] = s.table[k + i];
        bm->put(s.table[k + i]);
    }
    s.table.resize(k);
    s.swapped = n;
    return PA_OK;
}

int pa_bm_swap_in(pa_bm* bm, int64_t seq_id, int32_t* blocks_out, int cap, int* n_out) {
    if (!bm || !n_out || cap < 0 || (cap > 0 && !blocks_out)) return PA_ERR_INVALID_ARG;
    auto it = bm->seqs.find(seq_id);
    if (it == bm->seqs.end()) return PA_ERR_REFCOUNT;
    pa_bm::Seq& s = it->second;
    if (s.swapped < 0) return PA_ERR_INVALID_ARG;  // not swapped out
    const int n = (int)s.swapped;
    *n_out = n;
    if (n > cap) return PA_ERR_CAPACITY;
    if (n > bm->available()) return PA_ERR_OOM;
    for (int i = 0; i < n; ++i) {
        const int32_t b = bm->alloc();
        s.table.push_back(b);
        blocks_out[i] = b;
    }
    s.swapped = -1;
    return PA_OK;
}

int pa_bm_cache_blocks(pa_bm* bm, int64_t seq_id, const int32_t* tokens, int64_t n_tokens,
                       int* n_added_out) {
    if (!bm || !n_added_out || n_tokens < 0 || (n_tokens > 0 && !tokens)) return PA_ERR_INVALID_ARG;
    auto it = bm->seqs.find(seq_id);
    if (it == bm->seqs.end()) return PA_ERR_REFCOUNT;
    const pa_bm::Seq& s = it->second;
    if (s.swapped >= 0) return PA_ERR_INVALID_ARG;
    const int64_t bs = bm->block_size;
    const int64_t n_full = (n_tokens < s.len ? n_tokens : s.len) / bs;
    int added = 0;
    PrefixKey h = kEmptyPrefix;
    try {
        for (int64_t j = 0; j < n_full; ++j) {
            h = extend(h, tokens + j * bs, bs);
            const int32_t b = s.table[j];
            if (b < 0 || bm->index.count(h)) continue;  // released, or already cached
            bm->lru.push_back({h, b});
            bm->index.emplace(h, std::prev(bm->lru.end()));
            bm->inc(b);  // held by the table too, so it is not evictable
            bm->cached[b] = 1;
            ++added;
        }
    } catch (...) {
        *n_added_out = added;
        return PA_ERR_OOM;
    }
    *n_added_out = added;
    return PA_OK;
}

int pa_bm_add_seq_cached(pa_bm* bm, int64_t seq_id, const int32_t* tokens, int64_t n_tokens,
                         int64_t* n_cached_out) {
    if (!bm || !n_cached_out || n_tokens < 0 || (n_tokens > 0 && !tokens)) return PA_ERR_INVALID_ARG;
    if (bm->seqs.count(seq_id)) return PA_ERR_REFCOUNT;
    const int64_t bs = bm->block_size;
    pa_bm::Seq s;
    PrefixKey h = kEmptyPrefix;
    for (int64_t j = 0; j < n_tokens / bs; ++j) {
        h = extend(h, tokens + j * bs, bs);
        auto f = bm->index.find(h);
        if (f == bm->index.end()) break;
        bm->lru.splice(bm->lru.end(), bm->lru, f->second);  // most recently used
        const int32_t b = f->second->block;
        bm->inc(b);
        s.table.push_back(b);
    }
    s.len = (int64_t)s.table.size() * bs;
    *n_cached_out = s.len;
    bm->seqs.emplace(seq_id, std::move(s));
    return PA_OK;
}

int pa_bm_num_cached(const pa_bm* bm) {
    if (!bm) return PA_ERR_INVALID_ARG;
    return (int)bm->lru.size();
}

int pa_bm_block_table(const pa_bm* bm, int64_t seq_id, int32_t* out, int cap, int* n_out) {
    if (!bm || !n_out || cap < 0 || (cap > 0 && !out)) return PA_ERR_INVALID_ARG;
    auto it = bm->seqs.find(seq_id);
    if (it == bm->seqs.end()) return PA_ERR_REFCOUNT;
    const auto& t = it->second.table;
    *n_out = (int)t.size();
    if ((int)t.size() > cap) return PA_ERR_CAPACITY;
    for (size_t i = 0; i < t.size(); ++i) out[i] = t[i];
    return PA_OK;
}

int64_t pa_bm_seq_len(const pa_bm* bm, int64_t seq_id) {
    if (!bm) return PA_ERR_INVALID_ARG;
    auto it = bm->seqs.find(seq_id);
    if (it == bm->seqs.end()) return PA_ERR_REFCOUNT;
    return it->second.len;
}

int pa_bm_num_free(const pa_bm* bm) {
    if (!bm) return PA_ERR_INVALID_ARG;
    return (int)bm->free_list.size();
}

int pa_bm_refcount(const pa_bm* bm, int block_id) {
    if (!bm) return PA_ERR_INVALID_ARG;
    if (block_id < 0 || block_id >= (int)bm->ref.size()) return PA_ERR_INVALID_ARG;
    return bm->ref[block_id];
}

int pa_bm_build_batch(const pa_bm* bm, const int64_t* seq_ids, int n, int max_blocks,
                      int32_t* tables_out, int32_t* context_lens_out) {
    if (!bm || n < 0 || max_blocks < 0 || (n > 0 && (!seq_ids || !context_lens_out)) ||
        (n > 0 && max_blocks > 0 && !tables_out))
        return PA_ERR_INVALID_ARG;
    for (int i = 0; i < n; ++i) {
        auto it = bm->seqs.find(seq_ids[i]);
        if (it == bm->seqs.end()) return PA_ERR_REFCOUNT;
        if (it->second.swapped >= 0) return PA_ERR_INVALID_ARG;
        if ((int)it->second.table.size() > max_blocks) return PA_ERR_CAPACITY;
    }
    for (int i = 0; i < n; ++i) {
        const auto& s = bm->seqs.find(seq_ids[i])->second;
        int32_t* row = tables_out + (size_t)i * max_blocks;
        for (int j = 0; j < max_blocks; ++j) row[j] = j < (int)s.table.size() ? s.table[j] : -1;
        context_lens_out[i] = (int32_t)s.len;
    }
    return PA_OK;
}

}  // extern "C"
