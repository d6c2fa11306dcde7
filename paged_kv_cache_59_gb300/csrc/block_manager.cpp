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
#include <cstdint>
#include <new>
#include <unordered_map>
#include <vector>

#include "../../include/pagedkv.h"

struct pa_bm {
    int block_size = 16;
    std::vector<int32_t> free_list;  // LIFO: back() is the next allocation
    std::vector<int32_t> ref;
    struct Seq {
        std::vector<int32_t> table;
        int64_t len = 0;
    };
    std::unordered_map<int64_t, Seq> seqs;

    int32_t alloc() {
        int32_t b = free_list.back();
        free_list.pop_back();
        ref[b] = 1;
        return b;
    }
    void put(int32_t b) {
        if (--ref[b] == 0) free_list.push_back(b);
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
    const int64_t bs = bm->block_size;
    if (n_cow_out) *n_cow_out = 0;
    // blocks this append needs: a copy of a shared, partially filled tail
    // plus enough fresh blocks for the tokens that do not fit
    bool tail_cow = n > 0 && (s.len % bs) != 0 && bm->ref[s.table.back()] > 1;
    int64_t have = (int64_t)s.table.size() * bs - s.len;
    int64_t extra = n - have;
    int64_t need = (tail_cow ? 1 : 0) + (extra > 0 ? (extra + bs - 1) / bs : 0);
    if (need > (int64_t)bm->free_list.size()) return PA_ERR_OOM;
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
    if (logical_block < 0 || logical_block >= (int)s.table.size()) return PA_ERR_INVALID_ARG;
    *n_out = 0;
    int32_t b = s.table[logical_block];
    if (b < 0) return PA_ERR_INVALID_ARG;  // released by the window
    if (bm->ref[b] <= 1) return PA_OK;
    if (bm->free_list.empty()) return PA_ERR_OOM;
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
    pa_bm::Seq c = it->second;  // copy before emplace may rehash
    for (int32_t b : c.table)
        if (b >= 0) bm->ref[b] += 1;
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
