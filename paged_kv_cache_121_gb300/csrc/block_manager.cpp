// Host KV block manager: free queue, cdiv allocation, reference counts and
// copy-on-write decisions.
//
// Follows "Paged Attention: Virtual Memory for the KV Cache", sections
// "Paging: blocks handed out as tokens arrive" and "Inside vLLM: the block
// pool" (front-of-queue allocation, null block 0, freed blocks to the front),
// "PagedAttention, explained.", procedure steps 1-4 and 6, and
// "PagedAttention: KV cache virtual memory", section "Copy-on-write".
//
// The free queue is an intrusive doubly linked list over block ids (O(1)
// pop-front / push-front / unlink), the same shape of structure the pages
// describe for vLLM's pool; tables are per-sequence vectors in a hash map.
#include <algorithm>
#include <cstdint>
#include <new>
#include <unordered_map>
#include <vector>

#include "../../include/pa.h"

namespace {

struct Sequence {
    std::vector<int32_t> table;
    int64_t tokens = 0;
};

}  // namespace

struct pa_bm {
    int num_blocks = 0;
    int block_size = 0;
    bool null_reserved = false;
    // free queue as a linked list of block ids; -1 terminates
    std::vector<int32_t> next, prev;
    std::vector<uint8_t> on_queue;
    int32_t head = -1, tail = -1;
    int64_t free_count = 0;
    std::vector<int32_t> refcount;
    std::unordered_map<int64_t, Sequence> seqs;
    int64_t cow_copies = 0;

    void push_back(int32_t b) {
        prev[b] = tail;
        next[b] = -1;
        if (tail >= 0) next[tail] = b; else head = b;
        tail = b;
        on_queue[b] = 1;
        ++free_count;
    }
    void push_front(int32_t b) {
        next[b] = head;
        prev[b] = -1;
        if (head >= 0) prev[head] = b; else tail = b;
        head = b;
        on_queue[b] = 1;
        ++free_count;
    }
    int32_t pop_front() {
        int32_t b = head;
        head = next[b];
        if (head >= 0) prev[head] = -1; else tail = -1;
        on_queue[b] = 0;
        --free_count;
        refcount[b] = 1;
        return b;
    }
};

static pa_status bm_init(pa_bm *bm, int num_blocks, int block_size) {
    bm->num_blocks = num_blocks;
    bm->block_size = block_size;
    bm->next.assign(num_blocks, -1);
    bm->prev.assign(num_blocks, -1);
    bm->on_queue.assign(num_blocks, 0);
    bm->refcount.assign(num_blocks, 0);
    return PA_OK;
}

extern "C" {

PA_API pa_status pa_bm_create(int num_blocks, int block_size, int reserve_null_block, pa_bm **out) {
    if (!out || num_blocks <= 0 || block_size <= 0) return PA_ERR_INVALID_ARG;
    *out = nullptr;
    pa_bm *bm = new (std::nothrow) pa_bm();
    if (!bm) return PA_ERR_INVALID_ARG;
    bm_init(bm, num_blocks, block_size);
    bm->null_reserved = reserve_null_block != 0;
    for (int b = bm->null_reserved ? 1 : 0; b < num_blocks; ++b) bm->push_back(b);
    *out = bm;
    return PA_OK;
}

PA_API pa_status pa_bm_create_with_free_list(int num_blocks, int block_size,
                                             const int32_t *free_order, int n, pa_bm **out) {
    if (!out || num_blocks <= 0 || block_size <= 0 || n < 0 || n > num_blocks ||
        (n > 0 && !free_order))
        return PA_ERR_INVALID_ARG;
    *out = nullptr;
    pa_bm *bm = new (std::nothrow) pa_bm();
    if (!bm) return PA_ERR_INVALID_ARG;
    bm_init(bm, num_blocks, block_size);
    for (int i = 0; i < n; ++i) {
        int32_t b = free_order[i];
        if (b < 0 || b >= num_blocks || bm->on_queue[b]) {
            delete bm;
            return PA_ERR_INVALID_ARG;
        }
        bm->push_back(b);
    }
    bm->null_reserved = false;
    *out = bm;
    return PA_OK;
}

PA_API void pa_bm_destroy(pa_bm *bm) { delete bm; }

PA_API pa_status pa_bm_allocate(pa_bm *bm, int64_t seq, int num_tokens) {
    if (!bm || num_tokens < 0) return PA_ERR_INVALID_ARG;
    if (bm->seqs.count(seq)) return PA_ERR_INVALID_ARG;
    const int64_t need = (static_cast<int64_t>(num_tokens) + bm->block_size - 1) / bm->block_size;
    if (need > bm->free_count) return PA_ERR_OUT_OF_BLOCKS;
    Sequence s;
    s.table.reserve(static_cast<size_t>(need));
    for (int64_t i = 0; i < need; ++i) s.table.push_back(bm->pop_front());
    s.tokens = num_tokens;
    bm->seqs.emplace(seq, std::move(s));
    return PA_OK;
}

PA_API pa_status pa_bm_append_slot(pa_bm *bm, int64_t seq, int64_t *slot, int64_t *cow_src,
                                   int64_t *cow_dst) {
    if (!bm || !slot) return PA_ERR_INVALID_ARG;
    auto it = bm->seqs.find(seq);
    if (it == bm->seqs.end()) return PA_ERR_NOT_FOUND;
    Sequence &s = it->second;
    const int64_t pos = s.tokens;
    const int64_t logical = pos / bm->block_size;
    const int64_t offset = pos % bm->block_size;
    int64_t src = -1, dst = -1;
    if (logical >= static_cast<int64_t>(s.table.size())) {
        // the last block is full (or there is none): take a fresh one
        if (bm->free_count == 0) return PA_ERR_OUT_OF_BLOCKS;
        s.table.push_back(bm->pop_front());
    } else {
        const int32_t last = s.table[static_cast<size_t>(logical)];
        if (bm->refcount[last] > 1) {
            // shared block about to be written: clone it, repoint only this table
            if (bm->free_count == 0) return PA_ERR_OUT_OF_BLOCKS;
            const int32_t fresh = bm->pop_front();
            --bm->refcount[last];
            s.table[static_cast<size_t>(logical)] = fresh;
            src = last;
            dst = fresh;
            ++bm->cow_copies;
        }
    }
    *slot = static_cast<int64_t>(s.table[static_cast<size_t>(logical)]) * bm->block_size + offset;
    if (cow_src) *cow_src = src;
    if (cow_dst) *cow_dst = dst;
    s.tokens = pos + 1;
    return PA_OK;
}

PA_API pa_status pa_bm_fork(pa_bm *bm, int64_t parent, int64_t child) {
    if (!bm) return PA_ERR_INVALID_ARG;
    auto it = bm->seqs.find(parent);
    if (it == bm->seqs.end()) return PA_ERR_NOT_FOUND;
    if (bm->seqs.count(child)) return PA_ERR_INVALID_ARG;
    Sequence s = it->second;  // copy: table and token count
    for (int32_t b : s.table) ++bm->refcount[b];
    bm->seqs.emplace(child, std::move(s));
    return PA_OK;
}

PA_API pa_status pa_bm_free(pa_bm *bm, int64_t seq) {
    if (!bm) return PA_ERR_INVALID_ARG;
    auto it = bm->seqs.find(seq);
    if (it == bm->seqs.end()) return PA_ERR_NOT_FOUND;
    const std::vector<int32_t> &table = it->second.table;
    for (int32_t b : table) --bm->refcount[b];
    // released blocks go to the queue front, keeping their table order
    for (auto r = table.rbegin(); r != table.rend(); ++r)
        if (bm->refcount[*r] == 0 && !bm->on_queue[*r]) bm->push_front(*r);
    bm->seqs.erase(it);
    return PA_OK;
}

PA_API pa_status pa_bm_block_table(const pa_bm *bm, int64_t seq, int32_t *out, int cap, int *n) {
    if (!bm || !n) return PA_ERR_INVALID_ARG;
    auto it = bm->seqs.find(seq);
    if (it == bm->seqs.end()) return PA_ERR_NOT_FOUND;
    const std::vector<int32_t> &t = it->second.table;
    *n = static_cast<int>(t.size());
    if (cap < *n || (*n > 0 && !out)) return PA_ERR_INVALID_ARG;
    std::copy(t.begin(), t.end(), out);
    return PA_OK;
}

PA_API pa_status pa_bm_num_tokens(const pa_bm *bm, int64_t seq, int *n) {
    if (!bm || !n) return PA_ERR_INVALID_ARG;
    auto it = bm->seqs.find(seq);
    if (it == bm->seqs.end()) return PA_ERR_NOT_FOUND;
    *n = static_cast<int>(it->second.tokens);
    return PA_OK;
}

PA_API pa_status pa_bm_refcount(const pa_bm *bm, int block, int *refcount) {
    if (!bm || !refcount || block < 0 || block >= bm->num_blocks) return PA_ERR_INVALID_ARG;
    *refcount = bm->refcount[block];
    return PA_OK;
}

PA_API pa_status pa_bm_stats(const pa_bm *bm, pa_bm_stats_t *out) {
    if (!bm || !out) return PA_ERR_INVALID_ARG;
    pa_bm_stats_t s{};
    s.num_blocks = bm->num_blocks - (bm->null_reserved ? 1 : 0);
    s.free_blocks = bm->free_count;
    for (int32_t r : bm->refcount) {
        if (r >= 1) ++s.used_blocks;
        if (r >= 2) ++s.shared_blocks;
    }
    s.num_seqs = static_cast<int64_t>(bm->seqs.size());
    for (const auto &kv : bm->seqs) {
        s.logical_blocks += static_cast<int64_t>(kv.second.table.size());
        s.num_tokens += kv.second.tokens;
    }
    s.waste_slots = s.logical_blocks * bm->block_size - s.num_tokens;
    s.cow_copies = bm->cow_copies;
    *out = s;
    return PA_OK;
}

PA_API pa_status pa_bm_free_list(const pa_bm *bm, int32_t *out, int cap, int *n) {
    if (!bm || !n) return PA_ERR_INVALID_ARG;
    *n = static_cast<int>(bm->free_count);
    if (cap < *n || (*n > 0 && !out)) return PA_ERR_INVALID_ARG;
    int i = 0;
    for (int32_t b = bm->head; b >= 0; b = bm->next[b]) out[i++] = b;
    return PA_OK;
}

PA_API pa_status pa_compute_slot_mapping(int64_t *slot_mapping, const int32_t *block_tables,
                                         int num_seqs, int max_blocks_per_seq,
                                         const int32_t *seq_index, const int32_t *positions,
                                         int num_tokens, int block_size) {
    if (num_tokens < 0 || num_seqs < 0 || max_blocks_per_seq < 0 || block_size <= 0)
        return PA_ERR_INVALID_ARG;
    if (num_tokens == 0) return PA_OK;
    if (!slot_mapping || !block_tables || !seq_index || !positions) return PA_ERR_INVALID_ARG;
    for (int i = 0; i < num_tokens; ++i) {
        const int32_t s = seq_index[i];
        const int32_t p = positions[i];
        if (p < 0) {
            slot_mapping[i] = -1;
            continue;
        }
        if (s < 0 || s >= num_seqs || p / block_size >= max_blocks_per_seq) return PA_ERR_INVALID_ARG;
        const int64_t blk = block_tables[static_cast<int64_t>(s) * max_blocks_per_seq + p / block_size];
        slot_mapping[i] = blk * block_size + p % block_size;
    }
    return PA_OK;
}

}  // extern "C"
