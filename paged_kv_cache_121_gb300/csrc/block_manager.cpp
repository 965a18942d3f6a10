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
//
// Swapping ("PagedAttention, explained.", procedure steps 7-8; "What Does
// PagedAttention Actually Optimize?", section 12): an optional CPU pool with
// its own free queue. A group of sequences that holds every reference to its
// blocks (a request's beams, say) is moved out (its blocks re-homed in the
// CPU pool, the GPU blocks freed) and back in (fresh GPU blocks); the caller
// moves the data with pa_swap_blocks using the returned pairs.
#include <algorithm>
#include <cstdint>
#include <new>
#include <unordered_map>
#include <vector>

#include "../../include/pa.h"

namespace {

struct Sequence {
    std::vector<int32_t> table;   // device block ids, or host block ids while swapped out
    int64_t tokens = 0;
    bool swapped = false;
};

// A free queue of block ids: a doubly linked list over the ids, O(1)
// pop-front / push-front / push-back. Used for the GPU pool and the CPU pool.
struct FreeQueue {
    std::vector<int32_t> next, prev;
    std::vector<uint8_t> on_queue;
    int32_t head = -1, tail = -1;
    int64_t count = 0;

    void init(int n) {
        next.assign(n, -1);
        prev.assign(n, -1);
        on_queue.assign(n, 0);
        head = tail = -1;
        count = 0;
    }
    void push_back(int32_t b) {
        prev[b] = tail;
        next[b] = -1;
        if (tail >= 0) next[tail] = b; else head = b;
        tail = b;
        on_queue[b] = 1;
        ++count;
    }
    void push_front(int32_t b) {
        next[b] = head;
        prev[b] = -1;
        if (head >= 0) prev[head] = b; else tail = b;
        head = b;
        on_queue[b] = 1;
        ++count;
    }
    int32_t pop_front() {
        int32_t b = head;
        head = next[b];
        if (head >= 0) prev[head] = -1; else tail = -1;
        on_queue[b] = 0;
        --count;
        return b;
    }
};

}  // namespace

struct pa_bm {
    int num_blocks = 0;
    int block_size = 0;
    bool null_reserved = false;
    FreeQueue q;                      // GPU blocks
    std::vector<int32_t> refcount;
    std::unordered_map<int64_t, Sequence> seqs;
    int64_t cow_copies = 0;
    // CPU pool for swapped-out sequences (empty until pa_bm_enable_swap)
    FreeQueue hq;
    std::vector<int32_t> host_refcount;
    int64_t swapped_seqs = 0;

    void push_back(int32_t b) { q.push_back(b); }
    void push_front(int32_t b) { q.push_front(b); }
    int32_t pop_front() {
        const int32_t b = q.pop_front();
        refcount[b] = 1;
        return b;
    }
};

static pa_status bm_init(pa_bm *bm, int num_blocks, int block_size) {
    bm->num_blocks = num_blocks;
    bm->block_size = block_size;
    bm->q.init(num_blocks);
    bm->refcount.assign(num_blocks, 0);
    return PA_OK;
}

// Distinct blocks of a group of sequences' tables, in order of first
// appearance, with the number of references the group holds on each.
static void group_blocks(const std::vector<Sequence *> &group, std::vector<int32_t> &order,
                         std::unordered_map<int32_t, int32_t> &refs) {
    for (Sequence *s : group)
        for (int32_t b : s->table)
            if (refs[b]++ == 0) order.push_back(b);
}

// The sequences named by ids (each once, each present, each in the given
// swap state), or an error status.
static pa_status collect_group(pa_bm *bm, const int64_t *ids, int n, bool swapped, std::vector<Sequence *> &group) {
    if (n < 0 || (n > 0 && !ids)) return PA_ERR_INVALID_ARG;
    std::unordered_map<int64_t, int> seen;
    for (int i = 0; i < n; ++i) {
        auto it = bm->seqs.find(ids[i]);
        if (it == bm->seqs.end()) return PA_ERR_NOT_FOUND;
        if (it->second.swapped != swapped || seen[ids[i]]++) return PA_ERR_INVALID_ARG;
        group.push_back(&it->second);
    }
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
        if (b < 0 || b >= num_blocks || bm->q.on_queue[b]) {
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
    if (need > bm->q.count) return PA_ERR_OUT_OF_BLOCKS;
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
    if (s.swapped) return PA_ERR_INVALID_ARG;   // swap it in first
    const int64_t pos = s.tokens;
    const int64_t logical = pos / bm->block_size;
    const int64_t offset = pos % bm->block_size;
    int64_t src = -1, dst = -1;
    if (logical >= static_cast<int64_t>(s.table.size())) {
        // the last block is full (or there is none): take a fresh one
        if (bm->q.count == 0) return PA_ERR_OUT_OF_BLOCKS;
        s.table.push_back(bm->pop_front());
    } else {
        const int32_t last = s.table[static_cast<size_t>(logical)];
        if (bm->refcount[last] > 1) {
            // shared block about to be written: clone it, repoint only this table
            if (bm->q.count == 0) return PA_ERR_OUT_OF_BLOCKS;
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
    if (bm->seqs.count(child) || it->second.swapped) return PA_ERR_INVALID_ARG;
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
    if (it->second.swapped) {   // its blocks live in the CPU pool
        for (int32_t b : table) --bm->host_refcount[b];
        for (auto r = table.rbegin(); r != table.rend(); ++r)
            if (bm->host_refcount[*r] == 0 && !bm->hq.on_queue[*r]) bm->hq.push_front(*r);
        --bm->swapped_seqs;
        bm->seqs.erase(it);
        return PA_OK;
    }
    for (int32_t b : table) --bm->refcount[b];
    // released blocks go to the queue front, keeping their table order
    for (auto r = table.rbegin(); r != table.rend(); ++r)
        if (bm->refcount[*r] == 0 && !bm->q.on_queue[*r]) bm->push_front(*r);
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
    s.free_blocks = bm->q.count;
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
    *n = static_cast<int>(bm->q.count);
    if (cap < *n || (*n > 0 && !out)) return PA_ERR_INVALID_ARG;
    int i = 0;
    for (int32_t b = bm->q.head; b >= 0; b = bm->q.next[b]) out[i++] = b;
    return PA_OK;
}

PA_API pa_status pa_bm_enable_swap(pa_bm *bm, int num_host_blocks) {
    if (!bm || num_host_blocks <= 0 || bm->hq.next.size() != 0) return PA_ERR_INVALID_ARG;
    bm->hq.init(num_host_blocks);
    bm->host_refcount.assign(num_host_blocks, 0);
    for (int b = 0; b < num_host_blocks; ++b) bm->hq.push_back(b);
    return PA_OK;
}

// Move a group of sequences (all holders of their blocks) between the pools.
// out: to the CPU pool (pairs: GPU id, CPU id); else back (CPU id, GPU id).
static pa_status swap_group(pa_bm *bm, const int64_t *seqs, int n, bool out, int64_t *mapping, int cap,
                            int *num_pairs) {
    if (!bm || !num_pairs || bm->hq.next.empty()) return PA_ERR_INVALID_ARG;
    std::vector<Sequence *> group;
    pa_status st = collect_group(bm, seqs, n, !out, group);
    if (st != PA_OK) return st;
    std::vector<int32_t> order;
    std::unordered_map<int32_t, int32_t> refs;
    group_blocks(group, order, refs);
    std::vector<int32_t> &src_ref = out ? bm->refcount : bm->host_refcount;
    for (int32_t b : order)
        if (src_ref[b] != refs[b]) return PA_ERR_INVALID_ARG;   // a sequence outside the group holds it
    FreeQueue &dst_q = out ? bm->hq : bm->q;
    FreeQueue &src_q = out ? bm->q : bm->hq;
    std::vector<int32_t> &dst_ref = out ? bm->host_refcount : bm->refcount;
    if (static_cast<int64_t>(order.size()) > dst_q.count) return PA_ERR_OUT_OF_BLOCKS;
    if (cap < static_cast<int>(order.size()) || (!order.empty() && !mapping)) return PA_ERR_INVALID_ARG;
    std::unordered_map<int32_t, int32_t> moved;
    for (size_t i = 0; i < order.size(); ++i) {
        const int32_t from = order[i];
        const int32_t to = dst_q.pop_front();
        dst_ref[to] = src_ref[from];
        src_ref[from] = 0;
        moved[from] = to;
        mapping[2 * i] = from;
        mapping[2 * i + 1] = to;
    }
    // released blocks go to the front of their queue, in the order collected
    for (auto r = order.rbegin(); r != order.rend(); ++r) src_q.push_front(*r);
    for (Sequence *s : group) {
        for (int32_t &b : s->table) b = moved[b];
        s->swapped = out;
    }
    bm->swapped_seqs += out ? n : -n;
    *num_pairs = static_cast<int>(order.size());
    return PA_OK;
}

PA_API pa_status pa_bm_swap_out(pa_bm *bm, const int64_t *seqs, int num_seqs, int64_t *mapping, int cap,
                                int *num_pairs) {
    return swap_group(bm, seqs, num_seqs, true, mapping, cap, num_pairs);
}

PA_API pa_status pa_bm_swap_in(pa_bm *bm, const int64_t *seqs, int num_seqs, int64_t *mapping, int cap,
                               int *num_pairs) {
    return swap_group(bm, seqs, num_seqs, false, mapping, cap, num_pairs);
}

PA_API pa_status pa_bm_is_swapped(const pa_bm *bm, int64_t seq, int *swapped) {
    if (!bm || !swapped) return PA_ERR_INVALID_ARG;
    auto it = bm->seqs.find(seq);
    if (it == bm->seqs.end()) return PA_ERR_NOT_FOUND;
    *swapped = it->second.swapped ? 1 : 0;
    return PA_OK;
}

PA_API pa_status pa_bm_swap_stats(const pa_bm *bm, int64_t *host_blocks, int64_t *free_host_blocks,
                                  int64_t *swapped_seqs) {
    if (!bm || !host_blocks || !free_host_blocks || !swapped_seqs) return PA_ERR_INVALID_ARG;
    *host_blocks = static_cast<int64_t>(bm->host_refcount.size());
    *free_host_blocks = bm->hq.count;
    *swapped_seqs = bm->swapped_seqs;
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
