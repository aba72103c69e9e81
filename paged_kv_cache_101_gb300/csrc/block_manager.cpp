// block_manager.cpp -- host-side block manager of the paged KV pool (see
// include/pkv_block_manager.h for the contract and the passages it follows).
//
// State: one reference count per physical block, a LIFO free list, and per
// live sequence its length and block table. Every entry point takes the
// manager's mutex. Calls that can fail for lack of blocks count what they need
// first and change nothing unless all of it is available.
#include <limits.h>
#include <stdint.h>

#include <mutex>
#include <new>
#include <unordered_map>
#include <unordered_set>
#include <vector>

#include "pkv_block_manager.h"

namespace {

constexpr int64_t kBs = 16;

int64_t blocks_for(int64_t tokens) { return tokens / kBs + (tokens % kBs != 0); }

struct Sequence {
    int64_t length = 0;
    std::vector<int32_t> blocks;
};

}  // namespace

struct pkv_block_manager {
    mutable std::mutex mu;
    int64_t num_blocks = 0;
    std::vector<int32_t> refcount;
    std::vector<int32_t> free_list;  // back() is handed out next
    std::unordered_map<int64_t, Sequence> seqs;

    int32_t take()
    {
        const int32_t b = free_list.back();
        free_list.pop_back();
        refcount[b] = 1;
        return b;
    }
    void release(int32_t b)
    {
        if (--refcount[b] == 0)
            free_list.push_back(b);
    }
};

extern "C" {

pkv_block_manager *pkv_bm_create(int64_t num_blocks)
{
    if (num_blocks < 1 || num_blocks > INT32_MAX)
        return nullptr;
    pkv_block_manager *bm = new (std::nothrow) pkv_block_manager;
    if (!bm)
        return nullptr;
    try {
        bm->num_blocks = num_blocks;
        bm->refcount.assign(size_t(num_blocks), 0);
        bm->free_list.resize(size_t(num_blocks));
        for (int64_t i = 0; i < num_blocks; ++i)
            bm->free_list[size_t(i)] = int32_t(num_blocks - 1 - i);
    } catch (const std::bad_alloc &) {
        delete bm;
        return nullptr;
    }
    return bm;
}

void pkv_bm_destroy(pkv_block_manager *bm) { delete bm; }

int64_t pkv_bm_num_free(const pkv_block_manager *bm)
{
    if (!bm)
        return -1;
    std::lock_guard<std::mutex> lk(bm->mu);
    return int64_t(bm->free_list.size());
}

int64_t pkv_bm_num_blocks(const pkv_block_manager *bm) { return bm ? bm->num_blocks : -1; }

int64_t pkv_bm_num_sequences(const pkv_block_manager *bm)
{
    if (!bm)
        return -1;
    std::lock_guard<std::mutex> lk(bm->mu);
    return int64_t(bm->seqs.size());
}

int32_t pkv_bm_refcount(const pkv_block_manager *bm, int64_t block)
{
    if (!bm || block < 0 || block >= bm->num_blocks)
        return -1;
    std::lock_guard<std::mutex> lk(bm->mu);
    return bm->refcount[size_t(block)];
}

pkv_status pkv_bm_add_sequence(pkv_block_manager *bm, int64_t seq_id, int64_t num_tokens)
{
    if (!bm)
        return PKV_ERR_NULL;
    if (num_tokens < 0)
        return PKV_ERR_SHAPE;
    std::lock_guard<std::mutex> lk(bm->mu);
    if (bm->seqs.count(seq_id))
        return PKV_ERR_SEQUENCE;
    const int64_t need = blocks_for(num_tokens);
    if (need > int64_t(bm->free_list.size()))
        return PKV_ERR_NO_BLOCKS;
    try {
        Sequence s;
        s.length = num_tokens;
        s.blocks.reserve(size_t(need));
        auto it = bm->seqs.emplace(seq_id, std::move(s)).first;
        for (int64_t i = 0; i < need; ++i)
            it->second.blocks.push_back(bm->take());
    } catch (const std::bad_alloc &) {
        auto it = bm->seqs.find(seq_id);
        if (it != bm->seqs.end()) {
            for (int32_t b : it->second.blocks)
                bm->release(b);
            bm->seqs.erase(it);
        }
        return PKV_ERR_RANGE;
    }
    return PKV_OK;
}

pkv_status pkv_bm_fork(pkv_block_manager *bm, int64_t parent_id, int64_t child_id)
{
    if (!bm)
        return PKV_ERR_NULL;
    std::lock_guard<std::mutex> lk(bm->mu);
    auto p = bm->seqs.find(parent_id);
    if (p == bm->seqs.end() || parent_id == child_id || bm->seqs.count(child_id))
        return PKV_ERR_SEQUENCE;
    for (int32_t b : p->second.blocks)
        if (bm->refcount[b] == INT32_MAX)
            return PKV_ERR_RANGE;
    try {
        Sequence c = p->second;  // copy before the map may rehash
        bm->seqs.emplace(child_id, std::move(c));
    } catch (const std::bad_alloc &) {
        return PKV_ERR_RANGE;
    }
    for (int32_t b : bm->seqs[child_id].blocks)
        ++bm->refcount[b];
    return PKV_OK;
}

pkv_status pkv_bm_free_sequence(pkv_block_manager *bm, int64_t seq_id)
{
    if (!bm)
        return PKV_ERR_NULL;
    std::lock_guard<std::mutex> lk(bm->mu);
    auto it = bm->seqs.find(seq_id);
    if (it == bm->seqs.end())
        return PKV_ERR_SEQUENCE;
    for (int32_t b : it->second.blocks)
        bm->release(b);
    bm->seqs.erase(it);
    return PKV_OK;
}

pkv_status pkv_bm_append(pkv_block_manager *bm, const int64_t *seq_ids, int32_t num_seqs,
                         int32_t n_per_seq, int64_t *slot_mapping, int32_t *copy_src,
                         int32_t *copy_dst, int32_t *num_copies)
{
    if (!bm)
        return PKV_ERR_NULL;
    if (num_seqs < 0 || n_per_seq < 0)
        return PKV_ERR_SHAPE;
    if (num_seqs == 0 || n_per_seq == 0) {
        if (num_copies)
            *num_copies = 0;
        return PKV_OK;
    }
    if (!seq_ids || !slot_mapping || !copy_src || !copy_dst || !num_copies)
        return PKV_ERR_NULL;
    std::lock_guard<std::mutex> lk(bm->mu);

    // 1. resolve the ids and count the blocks the whole call takes
    std::vector<Sequence *> seq;
    std::unordered_set<int64_t> seen;
    std::unordered_map<int32_t, int32_t> released;  // shared block -> sharers that copy away
    int64_t need = 0;
    try {
        seq.resize(size_t(num_seqs));
        seen.reserve(size_t(num_seqs));
        for (int32_t i = 0; i < num_seqs; ++i) {
            auto it = bm->seqs.find(seq_ids[i]);
            if (it == bm->seqs.end() || !seen.insert(seq_ids[i]).second)
                return PKV_ERR_SEQUENCE;
            Sequence &s = it->second;
            seq[size_t(i)] = &s;
            const int64_t L = s.length;
            need += blocks_for(L + n_per_seq) - blocks_for(L);
            if (L % kBs != 0) {
                const int32_t last = s.blocks.back();
                int32_t &gone = released[last];
                if (bm->refcount[last] - gone > 1) {
                    ++need;  // private copy of the shared last block
                    ++gone;
                }
            }
        }
    } catch (const std::bad_alloc &) {
        return PKV_ERR_RANGE;
    }
    if (need > int64_t(bm->free_list.size()))
        return PKV_ERR_NO_BLOCKS;
    try {
        for (Sequence *s : seq)
            s->blocks.reserve(size_t(blocks_for(s->length + n_per_seq)));
    } catch (const std::bad_alloc &) {
        return PKV_ERR_RANGE;
    }

    // 2. place every token (cannot fail from here on)
    int32_t nc = 0;
    for (int32_t i = 0; i < num_seqs; ++i) {
        Sequence &s = *seq[size_t(i)];
        for (int32_t t = 0; t < n_per_seq; ++t) {
            const int64_t pos = s.length;
            if (pos % kBs == 0) {
                s.blocks.push_back(bm->take());
            } else {
                int32_t &last = s.blocks.back();
                if (bm->refcount[last] > 1) {
                    const int32_t fresh = bm->take();
                    copy_src[nc] = last;
                    copy_dst[nc] = fresh;
                    ++nc;
                    --bm->refcount[last];  // still >= 1: another sharer holds it
                    last = fresh;
                }
            }
            slot_mapping[int64_t(i) * n_per_seq + t] =
                int64_t(s.blocks[size_t(pos / kBs)]) * kBs + pos % kBs;
            s.length = pos + 1;
        }
    }
    *num_copies = nc;
    return PKV_OK;
}

int64_t pkv_bm_sequence_length(const pkv_block_manager *bm, int64_t seq_id)
{
    if (!bm)
        return -1;
    std::lock_guard<std::mutex> lk(bm->mu);
    auto it = bm->seqs.find(seq_id);
    return it == bm->seqs.end() ? -1 : it->second.length;
}

int64_t pkv_bm_sequence_blocks(const pkv_block_manager *bm, int64_t seq_id, int32_t *blocks,
                               int64_t capacity)
{
    if (!bm)
        return -1;
    std::lock_guard<std::mutex> lk(bm->mu);
    auto it = bm->seqs.find(seq_id);
    if (it == bm->seqs.end())
        return -1;
    const std::vector<int32_t> &t = it->second.blocks;
    const int64_t n = int64_t(t.size());
    if (blocks)
        for (int64_t i = 0; i < n && i < capacity; ++i)
            blocks[i] = t[size_t(i)];
    return n;
}

pkv_status pkv_bm_block_tables(const pkv_block_manager *bm, const int64_t *seq_ids,
                               int32_t num_seqs, int32_t *block_tables,
                               int32_t max_blocks_per_seq, int32_t *context_lens)
{
    if (!bm)
        return PKV_ERR_NULL;
    if (num_seqs < 0 || max_blocks_per_seq < 0)
        return PKV_ERR_SHAPE;
    if (num_seqs == 0)
        return PKV_OK;
    if (!seq_ids || !context_lens || (max_blocks_per_seq > 0 && !block_tables))
        return PKV_ERR_NULL;
    std::lock_guard<std::mutex> lk(bm->mu);
    for (int32_t i = 0; i < num_seqs; ++i) {
        auto it = bm->seqs.find(seq_ids[i]);
        if (it == bm->seqs.end())
            return PKV_ERR_SEQUENCE;
        if (int64_t(it->second.blocks.size()) > max_blocks_per_seq ||
            it->second.length > INT32_MAX)
            return PKV_ERR_RANGE;
    }
    for (int32_t i = 0; i < num_seqs; ++i) {
        const Sequence &s = bm->seqs.find(seq_ids[i])->second;
        int32_t *row = block_tables + int64_t(i) * max_blocks_per_seq;
        const int32_t n = int32_t(s.blocks.size());
        for (int32_t j = 0; j < max_blocks_per_seq; ++j)
            row[j] = j < n ? s.blocks[size_t(j)] : -1;
        context_lens[i] = int32_t(s.length);
    }
    return PKV_OK;
}

int32_t pkv_bm_check(const pkv_block_manager *bm)
{
    if (!bm)
        return -1;
    std::lock_guard<std::mutex> lk(bm->mu);
    int32_t bad = 0;
    std::vector<int64_t> holders(size_t(bm->num_blocks), 0);
    for (const auto &kv : bm->seqs) {
        const Sequence &s = kv.second;
        if (int64_t(s.blocks.size()) != blocks_for(s.length))
            bad |= 16;
        for (int32_t b : s.blocks)
            ++holders[size_t(b)];
    }
    int64_t held = 0;
    for (int64_t b = 0; b < bm->num_blocks; ++b) {
        if (holders[size_t(b)] != bm->refcount[size_t(b)])
            bad |= 1;
        held += holders[size_t(b)] > 0;
    }
    std::vector<uint8_t> in_free(size_t(bm->num_blocks), 0);
    for (int32_t b : bm->free_list) {
        if (in_free[size_t(b)])
            bad |= 2;
        in_free[size_t(b)] = 1;
        if (holders[size_t(b)] > 0)
            bad |= 4;
    }
    if (held + int64_t(bm->free_list.size()) != bm->num_blocks)
        bad |= 8;
    return bad;
}

}  // extern "C"
