// block_manager.cpp -- host-side block manager: the bookkeeping that produces
// the device calls' inputs (block tables, context lengths, slot mappings and
// copy-on-write pairs).
//
// Follows "KV Cache与PagedAttention深度解析" §5.2-5.3 (free block pool; when
// token t is appended a sequence needs ceil((t+1)/block_size) blocks, a new
// block is taken from the pool when the table is short, and the token goes to
// offset t % block_size of the last block), §6.2 (blocks of finished requests
// return to the pool) and §8.2-8.3 (blocks shared between sequences carry a
// reference count; a block is freed when its count reaches zero), plus the
// copy-on-write rule of the nano-vllm article (zwxr.cn) §2.3 / §5.5: a
// sequence about to write into a block that another sequence also references
// first gets a private copy.  An exhausted pool is an error, as in the
// PyTorch PagedKVCache sketch of "KV Cache从原理到实战" §6.2.
//
// Not thread-safe: one manager belongs to one scheduling thread.
#include <algorithm>
#include <cstdint>
#include <unordered_map>
#include <vector>

#include "../../include/pagedkv.h"

struct pkv_block_manager {
    int64_t num_blocks = 0;
    int block_size = 0;
    int max_blocks_per_seq = 0;
    std::vector<int32_t> free_stack;   // top = back(); initial order hands out 0, 1, 2, ...
    std::vector<int32_t> refcount;     // per physical block
    struct Seq {
        std::vector<int32_t> table;
        int64_t len = 0;
    };
    std::unordered_map<int64_t, Seq> seqs;

    int32_t take_block() {
        const int32_t b = free_stack.back();
        free_stack.pop_back();
        refcount[b] = 1;
        return b;
    }
    void release_block(int32_t b) {
        if (--refcount[b] == 0) free_stack.push_back(b);
    }
};

namespace {

pkv_block_manager::Seq *find(pkv_block_manager *bm, int64_t id) {
    auto it = bm->seqs.find(id);
    return it == bm->seqs.end() ? nullptr : &it->second;
}

}  // namespace

extern "C" {

PKV_API pkv_block_manager *pkv_bm_create(int64_t num_blocks, int block_size,
                                         int max_blocks_per_seq) {
    if (num_blocks <= 0 || num_blocks > 0x7fffffffLL || block_size <= 0 || max_blocks_per_seq <= 0)
        return nullptr;
    auto *bm = new pkv_block_manager();
    bm->num_blocks = num_blocks;
    bm->block_size = block_size;
    bm->max_blocks_per_seq = max_blocks_per_seq;
    bm->refcount.assign(static_cast<size_t>(num_blocks), 0);
    bm->free_stack.reserve(static_cast<size_t>(num_blocks));
    for (int64_t b = num_blocks - 1; b >= 0; --b) bm->free_stack.push_back(static_cast<int32_t>(b));
    return bm;
}

PKV_API void pkv_bm_destroy(pkv_block_manager *bm) { delete bm; }

PKV_API int64_t pkv_bm_num_free(const pkv_block_manager *bm) {
    return bm ? static_cast<int64_t>(bm->free_stack.size()) : -1;
}

PKV_API int32_t pkv_bm_refcount(const pkv_block_manager *bm, int64_t block) {
    if (!bm || block < 0 || block >= bm->num_blocks) return -1;
    return bm->refcount[static_cast<size_t>(block)];
}

PKV_API pkv_status pkv_bm_add_sequence(pkv_block_manager *bm, int64_t seq_id) {
    if (!bm || bm->seqs.count(seq_id)) return PKV_ERR_INVALID_ARG;
    bm->seqs.emplace(seq_id, pkv_block_manager::Seq{});
    return PKV_OK;
}

PKV_API pkv_status pkv_bm_fork(pkv_block_manager *bm, int64_t parent_id, int64_t child_id) {
    if (!bm || bm->seqs.count(child_id)) return PKV_ERR_INVALID_ARG;
    pkv_block_manager::Seq *parent = find(bm, parent_id);
    if (!parent) return PKV_ERR_INVALID_ARG;
    pkv_block_manager::Seq child = *parent;  // same physical blocks
    for (int32_t b : child.table) ++bm->refcount[b];
    bm->seqs.emplace(child_id, std::move(child));
    return PKV_OK;
}

PKV_API pkv_status pkv_bm_share_prefix(pkv_block_manager *bm, int64_t src_id, int64_t dst_id,
                                       int64_t num_tokens) {
    if (!bm) return PKV_ERR_INVALID_ARG;
    pkv_block_manager::Seq *src = find(bm, src_id);
    pkv_block_manager::Seq *dst = find(bm, dst_id);
    if (!src || !dst || src == dst || dst->len != 0 || num_tokens < 0 || num_tokens > src->len ||
        num_tokens % bm->block_size != 0 || num_tokens / bm->block_size > bm->max_blocks_per_seq)
        return PKV_ERR_INVALID_ARG;
    const int64_t nblk = num_tokens / bm->block_size;
    dst->table.assign(src->table.begin(), src->table.begin() + nblk);
    for (int32_t b : dst->table) ++bm->refcount[b];
    dst->len = num_tokens;
    return PKV_OK;
}

PKV_API pkv_status pkv_bm_append_token(pkv_block_manager *bm, int64_t seq_id, int64_t *slot,
                                       int64_t *cow_src, int64_t *cow_dst) {
    if (!bm || !slot || !cow_src || !cow_dst) return PKV_ERR_INVALID_ARG;
    pkv_block_manager::Seq *s = find(bm, seq_id);
    if (!s) return PKV_ERR_INVALID_ARG;
    const int64_t t = s->len;                             // position of the new token
    const int64_t need = (t + 1 + bm->block_size - 1) / bm->block_size;
    *cow_src = *cow_dst = -1;
    if (need > bm->max_blocks_per_seq) return PKV_ERR_INVALID_ARG;
    if (static_cast<int64_t>(s->table.size()) < need) {
        if (bm->free_stack.empty()) return PKV_ERR_OUT_OF_BLOCKS;
        s->table.push_back(bm->take_block());
    } else {
        const int32_t last = s->table.back();
        if (bm->refcount[last] > 1) {                     // shared: copy before writing
            if (bm->free_stack.empty()) return PKV_ERR_OUT_OF_BLOCKS;
            const int32_t fresh = bm->take_block();
            bm->release_block(last);
            s->table.back() = fresh;
            *cow_src = last;
            *cow_dst = fresh;
        }
    }
    *slot = static_cast<int64_t>(s->table[static_cast<size_t>(t / bm->block_size)]) * bm->block_size +
            t % bm->block_size;
    s->len = t + 1;
    return PKV_OK;
}

PKV_API pkv_status pkv_bm_free_sequence(pkv_block_manager *bm, int64_t seq_id) {
    if (!bm) return PKV_ERR_INVALID_ARG;
    auto it = bm->seqs.find(seq_id);
    if (it == bm->seqs.end()) return PKV_ERR_INVALID_ARG;
    for (int32_t b : it->second.table) bm->release_block(b);
    bm->seqs.erase(it);
    return PKV_OK;
}

PKV_API int64_t pkv_bm_seq_len(const pkv_block_manager *bm, int64_t seq_id) {
    if (!bm) return -1;
    auto it = bm->seqs.find(seq_id);
    return it == bm->seqs.end() ? -1 : it->second.len;
}

PKV_API pkv_status pkv_bm_block_table(const pkv_block_manager *bm, int64_t seq_id, int32_t *out,
                                      int capacity, int *num_entries) {
    if (!bm || !num_entries) return PKV_ERR_INVALID_ARG;
    auto it = bm->seqs.find(seq_id);
    if (it == bm->seqs.end()) return PKV_ERR_INVALID_ARG;
    const auto &tab = it->second.table;
    *num_entries = static_cast<int>(tab.size());
    if (static_cast<int>(tab.size()) > capacity || (!out && !tab.empty())) return PKV_ERR_INVALID_ARG;
    std::copy(tab.begin(), tab.end(), out);
    return PKV_OK;
}

PKV_API pkv_status pkv_bm_decode_step(pkv_block_manager *bm, const int64_t *seq_ids,
                                      int num_seqs, int64_t *slot_mapping,
                                      int32_t *block_tables, int32_t *context_lens,
                                      int64_t *cow_pairs, int64_t *num_cow_pairs) {
    if (!bm || num_seqs < 0 || !num_cow_pairs || (num_seqs > 0 && (!seq_ids || !slot_mapping ||
                                                                   !block_tables || !context_lens ||
                                                                   !cow_pairs)))
        return PKV_ERR_INVALID_ARG;
    std::unordered_map<int64_t, int> seen;
    for (int i = 0; i < num_seqs; ++i)
        if (!find(bm, seq_ids[i]) || seen[seq_ids[i]]++) return PKV_ERR_INVALID_ARG;
    // Check that the pool covers this step before changing anything: replay the
    // step's allocations on scratch reference counts (a block shared by several
    // sequences of the batch is copied by all but the last one to write).
    int64_t demand = 0;
    std::unordered_map<int32_t, int32_t> shared_left;
    for (int i = 0; i < num_seqs; ++i) {
        const pkv_block_manager::Seq *s = find(bm, seq_ids[i]);
        const int64_t need = (s->len + 1 + bm->block_size - 1) / bm->block_size;
        if (need > bm->max_blocks_per_seq) return PKV_ERR_INVALID_ARG;
        if (static_cast<int64_t>(s->table.size()) < need) {
            ++demand;
            continue;
        }
        const int32_t last = s->table.back();
        auto it = shared_left.find(last);
        int32_t &rc = it == shared_left.end() ? (shared_left[last] = bm->refcount[last]) : it->second;
        if (rc > 1) {
            ++demand;
            --rc;
        }
    }
    if (demand > static_cast<int64_t>(bm->free_stack.size())) return PKV_ERR_OUT_OF_BLOCKS;
    int64_t ncow = 0;
    for (int i = 0; i < num_seqs; ++i) {
        int64_t src = -1, dst = -1;
        const pkv_status st = pkv_bm_append_token(bm, seq_ids[i], &slot_mapping[i], &src, &dst);
        if (st != PKV_OK) return st;  // not reached: checked above
        if (src >= 0) {
            cow_pairs[2 * ncow] = src;
            cow_pairs[2 * ncow + 1] = dst;
            ++ncow;
        }
    }
    for (int i = 0; i < num_seqs; ++i) {
        const pkv_block_manager::Seq *s = find(bm, seq_ids[i]);
        int32_t *row = block_tables + static_cast<int64_t>(i) * bm->max_blocks_per_seq;
        std::fill(row, row + bm->max_blocks_per_seq, 0);
        std::copy(s->table.begin(), s->table.end(), row);
        context_lens[i] = static_cast<int32_t>(s->len);
    }
    *num_cow_pairs = ncow;
    return PKV_OK;
}

}  // extern "C"
