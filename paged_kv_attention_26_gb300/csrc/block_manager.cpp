// block_manager.cpp -- host-side paged-KV block bookkeeping (pd_bm_*).
//
// Rules (tutorial page "LLM 推理服务引擎深度拆解", section 2.3, BlockManager
// and Sequence): every block id starts on the free list in increasing order;
// allocation takes the last free id and sets its ref count to 1; dropping the
// last reference appends the id to the free list; a sequence appending at a
// block boundary gets a new block, otherwise a shared last block is replaced
// by a fresh copy (copy-on-write) and a private one is written in place; fork
// shares every block and copies nothing.  The allocation order is part of the
// contract so a replay of the same operations yields the same ids.
#include <algorithm>
#include <cstdint>
#include <new>
#include <unordered_map>
#include <vector>

#include "pd_attn.h"

struct pd_bm {
    int block_size;
    std::vector<int32_t> ref_count;
    std::vector<int32_t> free_ids;
    struct Seq {
        std::vector<int32_t> table;
        int64_t length = 0;
    };
    std::unordered_map<int, Seq> seqs;

    int32_t allocate() {
        if (free_ids.empty()) return -1;
        const int32_t b = free_ids.back();
        free_ids.pop_back();
        ref_count[b] = 1;
        return b;
    }
    void drop(int32_t b) {
        if (--ref_count[b] == 0) free_ids.push_back(b);
    }
};

extern "C" {

pd_bm* pd_bm_create(int num_blocks, int block_size) {
    if (num_blocks < 1 || block_size < 1) return nullptr;
    pd_bm* bm = new (std::nothrow) pd_bm();
    if (!bm) return nullptr;
    try {
        bm->block_size = block_size;
        bm->ref_count.assign(size_t(num_blocks), 0);
        bm->free_ids.resize(size_t(num_blocks));
        for (int i = 0; i < num_blocks; ++i) bm->free_ids[size_t(i)] = i;
    } catch (...) {
        delete bm;
        return nullptr;
    }
    return bm;
}

void pd_bm_destroy(pd_bm* bm) { delete bm; }

pd_status pd_bm_add_seq(pd_bm* bm, int seq_id) {
    if (!bm || seq_id < 0 || bm->seqs.count(seq_id)) return PD_ERR_INVALID_ARG;
    bm->seqs.emplace(seq_id, pd_bm::Seq{});
    return PD_OK;
}

pd_status pd_bm_append_slot(pd_bm* bm, int seq_id, int64_t* slot_out, int32_t* cow_src_out,
                            int32_t* cow_dst_out) {
    if (!bm || !slot_out) return PD_ERR_INVALID_ARG;
    auto it = bm->seqs.find(seq_id);
    if (it == bm->seqs.end()) return PD_ERR_NOT_FOUND;
    pd_bm::Seq& s = it->second;
    const int S = bm->block_size;
    int32_t src = -1, dst = -1;
    if (s.length % S == 0) {
        const int32_t b = bm->allocate();
        if (b < 0) return PD_ERR_NO_FREE_BLOCK;
        s.table.push_back(b);
    } else {
        const int32_t last = s.table.back();
        if (bm->ref_count[size_t(last)] != 1) {
            const int32_t b = bm->allocate();
            if (b < 0) return PD_ERR_NO_FREE_BLOCK;
            bm->drop(last);
            s.table.back() = b;
            src = last;
            dst = b;
        }
    }
    *slot_out = int64_t(s.table.back()) * S + s.length % S;
    s.length += 1;
    if (cow_src_out) *cow_src_out = src;
    if (cow_dst_out) *cow_dst_out = dst;
    return PD_OK;
}

pd_status pd_bm_fork(pd_bm* bm, int parent_id, int child_id) {
    if (!bm || child_id < 0) return PD_ERR_INVALID_ARG;
    auto it = bm->seqs.find(parent_id);
    if (it == bm->seqs.end()) return PD_ERR_NOT_FOUND;
    if (bm->seqs.count(child_id)) return PD_ERR_INVALID_ARG;
    pd_bm::Seq child = it->second;   // copy of the table and length
    for (int32_t b : child.table) bm->ref_count[size_t(b)] += 1;
    bm->seqs.emplace(child_id, std::move(child));
    return PD_OK;
}

pd_status pd_bm_release(pd_bm* bm, int seq_id) {
    if (!bm) return PD_ERR_INVALID_ARG;
    auto it = bm->seqs.find(seq_id);
    if (it == bm->seqs.end()) return PD_ERR_NOT_FOUND;
    for (int32_t b : it->second.table) bm->drop(b);
    bm->seqs.erase(it);
    return PD_OK;
}

pd_status pd_bm_block_table(const pd_bm* bm, int seq_id, int32_t* out, int cap, int* n_out) {
    if (!bm || cap < 0) return PD_ERR_INVALID_ARG;
    auto it = bm->seqs.find(seq_id);
    if (it == bm->seqs.end()) return PD_ERR_NOT_FOUND;
    const std::vector<int32_t>& t = it->second.table;
    if (n_out) *n_out = int(t.size());
    if (size_t(cap) < t.size() || (!out && !t.empty())) return PD_ERR_INVALID_ARG;
    for (size_t i = 0; i < t.size(); ++i) out[i] = t[i];
    return PD_OK;
}

int64_t pd_bm_seq_len(const pd_bm* bm, int seq_id) {
    if (!bm) return -1;
    auto it = bm->seqs.find(seq_id);
    return it == bm->seqs.end() ? -1 : it->second.length;
}

double pd_bm_usage(const pd_bm* bm) {
    if (!bm || bm->ref_count.empty()) return 0.0;
    const double n = double(bm->ref_count.size());
    return (n - double(bm->free_ids.size())) / n;
}

int pd_bm_ref_count(const pd_bm* bm, int block_id) {
    if (!bm || block_id < 0 || size_t(block_id) >= bm->ref_count.size()) return -1;
    return bm->ref_count[size_t(block_id)];
}

int pd_bm_num_free(const pd_bm* bm) { return bm ? int(bm->free_ids.size()) : -1; }

pd_status pd_bm_add_seq_shared(pd_bm* bm, int seq_id, const int32_t* blocks, int nblocks,
                               int64_t length) {
    if (!bm || seq_id < 0 || nblocks < 0 || (nblocks > 0 && !blocks) || bm->seqs.count(seq_id))
        return PD_ERR_INVALID_ARG;
    const int S = bm->block_size;
    if (length < 0 || length > int64_t(nblocks) * S ||
        (nblocks > 0 && length <= int64_t(nblocks - 1) * S))
        return PD_ERR_INVALID_ARG;
    for (int i = 0; i < nblocks; ++i) {
        const int32_t b = blocks[i];
        if (b < 0 || size_t(b) >= bm->ref_count.size() || bm->ref_count[size_t(b)] < 1)
            return PD_ERR_INVALID_ARG;     // only a block in use holds data to share
    }
    pd_bm::Seq s;
    s.table.assign(blocks, blocks + nblocks);
    s.length = length;
    for (int32_t b : s.table) bm->ref_count[size_t(b)] += 1;
    bm->seqs.emplace(seq_id, std::move(s));
    return PD_OK;
}

pd_status pd_bm_retain(pd_bm* bm, int block_id) {
    if (!bm || block_id < 0 || size_t(block_id) >= bm->ref_count.size() ||
        bm->ref_count[size_t(block_id)] < 1)
        return PD_ERR_INVALID_ARG;
    bm->ref_count[size_t(block_id)] += 1;
    return PD_OK;
}

pd_status pd_bm_drop(pd_bm* bm, int block_id) {
    if (!bm || block_id < 0 || size_t(block_id) >= bm->ref_count.size() ||
        bm->ref_count[size_t(block_id)] < 1)
        return PD_ERR_INVALID_ARG;
    bm->drop(block_id);
    return PD_OK;
}

}  // extern "C"

// Groups of consecutive sequences sharing leading blocks, for the
// shared-prefix decode (pd_attn.h states the rule).  Pure host code.
extern "C" pd_status pd_find_shared_prefixes(const int32_t* block_tables, int max_blocks_per_seq,
                                             const int32_t* context_lens, int B, int S,
                                             int max_group, int min_shared_tokens,
                                             int32_t* group_starts_out, int32_t* shared_lens_out,
                                             int* n_groups_out) {
    if ((B > 0 && (!block_tables || !context_lens || !shared_lens_out)) || !group_starts_out ||
        !n_groups_out || B < 0 || max_blocks_per_seq < 1 || S < 1 || max_group < 1 ||
        max_group > 32)
        return PD_ERR_INVALID_ARG;
    const int64_t cap = int64_t(max_blocks_per_seq) * S;
    auto ctx_of = [&](int i) -> int64_t {
        const int64_t c = context_lens[i];
        return c < 0 ? 0 : (c > cap ? cap : c);
    };
    // tokens of the leading full blocks that sequences i and f share
    auto common = [&](int i, int f) -> int64_t {
        const int64_t full = std::min(ctx_of(i), ctx_of(f)) / S;
        const int32_t* ti = block_tables + int64_t(i) * max_blocks_per_seq;
        const int32_t* tf = block_tables + int64_t(f) * max_blocks_per_seq;
        int64_t n = 0;
        while (n < full && ti[n] == tf[n]) ++n;
        return n * S;
    };
    const int64_t need = std::max<int64_t>(min_shared_tokens, S);
    int ng = 0, first = 0, members = B > 0 ? 1 : 0;
    int64_t shared = 0;
    group_starts_out[0] = 0;
    for (int i = 1; i < B; ++i) {
        const int64_t c = common(i, first);
        if (members < max_group && c >= need && (members == 1 || c >= shared)) {
            if (members == 1) shared = c;
            ++members;
            continue;
        }
        shared_lens_out[ng] = members > 1 ? int32_t(shared) : 0;
        group_starts_out[++ng] = i;
        first = i;
        members = 1;
        shared = 0;
    }
    if (B > 0) {
        shared_lens_out[ng] = members > 1 ? int32_t(shared) : 0;
        group_starts_out[++ng] = B;
    }
    *n_groups_out = ng;
    return PD_OK;
}
