// pa_block_manager.cpp -- host block manager: refcounted blocks, per-sequence
// block tables and the copy-on-write decision before an append.
//
// spindle, "Paging": a pool of fixed 16-token blocks with a block table per
// sequence bounds waste by the final partial block; reference counts give
// copy-on-write forking.  spindle, "Two bugs worth recording": appends name
// an explicit start position.  The readings where the page is silent are
// stated in pa.h next to the declarations.
#include <cstdint>
#include <new>
#include <set>
#include <unordered_map>
#include <vector>

#include "pa.h"

struct pa_block_manager {
    int32_t num_blocks = 0;
    std::vector<int32_t> refcount;
    std::set<int32_t> free_ids;   // lowest id first
    struct Seq {
        std::vector<int32_t> table;
        int32_t len = 0;
    };
    std::unordered_map<int32_t, Seq> seqs;
    int32_t next_id = 0;
    int64_t logical_tokens = 0;

    int32_t take() {
        const int32_t b = *free_ids.begin();
        free_ids.erase(free_ids.begin());
        refcount[b] = 1;
        return b;
    }
    void drop(int32_t b) {
        if (--refcount[b] == 0) free_ids.insert(b);
    }
    // Blocks an append over [start, start+n) needs from the free list.
    int32_t needed(const Seq& q, int32_t start, int32_t n) const {
        if (n <= 0) return 0;
        int32_t need = 0;
        const int32_t lb0 = start / PA_BLOCK_SIZE, lb1 = (start + n - 1) / PA_BLOCK_SIZE;
        for (int32_t lb = lb0; lb <= lb1; ++lb) {
            if (lb >= (int32_t)q.table.size() || refcount[q.table[lb]] > 1) ++need;
        }
        return need;
    }
    int32_t shared_touched(const Seq& q, int32_t start, int32_t n) const {
        if (n <= 0) return 0;
        int32_t k = 0;
        const int32_t lb0 = start / PA_BLOCK_SIZE, lb1 = (start + n - 1) / PA_BLOCK_SIZE;
        for (int32_t lb = lb0; lb <= lb1 && lb < (int32_t)q.table.size(); ++lb)
            if (refcount[q.table[lb]] > 1) ++k;
        return k;
    }
};

extern "C" {

pa_status pa_bm_create(int32_t num_blocks, pa_block_manager** out) {
    if (!out || num_blocks <= 0) return PA_ERR_INVALID_ARG;
    pa_block_manager* bm = new (std::nothrow) pa_block_manager();
    if (!bm) return PA_ERR_INVALID_ARG;
    bm->num_blocks = num_blocks;
    bm->refcount.assign(num_blocks, 0);
    for (int32_t b = 0; b < num_blocks; ++b) bm->free_ids.insert(bm->free_ids.end(), b);
    *out = bm;
    return PA_OK;
}

void pa_bm_destroy(pa_block_manager* bm) { delete bm; }

pa_status pa_bm_add_seq(pa_block_manager* bm, int32_t* seq_out) {
    if (!bm || !seq_out || bm->next_id == INT32_MAX) return PA_ERR_INVALID_ARG;
    const int32_t id = bm->next_id++;
    bm->seqs.emplace(id, pa_block_manager::Seq());
    *seq_out = id;
    return PA_OK;
}

pa_status pa_bm_fork(pa_block_manager* bm, int32_t parent, int32_t* child_out) {
    if (!bm || !child_out || bm->next_id == INT32_MAX) return PA_ERR_INVALID_ARG;
    auto it = bm->seqs.find(parent);
    if (it == bm->seqs.end()) return PA_ERR_INVALID_ARG;
    pa_block_manager::Seq child = it->second;   // copy of table and length
    for (int32_t b : child.table) ++bm->refcount[b];
    bm->logical_tokens += child.len;
    const int32_t id = bm->next_id++;
    bm->seqs.emplace(id, std::move(child));
    *child_out = id;
    return PA_OK;
}

pa_status pa_bm_free_seq(pa_block_manager* bm, int32_t seq) {
    if (!bm) return PA_ERR_INVALID_ARG;
    auto it = bm->seqs.find(seq);
    if (it == bm->seqs.end()) return PA_ERR_INVALID_ARG;
    for (int32_t b : it->second.table) bm->drop(b);
    bm->logical_tokens -= it->second.len;
    bm->seqs.erase(it);
    return PA_OK;
}

pa_status pa_bm_blocks_needed(const pa_block_manager* bm, int32_t seq, int32_t start_pos,
                              int32_t num_tokens, int32_t* blocks_out) {
    if (!bm || !blocks_out || start_pos < 0 || num_tokens < 0) return PA_ERR_INVALID_ARG;
    auto it = bm->seqs.find(seq);
    if (it == bm->seqs.end()) return PA_ERR_INVALID_ARG;
    if ((int64_t)start_pos + num_tokens > INT32_MAX) return PA_ERR_INVALID_ARG;
    *blocks_out = bm->needed(it->second, start_pos, num_tokens);
    return PA_OK;
}

pa_status pa_bm_prepare_append(pa_block_manager* bm, int32_t seq, int32_t start_pos,
                               int32_t num_tokens, int32_t* pairs_out, int32_t max_pairs,
                               int32_t* num_pairs_out) {
    if (!bm || !num_pairs_out || start_pos < 0 || num_tokens < 0 || max_pairs < 0)
        return PA_ERR_INVALID_ARG;
    auto it = bm->seqs.find(seq);
    if (it == bm->seqs.end()) return PA_ERR_INVALID_ARG;
    pa_block_manager::Seq& q = it->second;
    *num_pairs_out = 0;
    if (num_tokens == 0) return PA_OK;
    if ((int64_t)start_pos + num_tokens > INT32_MAX) return PA_ERR_INVALID_ARG;
    if ((int64_t)start_pos > (int64_t)q.table.size() * PA_BLOCK_SIZE) return PA_ERR_INVALID_ARG;
    const int32_t copies = bm->shared_touched(q, start_pos, num_tokens);
    if (copies > max_pairs || (copies > 0 && !pairs_out)) return PA_ERR_INVALID_ARG;
    if (bm->needed(q, start_pos, num_tokens) > (int32_t)bm->free_ids.size())
        return PA_ERR_OUT_OF_BLOCKS;
    int32_t np = 0;
    const int32_t lb0 = start_pos / PA_BLOCK_SIZE, lb1 = (start_pos + num_tokens - 1) / PA_BLOCK_SIZE;
    for (int32_t lb = lb0; lb <= lb1; ++lb) {
        if (lb >= (int32_t)q.table.size()) {
            q.table.push_back(bm->take());
        } else if (bm->refcount[q.table[lb]] > 1) {
            const int32_t old = q.table[lb];
            const int32_t fresh = bm->take();
            bm->drop(old);
            q.table[lb] = fresh;
            pairs_out[2 * np] = old;
            pairs_out[2 * np + 1] = fresh;
            ++np;
        }
    }
    const int32_t end = start_pos + num_tokens;
    if (end > q.len) {
        bm->logical_tokens += end - q.len;
        q.len = end;
    }
    *num_pairs_out = np;
    return PA_OK;
}

pa_status pa_bm_block_table(const pa_block_manager* bm, int32_t seq, int32_t* row_out,
                            int32_t max_blocks, int32_t* num_blocks_out) {
    if (!bm || max_blocks < 0 || (max_blocks > 0 && !row_out)) return PA_ERR_INVALID_ARG;
    auto it = bm->seqs.find(seq);
    if (it == bm->seqs.end()) return PA_ERR_INVALID_ARG;
    const auto& t = it->second.table;
    if ((int32_t)t.size() > max_blocks) return PA_ERR_INVALID_ARG;
    for (int32_t i = 0; i < max_blocks; ++i) row_out[i] = i < (int32_t)t.size() ? t[i] : -1;
    if (num_blocks_out) *num_blocks_out = (int32_t)t.size();
    return PA_OK;
}

pa_status pa_bm_block_tables(const pa_block_manager* bm, const int32_t* seqs, int32_t num_seqs,
                             int32_t* rows_out, int32_t max_blocks) {
    if (!bm || num_seqs < 0 || max_blocks < 0 || (num_seqs > 0 && !seqs)) return PA_ERR_INVALID_ARG;
    if (num_seqs > 0 && max_blocks > 0 && !rows_out) return PA_ERR_INVALID_ARG;
    for (int32_t i = 0; i < num_seqs; ++i) {
        const pa_status st = pa_bm_block_table(bm, seqs[i], rows_out + (size_t)i * max_blocks,
                                               max_blocks, nullptr);
        if (st != PA_OK) return st;
    }
    return PA_OK;
}

pa_status pa_bm_seq_len(const pa_block_manager* bm, int32_t seq, int32_t* len_out) {
    if (!bm || !len_out) return PA_ERR_INVALID_ARG;
    auto it = bm->seqs.find(seq);
    if (it == bm->seqs.end()) return PA_ERR_INVALID_ARG;
    *len_out = it->second.len;
    return PA_OK;
}

pa_status pa_bm_refcount(const pa_block_manager* bm, int32_t block, int32_t* refcount_out) {
    if (!bm || !refcount_out || block < 0 || block >= bm->num_blocks) return PA_ERR_INVALID_ARG;
    *refcount_out = bm->refcount[block];
    return PA_OK;
}

pa_status pa_bm_stats(const pa_block_manager* bm, pa_bm_stats_t* out) {
    if (!bm || !out) return PA_ERR_INVALID_ARG;
    out->free_blocks = (int64_t)bm->free_ids.size();
    out->physical_blocks = (int64_t)bm->num_blocks - out->free_blocks;
    out->logical_tokens = bm->logical_tokens;
    out->num_seqs = (int64_t)bm->seqs.size();
    return PA_OK;
}

}  // extern "C"
