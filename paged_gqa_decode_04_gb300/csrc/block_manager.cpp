// Host block manager of the paged KV cache (include/paged_kv_manager.h).
//
// Blocks are handed out only when a sequence needs one and come back when the
// last sequence holding them ends ("The Ultimate Guide to LLM Inference
// Optimization - Part 2", section "Paged Attention").  Sequences can share the
// blocks of a common prefix; every block carries a reference count and a
// write into a shared block first copies it (copy-on-write, "Modern LLM
// Inference ...", section 8.2 "Prefix Sharing").  Host memory only: the copies
// it decides on are carried out by paged_kv_copy_blocks on the device.
#include <stdint.h>

#include <new>
#include <vector>

#include "paged_kv_manager.h"

struct pgd_kvm_s {
    int64_t num_blocks;
    int block_size;
    int max_seqs;
    int max_blocks_per_seq;
    std::vector<int32_t> free_list;  // stack; back() is handed out next
    std::vector<int32_t> refs;       // per block
    struct Seq {
        bool live = false;
        int64_t len = 0;
        std::vector<int32_t> blocks;
    };
    std::vector<Seq> seqs;
};

namespace {

bool seq_ok(const pgd_kvm_s* m, int s) { return s >= 0 && s < m->max_seqs; }

}  // namespace

extern "C" {

int pgd_kvm_create(pgd_kvm_t* out, int64_t num_blocks, int block_size, int max_seqs,
                   int max_blocks_per_seq) {
    if (!out) return PGD_ERR_ARG;
    *out = nullptr;
    if (num_blocks < 1 || num_blocks > INT32_MAX || block_size < 1 || max_seqs < 1 ||
        max_blocks_per_seq < 1)
        return PGD_ERR_ARG;
    pgd_kvm_s* m = new (std::nothrow) pgd_kvm_s;
    if (!m) return PGD_ERR_ARG;
    try {
        m->num_blocks = num_blocks;
        m->block_size = block_size;
        m->max_seqs = max_seqs;
        m->max_blocks_per_seq = max_blocks_per_seq;
        m->refs.assign((size_t)num_blocks, 0);
        m->free_list.reserve((size_t)num_blocks);
        for (int64_t b = num_blocks - 1; b >= 0; --b) m->free_list.push_back((int32_t)b);
        m->seqs.resize((size_t)max_seqs);
    } catch (...) {
        delete m;
        return PGD_ERR_ARG;
    }
    *out = m;
    return PGD_OK;
}

int pgd_kvm_destroy(pgd_kvm_t m) {
    delete m;
    return PGD_OK;
}

int pgd_kvm_add_sequence(pgd_kvm_t m, int seq) {
    if (!m) return PGD_ERR_ARG;
    if (!seq_ok(m, seq)) return PGD_ERR_NO_SEQ;
    auto& s = m->seqs[(size_t)seq];
    if (s.live) return PGD_ERR_SEQ_EXISTS;
    s.live = true;
    s.len = 0;
    s.blocks.clear();
    return PGD_OK;
}

int pgd_kvm_fork(pgd_kvm_t m, int parent, int child) {
    if (!m) return PGD_ERR_ARG;
    if (!seq_ok(m, parent) || !seq_ok(m, child) || !m->seqs[(size_t)parent].live)
        return PGD_ERR_NO_SEQ;
    auto& c = m->seqs[(size_t)child];
    if (c.live) return PGD_ERR_SEQ_EXISTS;
    const auto& p = m->seqs[(size_t)parent];
    c.blocks = p.blocks;
    c.len = p.len;
    c.live = true;
    for (int32_t b : c.blocks) ++m->refs[(size_t)b];
    return PGD_OK;
}

int pgd_kvm_free_sequence(pgd_kvm_t m, int seq) {
    if (!m) return PGD_ERR_ARG;
    if (!seq_ok(m, seq) || !m->seqs[(size_t)seq].live) return PGD_ERR_NO_SEQ;
    auto& s = m->seqs[(size_t)seq];
    for (int32_t b : s.blocks) {
        if (--m->refs[(size_t)b] == 0) m->free_list.push_back(b);
    }
    s.blocks.clear();
    s.len = 0;
    s.live = false;
    return PGD_OK;
}

int pgd_kvm_append_slots(pgd_kvm_t m, const int* seqs, int n, int32_t* slot_mapping,
                         int32_t* copy_src, int32_t* copy_dst, int* n_copies) {
    if (!m || n < 0 || (n > 0 && (!seqs || !slot_mapping || !copy_src || !copy_dst)) ||
        !n_copies)
        return PGD_ERR_ARG;
    *n_copies = 0;
    const int bs = m->block_size;
    // Pass 1: check everything and count the blocks needed, changing nothing.
    int64_t need = 0;
    for (int i = 0; i < n; ++i) {
        if (!seq_ok(m, seqs[i]) || !m->seqs[(size_t)seqs[i]].live) return PGD_ERR_NO_SEQ;
        for (int j = 0; j < i; ++j)
            if (seqs[j] == seqs[i]) return PGD_ERR_ARG;  // one token per sequence per call
        const auto& s = m->seqs[(size_t)seqs[i]];
        if (s.len % bs == 0) {
            if ((int64_t)s.blocks.size() >= m->max_blocks_per_seq) return PGD_ERR_SEQ_FULL;
            ++need;
        } else if (m->refs[(size_t)s.blocks.back()] > 1) {
            ++need;  // the shared last block gets a private copy
        }
    }
    if (need > (int64_t)m->free_list.size()) return PGD_ERR_NO_BLOCKS;
    // Pass 2: apply.
    for (int i = 0; i < n; ++i) {
        auto& s = m->seqs[(size_t)seqs[i]];
        if (s.len % bs == 0) {
            const int32_t b = m->free_list.back();
            m->free_list.pop_back();
            m->refs[(size_t)b] = 1;
            s.blocks.push_back(b);
        } else if (m->refs[(size_t)s.blocks.back()] > 1) {
            const int32_t old = s.blocks.back();
            const int32_t b = m->free_list.back();
            m->free_list.pop_back();
            m->refs[(size_t)b] = 1;
            --m->refs[(size_t)old];
            s.blocks.back() = b;
            copy_src[*n_copies] = old;
            copy_dst[*n_copies] = b;
            ++*n_copies;
        }
        slot_mapping[i] = (int32_t)((int64_t)s.blocks.back() * bs + s.len % bs);
        ++s.len;
    }
    return PGD_OK;
}

int pgd_kvm_block_tables(pgd_kvm_t m, const int* seqs, int n, int32_t* table, int max_blocks,
                         int32_t* lens) {
    if (!m || n < 0 || max_blocks < 1 || (n > 0 && (!seqs || !table || !lens)))
        return PGD_ERR_ARG;
    for (int i = 0; i < n; ++i) {
        if (!seq_ok(m, seqs[i]) || !m->seqs[(size_t)seqs[i]].live) return PGD_ERR_NO_SEQ;
        if ((int64_t)m->seqs[(size_t)seqs[i]].blocks.size() > max_blocks) return PGD_ERR_SHAPE;
    }
    for (int i = 0; i < n; ++i) {
        const auto& s = m->seqs[(size_t)seqs[i]];
        int32_t* row = table + (int64_t)i * max_blocks;
        for (int j = 0; j < max_blocks; ++j)
            row[j] = j < (int)s.blocks.size() ? s.blocks[(size_t)j] : -1;
        lens[i] = (int32_t)s.len;
    }
    return PGD_OK;
}

int pgd_kvm_num_free(pgd_kvm_t m, int64_t* n_free) {
    if (!m || !n_free) return PGD_ERR_ARG;
    *n_free = (int64_t)m->free_list.size();
    return PGD_OK;
}

int pgd_kvm_ref_count(pgd_kvm_t m, int64_t block, int* count) {
    if (!m || !count || block < 0 || block >= m->num_blocks) return PGD_ERR_ARG;
    *count = m->refs[(size_t)block];
    return PGD_OK;
}

}  // extern "C"
