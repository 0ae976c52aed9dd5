/*
 * paged_kv_manager.h -- the KV write path of libpaged_gqa.so: a host block
 * manager for the paged cache and the device kernels that store new tokens and
 * copy blocks.
 *
 * Sources: blocks are allocated only when a sequence needs a new one and are
 * freed when the request finishes ("The Ultimate Guide to LLM Inference
 * Optimization - Part 2", section "Paged Attention"); several sequences can
 * point at the same blocks of a shared prefix, each block carrying a
 * reference count, and when sequences diverge only the modified block is
 * copied ("Modern LLM Inference - Workloads, Bottlenecks, and Optimization
 * Techniques", section 8.2, "Prefix Sharing (Copy-on-Write)").
 *
 * Slots.  A physical slot is block * block_size + position-in-block; the K (and
 * V) row of a slot is pool[slot / block_size][slot % block_size][:, :], i.e.
 * Hkv * D contiguous elements starting at element slot * Hkv * D.
 *
 * Threading.  A manager is not thread-safe; one owner thread drives it.  The
 * device calls are asynchronous on `stream` and take device pointers.
 * Statuses are the pgd_status codes of paged_gqa.h.
 */
#ifndef PAGED_KV_MANAGER_H
#define PAGED_KV_MANAGER_H

#include <stddef.h>
#include <stdint.h>

#include "paged_gqa.h"

#ifdef __cplusplus
extern "C" {
#endif

typedef struct pgd_kvm_s *pgd_kvm_t;

/* Extra statuses of the manager. */
enum pgd_kvm_status {
    PGD_ERR_NO_BLOCKS = 20,  /* the pool has no free block left (nothing changed) */
    PGD_ERR_NO_SEQ = 21,     /* unknown sequence id */
    PGD_ERR_SEQ_EXISTS = 22, /* sequence id already in use */
    PGD_ERR_SEQ_FULL = 23    /* sequence already holds max_blocks_per_seq blocks */
};

/*
 * A manager for a pool of `num_blocks` blocks of `block_size` tokens, serving
 * sequence ids 0 .. max_seqs-1, each holding at most max_blocks_per_seq
 * blocks.  Host memory only (no CUDA call).  All blocks start free.
 */
int pgd_kvm_create(pgd_kvm_t *out, int64_t num_blocks, int block_size, int max_seqs,
                   int max_blocks_per_seq);
int pgd_kvm_destroy(pgd_kvm_t m);

/* Start an empty sequence. */
int pgd_kvm_add_sequence(pgd_kvm_t m, int seq);

/*
 * Start `child` as a copy of `parent` that shares every block of it: no data
 * is copied, each shared block's reference count goes up by one.  The first
 * later append that writes into a shared last block copies that block first
 * (copy-on-write).
 */
int pgd_kvm_fork(pgd_kvm_t m, int parent, int child);

/* End a sequence: drop one reference from each of its blocks; blocks that
 * reach zero return to the free list. */
int pgd_kvm_free_sequence(pgd_kvm_t m, int seq);

/*
 * Reserve the next token position of each of the n sequences `seqs` (distinct
 * ids), in order.  slot_mapping[i] receives the physical slot the new token of
 * seqs[i] must be written to.  A sequence whose last block is full gets a
 * fresh block; one whose last block is shared gets a private copy of it, and
 * the pair (source block, new block) is appended to copy_src / copy_dst (room
 * for n pairs), with their count in *n_copies; those block copies must be run
 * (paged_kv_copy_blocks) before the new tokens are written.  If the pool runs
 * out of blocks, the call returns PGD_ERR_NO_BLOCKS and changes nothing.
 */
int pgd_kvm_append_slots(pgd_kvm_t m, const int *seqs, int n, int32_t *slot_mapping,
                         int32_t *copy_src, int32_t *copy_dst, int *n_copies);

/*
 * Write the block tables and lengths of sequences `seqs` for paged_gqa_decode:
 * table is [n, max_blocks] int32 (row i for seqs[i], entries past the
 * sequence's blocks set to -1), lens is [n] int32.  Requires max_blocks >= the
 * blocks any of the sequences holds.
 */
int pgd_kvm_block_tables(pgd_kvm_t m, const int *seqs, int n, int32_t *table, int max_blocks,
                         int32_t *lens);

/* Free blocks, and the reference count of one block (0 when free). */
int pgd_kvm_num_free(pgd_kvm_t m, int64_t *n_free);
int pgd_kvm_ref_count(pgd_kvm_t m, int64_t block, int *count);

/*
 * Device: copy whole blocks, K and V, from src[i] to dst[i] for i < n (device
 * int32 arrays).  Destinations must be distinct and differ from every source.
 * For 8-bit pages with a scale per block and KV head (paged_kv_pool_create_q8
 * with PGD_SCALE_PER_BLOCK) the destination blocks' K and V scale rows are
 * copied from the sources' too (the handle's scale arrays are written).
 */
int paged_kv_copy_blocks(pgd_pool_t pool, const int32_t *src, const int32_t *dst, int n,
                         void *stream);

/*
 * Device: store n new tokens.  k_new and v_new are [n, Hkv, D] in the pool's
 * dtype (8-bit pages: codes, already quantized with the scales of the blocks
 * they go to); slot_mapping is a device int32 array of n physical slots
 * (distinct, in [0, num_blocks * block_size)).  A slot out of range is skipped
 * and latches PGD_ERR_BLOCK_ID (read it with paged_gqa_get_error).
 */
int paged_kv_append(pgd_pool_t pool, const void *k_new, const void *v_new,
                    const int32_t *slot_mapping, int n, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* PAGED_KV_MANAGER_H */
