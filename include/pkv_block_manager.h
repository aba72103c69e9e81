/*
 * pkv_block_manager.h -- host-side manager of the paged KV pool: free list,
 * per-sequence block tables, reference counts, forks and copy-on-write.
 *
 * Passages: "ML Interview Prep, Lesson 13" section 3.5 "Paged attention" (a
 * pool of fixed-size 16-token blocks; each sequence has a block table; a
 * sequence gets a new block only when its last block is full; a block can
 * belong to several sequences and a reference count says how many; before a
 * sequence writes into a block whose count is above 1 it gets a private copy
 * and the shared block's count drops by one; finished sequences free their
 * blocks by decreasing the counts) and "LLM Serving: Continuous Batching &
 * PagedAttention" sections 4.1 (the block for token 16 is taken from the free
 * list), 4.2 (forked outputs share the prompt's blocks) and 7 (block manager:
 * allocate from a free list with count 1; release lowers the count and
 * returns the block at zero).
 *
 * One decode step with this manager and pkv.h:
 *   1. pkv_bm_append       -> slot_mapping for the step's new tokens and the
 *                             copy-on-write pairs;
 *   2. pkv_copy_blocks     (the pairs, on the device);
 *   3. pkv_kv_append       (the new rows at slot_mapping);
 *   4. pkv_bm_block_tables -> block tables and context lengths;
 *   5. pkv_paged_decode_attention.
 *
 * Everything here runs on the host and touches no device memory; the caller
 * copies slot mappings, pairs and tables to the device. A manager is safe to
 * call from several threads (each call takes the manager's lock). Physical
 * block ids are handed out by a last-in first-out free list whose first pops
 * on a new manager give 0, 1, 2, ...; callers must not rely on the ids.
 *
 * Readings of the pages: a sequence of n tokens holds exactly ceil(n/16)
 * blocks (one created with 0 tokens holds none until its first append). A
 * call that cannot get every block it needs changes nothing and returns
 * PKV_ERR_NO_BLOCKS (the scheduler then preempts or waits; scheduling is not
 * this library's job).
 */
#ifndef PKV_BLOCK_MANAGER_H
#define PKV_BLOCK_MANAGER_H

#include <stdint.h>

#include "pkv.h"

#ifdef __cplusplus
extern "C" {
#endif

typedef struct pkv_block_manager pkv_block_manager;

/* A manager of a pool of num_blocks blocks (1 .. 2^31-1), all free. Returns
 * NULL for an invalid size or when host memory runs out. */
pkv_block_manager *pkv_bm_create(int64_t num_blocks);

/* Frees the manager (NULL is a no-op). The pool's device memory is the
 * caller's and is not touched. */
void pkv_bm_destroy(pkv_block_manager *bm);

/* Free blocks, pool size, live sequences; -1 for a NULL manager. */
int64_t pkv_bm_num_free(const pkv_block_manager *bm);
int64_t pkv_bm_num_blocks(const pkv_block_manager *bm);
int64_t pkv_bm_num_sequences(const pkv_block_manager *bm);

/* Reference count of a block (0 = free); -1 for an id outside the pool or a
 * NULL manager. */
int32_t pkv_bm_refcount(const pkv_block_manager *bm, int64_t block);

/*
 * A new sequence whose first num_tokens tokens (its prompt) get
 * ceil(num_tokens/16) fresh blocks, count 1 each. The caller writes the
 * prompt's rows (e.g. with pkv_kv_append at the slots its table gives).
 * PKV_ERR_SEQUENCE if seq_id is live, PKV_ERR_SHAPE if num_tokens < 0,
 * PKV_ERR_NO_BLOCKS if the free list is too short (nothing changes).
 */
pkv_status pkv_bm_add_sequence(pkv_block_manager *bm, int64_t seq_id, int64_t num_tokens);

/*
 * child_id shares every block of parent_id (parallel sampling, beam search):
 * same table and length, each block's count raised by one. No block is taken.
 * PKV_ERR_SEQUENCE if the parent is unknown, the child is live, or they are
 * equal; PKV_ERR_RANGE if a count would overflow.
 */
pkv_status pkv_bm_fork(pkv_block_manager *bm, int64_t parent_id, int64_t child_id);

/* The sequence ends: each of its blocks' counts drops by one and blocks that
 * reach zero return to the free list. PKV_ERR_SEQUENCE if unknown. */
pkv_status pkv_bm_free_sequence(pkv_block_manager *bm, int64_t seq_id);

/*
 * Room for n_per_seq new tokens at the end of each of num_seqs sequences,
 * handled in the order given, each sequence's tokens one after another:
 *   - a token at a multiple of 16 opens a fresh block;
 *   - otherwise, if the last block is shared (count > 1), the sequence first
 *     gets a fresh private block, the pair (shared, fresh) is reported for
 *     pkv_copy_blocks, and the shared block's count drops by one (so of the
 *     sharers appended in one call, the last one writes in place).
 *   slot_mapping  host, int64 [num_seqs * n_per_seq]: token t of seq_ids[i]
 *                 goes to slot_mapping[i * n_per_seq + t] = block*16 + offset
 *                 (the pkv_kv_append convention).
 *   copy_src, copy_dst host, int32 [num_seqs] capacity (at most one pair per
 *                 sequence); *num_copies receives the number of pairs. The
 *                 destinations are distinct and none is a source.
 * All-or-nothing: PKV_ERR_NO_BLOCKS if the free blocks do not cover every
 * sequence (nothing changes). PKV_ERR_SEQUENCE for an unknown or repeated id,
 * PKV_ERR_SHAPE for a negative count, PKV_ERR_NULL for a missing pointer
 * (pointers may be NULL when num_seqs * n_per_seq == 0).
 */
pkv_status pkv_bm_append(pkv_block_manager *bm, const int64_t *seq_ids, int32_t num_seqs,
                         int32_t n_per_seq, int64_t *slot_mapping, int32_t *copy_src,
                         int32_t *copy_dst, int32_t *num_copies);

/* Tokens of a sequence, -1 if unknown. */
int64_t pkv_bm_sequence_length(const pkv_block_manager *bm, int64_t seq_id);

/* A sequence's block table: writes min(count, capacity) ids to `blocks` (host)
 * and returns the count (ceil(length/16)); -1 if unknown. */
int64_t pkv_bm_sequence_blocks(const pkv_block_manager *bm, int64_t seq_id, int32_t *blocks,
                               int64_t capacity);

/*
 * The attention call's inputs for a batch: block_tables (host, int32
 * [num_seqs][max_blocks_per_seq], rows padded with -1) and context_lens
 * (host, int32 [num_seqs]). PKV_ERR_SEQUENCE for an unknown id, PKV_ERR_RANGE
 * if a sequence has more than max_blocks_per_seq blocks or 2^31 tokens
 * (checked before anything is written), PKV_ERR_SHAPE for negative sizes.
 */
pkv_status pkv_bm_block_tables(const pkv_block_manager *bm, const int64_t *seq_ids,
                               int32_t num_seqs, int32_t *block_tables,
                               int32_t max_blocks_per_seq, int32_t *context_lens);

/*
 * Full audit of the manager's own state: every count equals the number of
 * table entries naming the block, the free list holds each count-0 block
 * exactly once and nothing else, and every table has ceil(length/16) blocks.
 * Returns 0 when consistent, else a nonzero bit set (1 count mismatch, 2 a
 * block twice in the free list, 4 a held block in the free list, 8 free +
 * held != pool, 16 a table of the wrong size); -1 for a NULL manager.
 */
int32_t pkv_bm_check(const pkv_block_manager *bm);

#ifdef __cplusplus
}
#endif

#endif /* PKV_BLOCK_MANAGER_H */
