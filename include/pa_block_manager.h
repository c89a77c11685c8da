/*
 * pa_block_manager.h -- host-side block manager of a paged KV pool (part of libpa.so).
 *
 * What it implements: the bookkeeping that turns sequences into the inputs the
 * kernels consume ("vLLM's PagedAttention: why the KV cache is paged", §4.1
 * logical -> physical mapping, §4.2 block reuse and copy-on-write; "KV Cache and
 * PagedAttention memory management", the paging section):
 *   - a pool of `num_blocks` physical blocks of `block_size` token slots, handed
 *     out from a free list and returned to it when no sequence references them;
 *   - per sequence, its length and its logical -> physical block list (a row of
 *     block_tables); token i of a sequence lives in slot
 *     block_list[i / block_size] * block_size + i % block_size;
 *   - sharing: a forked sequence references its parent's blocks (reference
 *     count + 1 per block) instead of copying them;
 *   - copy-on-write: before a token is appended into a block that more than one
 *     sequence references, the appending sequence gets a fresh block, the pair
 *     (shared block, fresh block) is reported for pa_copy_blocks, and the shared
 *     block loses one reference.
 *
 * A decode step with this manager: pa_bm_append_tokens for the batch (slots and
 * copy pairs), pa_bm_block_tables for the batch, then pa_copy_blocks (the copy
 * pairs), pa_reshape_and_cache (the slots) and pa_decode (the tables and lengths),
 * in that order, on one stream.
 *
 * Everything here is host memory and host code; no call touches the GPU.  A
 * manager is safe to use from several threads (calls are serialised).  Failed
 * calls change nothing.
 */
#ifndef PA_BLOCK_MANAGER_H_
#define PA_BLOCK_MANAGER_H_

#include <stdint.h>

#include "pa.h"

#ifdef __cplusplus
extern "C" {
#endif

typedef struct pa_block_manager pa_block_manager;

/* A manager of num_blocks >= 1 blocks of block_size >= 1 slots, all free.
 * Blocks are handed out lowest id first.  *out receives the handle. */
PA_API pa_status pa_bm_create(int64_t num_blocks, int block_size, pa_block_manager** out);

/* Frees the manager (NULL is a no-op). */
PA_API void pa_bm_destroy(pa_block_manager* bm);

/* Free blocks (referenced by no sequence). */
PA_API int64_t pa_bm_num_free_blocks(const pa_block_manager* bm);

/* A new sequence `seq_id` (not yet known) holding num_tokens >= 0 tokens, e.g. a
 * prompt: ceil(num_tokens / block_size) fresh blocks.  When slots is not NULL
 * it receives the num_tokens slots in token order (the slot_mapping of the
 * prompt's write).  PA_ERR_OUT_OF_BLOCKS when the pool cannot hold it. */
PA_API pa_status pa_bm_add_sequence(pa_block_manager* bm, int64_t seq_id, int64_t num_tokens, int64_t* slots);

/* A new sequence `child_id` sharing every block of `parent_id` (its whole
 * history, the partly filled last block included); one more reference per block. */
PA_API pa_status pa_bm_fork(pa_block_manager* bm, int64_t parent_id, int64_t child_id);

/* Drops a sequence; each of its blocks loses a reference and returns to the free
 * list at zero. */
PA_API pa_status pa_bm_free_sequence(pa_block_manager* bm, int64_t seq_id);

/* One new token for each of the num_seqs listed sequences (distinct ids): a
 * sequence whose last block is full gets a fresh block; a sequence whose last
 * block is partly filled and shared gets a fresh block and a copy pair.
 * slot_mapping[i] receives the slot of sequence i's new token; copies receives
 * *num_copies (src, dst) pairs, int64 [n, 2], to run with pa_copy_blocks before
 * the write (room for max_copies pairs; num_seqs pairs always suffice).
 * PA_ERR_OUT_OF_BLOCKS when the pool cannot serve the whole batch, and
 * PA_ERR_WORKSPACE when max_copies is too small; nothing changes then. */
PA_API pa_status pa_bm_append_tokens(pa_block_manager* bm, const int64_t* seq_ids, int num_seqs, int64_t* slot_mapping,
                                     int64_t* copies, int64_t max_copies, int64_t* num_copies);

/* Length (tokens) of a sequence. */
PA_API pa_status pa_bm_seq_len(const pa_block_manager* bm, int64_t seq_id, int64_t* len);

/* Rows of block_tables and seq_lens for the listed sequences: block_tables is
 * int32 [num_seqs, max_blocks_per_seq], entries past a sequence's blocks set to
 * -1; seq_lens int32 [num_seqs].  PA_ERR_INVALID_ARG when a sequence has more
 * blocks than max_blocks_per_seq or a length beyond int32. */
PA_API pa_status pa_bm_block_tables(const pa_block_manager* bm, const int64_t* seq_ids, int num_seqs,
                                    int32_t* block_tables, int max_blocks_per_seq, int32_t* seq_lens);

/* For pa_decode_shared: the listed sequences' prefix groups -- runs of consecutive
 * entries whose first logical block is one physical block (sequences of one fork
 * family that still share their prefix) -- with prefix_group[i] the index of the
 * run's first entry, and prefix_blocks[i] the leading logical blocks sequence i
 * holds in the same physical blocks as the run's longest sequence (0 for a run
 * of one).  List the sequences of a fork family next to each other to let decode
 * read their common blocks once. */
PA_API pa_status pa_bm_prefix_groups(const pa_block_manager* bm, const int64_t* seq_ids, int num_seqs,
                                     int32_t* prefix_group, int32_t* prefix_blocks);

/* Number of sequences that reference a block (0 when it is free). */
PA_API pa_status pa_bm_refcount(const pa_block_manager* bm, int64_t block, int* refcount);

#ifdef __cplusplus
}
#endif

#endif /* PA_BLOCK_MANAGER_H_ */
