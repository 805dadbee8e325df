/*
 * pkv_block_manager.h -- host-side manager of a paged KV-cache block pool.
 *
 * "Running Out of Cache" (paragraph on PagedAttention, and "Fragmentation is
 * lost users"): the cache is split into fixed blocks of block_size tokens; a
 * sequence holds a list of blocks (its block table) that need not be
 * adjacent and takes a new block only when its last one is full, so it
 * wastes less than one block; sequences that share a prompt point at the
 * same blocks and copy a block only when one of them writes into it.
 * "Efficient Memory Management for Large Language Model Serving with
 * PagedAttention" (summary) states the same sharing with copy on write.
 *
 * The manager produces what the device calls consume: block tables and
 * context lengths (pkv_paged_decode_attention), slot mappings (pkv_kv_append,
 * pkv_paged_decode_step) and copy-on-write pairs (pkv_block_copy).  It is
 * plain host code: no CUDA call, no device memory.  A manager is not
 * thread-safe; use one per thread or lock around it.  Every call that
 * changes state either completes or changes nothing.
 *
 * Rules (the decode step, one token per sequence, "Insights into LLM Serving
 * Systems: KV-Cache Memory Allocation Patterns" section 4, Observation-1):
 *   - add_sequence(n) takes ceil(n / block_size) blocks from the free list.
 *   - fork(s) makes a sequence with s's blocks and length; every block's
 *     reference count grows by one.
 *   - append(seqs) gives each listed sequence one token at position len:
 *     if len % block_size == 0 the token opens a new block from the free
 *     list; else it goes into the last block, and if that block is shared
 *     (reference count > 1) the sequence first takes a new block, records
 *     the pair (old, new) for pkv_block_copy and drops its reference to the
 *     old one.  Sequences are handled in the order given.
 *   - free_sequence(s) drops s's references; blocks that no sequence holds
 *     return to the free list.
 * Blocks leave the free list in the order of free_order (pkv_bm_create) and
 * freed blocks are handed out again before untouched ones, most recently
 * freed first.
 */
#ifndef PKV_BLOCK_MANAGER_H_
#define PKV_BLOCK_MANAGER_H_

#include "pkv.h"

#ifdef __cplusplus
extern "C" {
#endif

typedef struct pkv_block_manager pkv_block_manager;

/* A pool of num_blocks blocks of block_size tokens.  free_order (host,
 * nullable) lists the block ids in the order they are handed out (a
 * permutation of 0 .. num_blocks-1; NULL = ascending).  Returns NULL on a bad
 * argument (message in pkv_last_error).  The caller owns the manager. */
PKV_API pkv_block_manager *pkv_bm_create(int32_t num_blocks, int32_t block_size,
                                         const int32_t *free_order);
PKV_API void pkv_bm_destroy(pkv_block_manager *bm);

/* A new sequence holding num_tokens tokens (>= 0).  Returns its id (ids are
 * 0, 1, 2, ... in creation order, forks included) or -1: PKV_ERR_OUT_OF_BLOCKS
 * when the free list is too short, PKV_ERR_INVALID_ARG otherwise. */
PKV_API int32_t pkv_bm_add_sequence(pkv_block_manager *bm, int64_t num_tokens);

/* A new sequence sharing all of parent's blocks.  Returns its id or -1. */
PKV_API int32_t pkv_bm_fork(pkv_block_manager *bm, int32_t parent);

/* One decode step for n sequences (ids, host): slot_mapping_out[i] (host,
 * int64) receives seq_ids[i]'s new slot block * block_size + offset;
 * cow_pairs_out (host, int64 [n][2]) receives the (src, dst) copies to run
 * before the append and *num_cow_out their count.  A sequence may appear
 * once per call.  PKV_ERR_OUT_OF_BLOCKS (nothing changed) when the step
 * needs more blocks than are free. */
PKV_API pkv_status pkv_bm_append(pkv_block_manager *bm, const int32_t *seq_ids, int32_t n,
                                 int64_t *slot_mapping_out, int64_t *cow_pairs_out,
                                 int32_t *num_cow_out);

/* Drops the sequence; its id stays retired. */
PKV_API pkv_status pkv_bm_free_sequence(pkv_block_manager *bm, int32_t seq);

/* Block table of one sequence into out[0 .. max_blocks-1] (host); returns the
 * number of blocks the sequence holds, or -1 (bad id, retired sequence, or
 * max_blocks too small). */
PKV_API int32_t pkv_bm_block_table(const pkv_block_manager *bm, int32_t seq, int32_t *out,
                                   int32_t max_blocks);

/* The inputs of a decode call for n sequences (host): tables_out [n][max_blocks]
 * (rows padded with filler), context_lens_out [n] (tokens held). */
PKV_API pkv_status pkv_bm_export(const pkv_block_manager *bm, const int32_t *seq_ids, int32_t n,
                                 int32_t *tables_out, int32_t max_blocks, int32_t filler,
                                 int32_t *context_lens_out);

/* Tokens the sequence holds (-1 for a bad or retired id). */
PKV_API int64_t pkv_bm_length(const pkv_block_manager *bm, int32_t seq);
/* Blocks on the free list; reference count of one block (-1 if bad id). */
PKV_API int32_t pkv_bm_num_free_blocks(const pkv_block_manager *bm);
PKV_API int32_t pkv_bm_ref_count(const pkv_block_manager *bm, int32_t block);

#ifdef __cplusplus
}
#endif

#endif /* PKV_BLOCK_MANAGER_H_ */
