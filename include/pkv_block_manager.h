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

/* Drops a live sequence (running, swapped or waiting for recompute); its
 * id stays retired. */
PKV_API pkv_status pkv_bm_free_sequence(pkv_block_manager *bm, int32_t seq);

/* Block table of one sequence into out[0 .. max_blocks-1] (host); returns the
 * number of entries, or -1 (bad id, retired sequence, or max_blocks too
 * small).  The entries are device blocks for a running sequence, host slots
 * for a swapped one, and none for one waiting for recompute. */
PKV_API int32_t pkv_bm_block_table(const pkv_block_manager *bm, int32_t seq, int32_t *out,
                                   int32_t max_blocks);

/* The inputs of a decode call for n sequences (host): tables_out [n][max_blocks]
 * (rows padded with filler), context_lens_out [n] (tokens held). */
PKV_API pkv_status pkv_bm_export(const pkv_block_manager *bm, const int32_t *seq_ids, int32_t n,
                                 int32_t *tables_out, int32_t max_blocks, int32_t filler,
                                 int32_t *context_lens_out);

/* ---------------------------------------------------------------- pre-emption
 *
 * "Running Out of Cache" (closing paragraph, and the glossary entry
 * "Pre-emption"): when even a paged cache runs out, a server evicts a running
 * request's cache and later either recomputes it or swaps it back in.
 *
 * A sequence is in one of three live states:
 *   PKV_BM_RUNNING     holds device blocks; every call above applies to it.
 *   PKV_BM_SWAPPED     its cache lives in host slots of the swap space; it
 *                      holds no device block.
 *   PKV_BM_RECOMPUTE   holds nothing; its length is kept, and its rows must be
 *                      written again (a prefill of its tokens) after resume.
 * append, fork and export accept running sequences only; free_sequence
 * accepts any live sequence (a swapped one returns its host slots).
 *
 * Host slots are handed out like device blocks: ascending at first, most
 * recently freed first afterwards, with a reference count each.
 */
enum { PKV_BM_RETIRED = 0, PKV_BM_RUNNING = 1, PKV_BM_SWAPPED = 2, PKV_BM_RECOMPUTE = 3 };
enum { PKV_PREEMPT_RECOMPUTE = 0, PKV_PREEMPT_SWAP = 1 };

/* Sets the swap space to num_host_blocks host slots.  Allowed only while no
 * sequence is swapped (PKV_ERR_INVALID_ARG otherwise); 0 (the default)
 * disables swapping. */
PKV_API pkv_status pkv_bm_set_swap_space(pkv_block_manager *bm, int32_t num_host_blocks);

/* Free device blocks an append of these n running sequences needs, new
 * blocks and copy-on-write copies together (the count pkv_bm_append checks
 * against the free list); -1 on a bad argument. */
PKV_API int64_t pkv_bm_step_blocks(const pkv_block_manager *bm, const int32_t *seq_ids,
                                   int32_t n);

/* Victims for one decode step.  seq_ids lists n running sequences in
 * priority order (the first is kept longest, for instance arrival order).
 * *num_victims_out receives the smallest k such that, once the last k are
 * evicted (their device references dropped), the first n - k can each append
 * one token.  k = n when even the first sequence cannot.  Changes nothing. */
PKV_API pkv_status pkv_bm_plan_preemption(const pkv_block_manager *bm, const int32_t *seq_ids,
                                          int32_t n, int32_t *num_victims_out);

/* Evicts n running sequences (mode PKV_PREEMPT_*).
 * RECOMPUTE: drops their device references, as free_sequence does, and keeps
 *   their lengths; *num_swap_out = 0.
 * SWAP: every distinct device block the n sequences hold gets one host slot,
 *   shared by those of the n that held the block.  swap_pairs_out (host,
 *   int64 [..][2], room for as many pairs as the n sequences hold blocks)
 *   receives the (device block, host slot) copies and *num_swap_out their
 *   count.  The caller runs them (pkv_block_swap from the device cache to the
 *   host pool) before any later write into the device blocks, which this
 *   call may return to the free list.
 * PKV_ERR_OUT_OF_BLOCKS (nothing changed) when the swap space is too small. */
PKV_API pkv_status pkv_bm_preempt(pkv_block_manager *bm, const int32_t *seq_ids, int32_t n,
                                  int32_t mode, int64_t *swap_pairs_out,
                                  int32_t *num_swap_out);

/* Brings n evicted sequences back to running, in the order given.
 * SWAPPED: every distinct host slot among them gets one new device block,
 *   shared by those of the n that held the slot; swap_pairs_out receives the
 *   (host slot, device block) copies (pkv_block_swap from the host pool to
 *   the device cache, run before the sequences' next attention); host slots
 *   no swapped sequence holds any more return to the swap space.
 * RECOMPUTE: each takes ceil(length / block_size) new blocks; the caller
 *   writes its rows again (pkv_kv_append at the slots its table gives)
 *   before its next attention.
 * swap_pairs_out needs room for as many pairs as the swapped ones hold slots.
 * PKV_ERR_OUT_OF_BLOCKS (nothing changed) when the free list is too short. */
PKV_API pkv_status pkv_bm_resume(pkv_block_manager *bm, const int32_t *seq_ids, int32_t n,
                                 int64_t *swap_pairs_out, int32_t *num_swap_out);

/* PKV_BM_* state of a sequence (PKV_BM_RETIRED for a bad or retired id). */
PKV_API int32_t pkv_bm_state(const pkv_block_manager *bm, int32_t seq);
/* Host slots free in the swap space; reference count of one slot (-1 if bad). */
PKV_API int32_t pkv_bm_num_free_host_blocks(const pkv_block_manager *bm);
PKV_API int32_t pkv_bm_host_ref_count(const pkv_block_manager *bm, int32_t slot);

/* Running totals since pkv_bm_create. */
typedef struct {
  int64_t cow_copies;          /* copy-on-write pairs pkv_bm_append emitted   */
  int64_t preempted_recompute; /* sequences evicted for recompute             */
  int64_t preempted_swap;      /* sequences evicted to the swap space         */
  int64_t resumed;             /* sequences brought back                      */
  int64_t blocks_swapped_out;  /* device-to-host block copies emitted         */
  int64_t blocks_swapped_in;   /* host-to-device block copies emitted         */
  int64_t tokens_recomputed;   /* tokens whose rows resume asked to rewrite   */
} pkv_bm_counters;
PKV_API pkv_status pkv_bm_get_counters(const pkv_block_manager *bm, pkv_bm_counters *out);

/* Tokens the sequence holds, in any live state (-1 for a bad or retired id). */
PKV_API int64_t pkv_bm_length(const pkv_block_manager *bm, int32_t seq);
/* Blocks on the free list; reference count of one block (-1 if bad id). */
PKV_API int32_t pkv_bm_num_free_blocks(const pkv_block_manager *bm);
PKV_API int32_t pkv_bm_ref_count(const pkv_block_manager *bm, int32_t block);

#ifdef __cplusplus
}
#endif

#endif /* PKV_BLOCK_MANAGER_H_ */
