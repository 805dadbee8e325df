/*
 * pkv.h -- C ABI of the paged / contiguous KV-cache decode library (sm_103a).
 *
 * Four operations make one decode step over a KV cache:
 *   pkv_kv_append                 write each new token's K and V into its slot
 *   pkv_paged_decode_attention    single-query attention through block tables
 *   pkv_contig_decode_attention   the same over per-request sub-tensors
 *   pkv_block_copy                copy whole blocks (copy on write)
 * and pkv_paged_decode_step / pkv_contig_decode_step run append + attention
 * of one layer as one call.  pkv_paged_prefill_attention /
 * pkv_contig_prefill_attention attend chunks of new tokens causally (prefill).
 * pkv_block_swap moves whole blocks between the device cache and a pool in
 * page-locked host memory (pre-emption by swapping).
 *
 * Conventions for every call:
 *   - All tensor arguments are DEVICE pointers on the current CUDA device,
 *     owned by the caller; the library never allocates or frees them and
 *     keeps no per-call state.  `stream` is a cudaStream_t (NULL = the legacy
 *     default stream); every call is asynchronous on it.
 *   - Element types: K, V, Q and outputs are bf16 (passed as void*), block
 *     tables, context lengths and request ids are int32, slots and copy
 *     pairs are int64.  head_dim must be 128 (PKV_ERR_UNSUPPORTED otherwise);
 *     num_q_heads must be a multiple of num_kv_heads with a ratio of 1..8.
 *   - bf16 base pointers must be 16-byte aligned, int32 arrays 4-byte and
 *     int64 arrays 8-byte aligned (PKV_ERR_INVALID_ARG otherwise).
 *   - The return value covers host-side validation and the launch
 *     (cudaGetLastError).  Device-side index checks run only in checked mode
 *     (pkv_set_checked); they record the first violation in a per-device
 *     error word read by pkv_get_device_error and skip the bad access.  In
 *     the default mode indices are trusted, as a page table is.
 *   - A query head h reads KV head h / (num_q_heads / num_kv_heads).
 *
 * Layouts (the pages fix none; these are this library's contracts):
 *   paged cache     [num_blocks][num_kv_heads][block_size][head_dim]
 *   contig buffer   [max_reqs][num_kv_heads][S][head_dim]
 *   q, out          [num_seqs][num_q_heads][head_dim]
 *   new k, v        [num_tokens][num_kv_heads][head_dim]
 *   block_tables    [num_seqs][max_blocks_per_seq]
 */
#ifndef PKV_H
#define PKV_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define PKV_API __attribute__((visibility("default")))
#else
#define PKV_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum pkv_status {
    PKV_OK = 0,
    PKV_ERR_INVALID_ARG = 1,   /* null/misaligned pointer, bad size        */
    PKV_ERR_UNSUPPORTED = 2,   /* head_dim != 128, group ratio > 8, ...     */
    PKV_ERR_WORKSPACE = 3,     /* workspace missing or smaller than needed  */
    PKV_ERR_CUDA = 4,          /* a CUDA runtime call failed                */
    PKV_ERR_DEVICE_BOUNDS = 5, /* pkv_get_device_error found a device error */
    PKV_ERR_OUT_OF_BLOCKS = 6  /* block manager: not enough free blocks     */
} pkv_status;

/* Codes stored in the device error word (checked mode, and wait limits). */
enum {
    PKV_DEVERR_NONE = 0,
    PKV_DEVERR_BLOCK_ID = 1,   /* block table entry outside [0, num_blocks) */
    PKV_DEVERR_SLOT = 2,       /* slot outside [0, num_slots)               */
    PKV_DEVERR_REQ_ID = 3,     /* request id outside [0, max_reqs)          */
    PKV_DEVERR_CONTEXT = 4,    /* context longer than max_context, than the
                                  block table holds, or than S             */
    PKV_DEVERR_COPY_PAIR = 5,  /* block_copy id outside [0, num_blocks)     */
    PKV_DEVERR_TIMEOUT = 6     /* a copy into shared memory never completed */
};

typedef struct pkv_heads {
    int32_t num_q_heads;
    int32_t num_kv_heads;
    int32_t head_dim;
} pkv_heads;

/*
 * KV append.  "Insights into LLM Serving Systems: KV-Cache Memory Allocation
 * Patterns", section 4, Observation-1: each decode iteration grows every
 * request's KV cache by exactly one token; "Running Out of Cache": a new
 * block is taken only when the last one is full.
 *
 * For each token t < num_tokens and KV head h, copies k[t][h][:] to
 * k_cache[slot / block_size][h][slot % block_size][:] and v likewise, where
 * slot = slot_mapping[t] (device, int64).  A negative slot skips the token
 * (padding).  For the contiguous layout pass block_size = S and slot =
 * reqId * S + position.  num_slots = num_blocks * block_size bounds the
 * slots in checked mode.  Bit-exact: the bytes are moved, not converted.
 */
PKV_API pkv_status pkv_kv_append(const int64_t *slot_mapping, int64_t num_tokens,
                         const void *k, const void *v,
                         void *k_cache, void *v_cache,
                         int64_t num_slots, int64_t block_size,
                         pkv_heads heads, void *stream);

/*
 * Number of context splits the decode calls use, and the fp32 workspace they
 * need, for num_seqs sequences of at most max_context positions on the
 * current device.  The split count depends only on these arguments, the
 * device's SM count and pkv_set_split_tiles; both decode calls use the same
 * rule.  The size covers whichever decode kernel the call selects.
 */
/*
 * Whether the decode calls (paged with this block_size, or contiguous with
 * block_size 0) run the tensor-core kernel (1) or the split kernel (0) for
 * num_seqs sequences of at most max_context positions, under the current
 * pkv_set_decode_variant; -1 on bad arguments.  (The paged call also needs
 * fewer than 2^31 cache rows for the tensor-core kernel.)
 */
PKV_API int32_t pkv_decode_uses_tensor_cores(int32_t num_seqs, pkv_heads heads,
                                             int32_t max_context, int32_t block_size);

PKV_API int32_t pkv_decode_num_splits(int32_t num_seqs, pkv_heads heads,
                              int32_t max_context);
PKV_API size_t pkv_decode_workspace_size(int32_t num_seqs, pkv_heads heads,
                                 int32_t max_context);

/*
 * Paged decode attention.  "Running Out of Cache": the cache is divided into
 * fixed blocks, a sequence's blocks need not be adjacent, and a block table
 * maps positions to blocks as a page table maps virtual to physical memory;
 * "Efficient Memory Management for Large Language Model Serving with
 * PagedAttention" (summary): the PagedAttention algorithm over such blocks.
 *
 * For sequence i and query head h, with ctx = context_lens[i]:
 *   K_j = k_cache[block_tables[i][j / block_size]][h / G][j % block_size]
 *   out[i][h] = sum_j softmax_j(scale * q[i][h] . K_j) V_j,  j < ctx
 * accumulated in fp32, rounded to bf16.  ctx <= 0 writes zeros.  Entries of
 * a block table past ceil(ctx / block_size) are never read.
 * max_context is a host-side upper bound on every context_lens[i] (it sizes
 * the grid without reading device memory); max_blocks_per_seq *
 * block_size must be >= max_context.  workspace must hold
 * pkv_decode_workspace_size(num_seqs, heads, max_context) bytes (16-byte
 * aligned) when that size is non-zero; its contents need no initialisation.
 */
PKV_API pkv_status pkv_paged_decode_attention(
    const void *q, const void *k_cache, const void *v_cache,
    const int32_t *block_tables, int32_t max_blocks_per_seq, int32_t num_blocks,
    const int32_t *context_lens, int32_t num_seqs, int32_t max_context,
    int32_t block_size, float scale, pkv_heads heads, void *out,
    void *workspace, size_t workspace_bytes, void *stream);

/*
 * Contiguous-layout decode attention.  "Leveraging Low-Level CUDA APIs for
 * vAttention's Dynamic Memory", section 5.2.3: each layer's K (and V) tensor
 * holds the maximum batch; the sub-tensor of a request sits at offset
 * reqId x S, S being the per-request maximum (counted here in tokens).
 *
 * Same result as the paged call with K_j = k_buf[req_ids[i]][h / G][j],
 * i.e. the paged layout with block_size = S and the table [req_ids[i]].
 * Requires context_lens[i] <= S and 0 <= req_ids[i] < max_reqs.
 */
PKV_API pkv_status pkv_contig_decode_attention(
    const void *q, const void *k_buf, const void *v_buf,
    const int32_t *req_ids, int32_t max_reqs,
    const int32_t *context_lens, int32_t num_seqs, int32_t max_context,
    int64_t S, float scale, pkv_heads heads, void *out,
    void *workspace, size_t workspace_bytes, void *stream);

/*
 * One decode step of one layer in one call: the append of this step's token
 * ("Insights into LLM Serving Systems: KV-Cache Memory Allocation Patterns",
 * section 4, Observation-1: every request grows by one token per iteration)
 * followed by the attention over the grown cache.  Same result, bit for bit,
 * as
 *   pkv_kv_append(slot_mapping, num_seqs, k_new, v_new, k_cache, v_cache,
 *                 num_blocks * block_size, block_size, heads, stream);
 *   pkv_paged_decode_attention(q, k_cache, v_cache, ..., stream);
 * (contiguous: block_size = S, num_slots = max_reqs * S and
 * pkv_contig_decode_attention), with one new token per sequence (k_new,
 * v_new [num_seqs][Hkv][128]), as long as slot_mapping[i] is the slot of
 * sequence i's newest position context_lens[i] - 1, or negative (no new
 * token): when the tensor-core kernel runs (the automatic choice for all
 * but small batches), it does the append itself, in the same launch, and
 * takes that position's K and V from k_new / v_new instead of from the
 * cache (the same bytes); checked mode reports a slot that is not that
 * position's (PKV_DEVERR_SLOT).  Otherwise the append kernel runs first and
 * the attention kernel starts while it runs: it reads q, context_lens and
 * block_tables (req_ids) at once and waits for the append only before it
 * loads K/V.  Either way none of those, nor out, may alias k_new, v_new or
 * the caches (they never do in a decode step).  All arguments are checked
 * before anything is launched.  Errors as for the two calls.  The pages
 * have no counterpart beyond the two operations it combines.
 */
PKV_API pkv_status pkv_paged_decode_step(
    const int64_t *slot_mapping, const void *k_new, const void *v_new,
    const void *q, void *k_cache, void *v_cache,
    const int32_t *block_tables, int32_t max_blocks_per_seq, int32_t num_blocks,
    const int32_t *context_lens, int32_t num_seqs, int32_t max_context,
    int32_t block_size, float scale, pkv_heads heads, void *out,
    void *workspace, size_t workspace_bytes, void *stream);

PKV_API pkv_status pkv_contig_decode_step(
    const int64_t *slot_mapping, const void *k_new, const void *v_new,
    const void *q, void *k_buf, void *v_buf,
    const int32_t *req_ids, int32_t max_reqs,
    const int32_t *context_lens, int32_t num_seqs, int32_t max_context,
    int64_t S, float scale, pkv_heads heads, void *out,
    void *workspace, size_t workspace_bytes, void *stream);

/*
 * Paged decode attention for batches whose sequences share prompt blocks
 * ("Running Out of Cache", "Fragmentation is lost users", and the
 * PagedAttention summary: sequences sampled from one prompt share its
 * physical blocks until one of them writes into one).  The batch is split
 * into num_groups groups of consecutive sequences: group g is sequences
 * group_start[g] .. group_start[g+1]-1 (device int32 [num_groups + 1],
 * group_start[0] = 0, group_start[num_groups] = num_seqs, at most
 * max_group_size sequences per group), and its members' block tables begin
 * with the same shared_blocks[g] entries (device int32 [num_groups]; every
 * member's context covers them).  Singleton groups with shared_blocks 0 are
 * plain sequences.  The shared positions are read once per group (all its
 * members' query heads are rows of one tensor-core tile) instead of once per
 * member; each member's own later positions are read as usual, and the
 * softmax parts are merged.  max_own_tokens is a host bound on every
 * sequence's own positions (context_lens[i] minus its group's shared
 * positions), or -1 if unknown.  With a bound of at most 256 the own
 * positions are attended without a second tensor-core pass: as masked key
 * tiles of the shared-prefix kernel when max_group_size times the bound
 * (rounded up to whole boxes of gcd(block_size, 128) rows) fits 512 key
 * slots -- and if the shared positions then take one chunk per group, that
 * kernel writes the output and the call is one launch -- else on CUDA cores
 * inside the final merge (checked mode reports a sequence beyond the bound,
 * PKV_DEVERR_CONTEXT, and its later positions are left out).  Result:
 * the same attention as
 * pkv_paged_decode_attention within the attention tolerance (a different
 * summation order).  Other arguments as there; block_size must be a multiple
 * of 16.  workspace (256-byte aligned) must hold
 * pkv_shared_decode_workspace_size(num_seqs, num_groups, max_group_size,
 * max_blocks_per_seq, heads) bytes.  Checked mode also reports a member whose
 * context does not cover its group's shared blocks (PKV_DEVERR_CONTEXT).
 */
/*
 * Kernel launches one pkv_paged_decode_attention_shared call with these
 * sizes makes on the current device (1 to 4, more for a tensor-core pass over
 * a batch of many long sequences), or -1 for sizes the call rejects.  No
 * counterpart in the pages: it reports which of the modes above a call runs.
 */
PKV_API int32_t pkv_shared_decode_launches(int32_t num_seqs, int32_t num_groups,
                                           int32_t max_group_size, int32_t max_blocks_per_seq,
                                           int32_t max_context, int32_t block_size,
                                           int32_t max_own_tokens, pkv_heads heads);
PKV_API size_t pkv_shared_decode_workspace_size(int32_t num_seqs, int32_t num_groups,
                                                int32_t max_group_size,
                                                int32_t max_blocks_per_seq, pkv_heads heads);
PKV_API pkv_status pkv_paged_decode_attention_shared(
    const void *q, const void *k_cache, const void *v_cache,
    const int32_t *block_tables, int32_t max_blocks_per_seq, int32_t num_blocks,
    const int32_t *context_lens, int32_t num_seqs, int32_t max_context,
    int32_t block_size, const int32_t *group_start, const int32_t *shared_blocks,
    int32_t num_groups, int32_t max_group_size, int32_t max_own_tokens, float scale,
    pkv_heads heads, void *out, void *workspace, size_t workspace_bytes, void *stream);

/*
 * Causal prefill attention over a paged cache (chunked prefill).  The pages
 * name prefill only as a serving phase ("Insights into LLM Serving Systems:
 * KV-Cache Memory Allocation Patterns", section headings); the reading here
 * is the standard one.  Sequence i's chunk of new tokens is rows
 * cu_seqlens_q[i] .. cu_seqlens_q[i+1]-1 of q (device int32 [num_seqs + 1],
 * cu_seqlens_q[0] = 0, cu_seqlens_q[num_seqs] = num_tokens) and holds the
 * last Lq_i of its context_lens[i] positions; their K and V rows must already
 * be in the cache (pkv_kv_append).  New token j of sequence i, at position
 * ctx_i - Lq_i + j, gives
 *   out[row][h] = sum_{p <= ctx_i - Lq_i + j} softmax_p(scale * q[row][h] . K_p) V_p
 * with K_p, V_p found through block_tables[i] as in pkv_paged_decode_attention
 * (a chunk of one token is exactly that call).  q, out: bf16 [num_tokens][Hq][128].
 * max_q_tokens is a host bound on every chunk's length (it sizes the list of
 * work items; the grid is one CTA per SM at most); block_size must be a
 * multiple of 16.  Accumulation in fp32, output bf16.  q is read through a
 * tensor map of exactly num_tokens rows, so no read leaves q.  Returns
 * PKV_ERR_CUDA when the driver refuses a tensor map.  Checked mode reports a
 * chunk longer than its context or than max_q_tokens, or a context beyond the
 * block table (PKV_DEVERR_CONTEXT), and bad block ids.
 */
PKV_API pkv_status pkv_paged_prefill_attention(
    const void *q, const int32_t *cu_seqlens_q, int32_t num_tokens,
    const void *k_cache, const void *v_cache, const int32_t *block_tables,
    int32_t max_blocks_per_seq, int32_t num_blocks, const int32_t *context_lens,
    int32_t num_seqs, int32_t max_q_tokens, int32_t block_size, float scale,
    pkv_heads heads, void *out, void *stream);

/*
 * The same causal prefill over per-request sub-tensors ("Leveraging Low-Level
 * CUDA APIs for vAttention's Dynamic Memory", 5.2.3: request reqId's K rows
 * at offset reqId x S of a per-layer buffer).  k_buf, v_buf: bf16
 * [max_reqs][Hkv][S][128]; sequence i reads request req_ids[i] (device int32
 * [num_seqs]); q, cu_seqlens_q, context_lens (<= S), out as in
 * pkv_paged_prefill_attention.  S must be a multiple of 16.  No row at or
 * past round_up(context_lens[i], 16) of a request is read, so buffers whose
 * pages are mapped on demand (pkv_vmm_ensure) need only that many rows
 * backed.  Checked mode also reports req_ids outside [0, max_reqs) as
 * PKV_DEVERR_BLOCK_ID.
 */
PKV_API pkv_status pkv_contig_prefill_attention(
    const void *q, const int32_t *cu_seqlens_q, int32_t num_tokens,
    const void *k_buf, const void *v_buf, const int32_t *req_ids, int32_t max_reqs,
    const int32_t *context_lens, int32_t num_seqs, int32_t max_q_tokens, int64_t S,
    float scale, pkv_heads heads, void *out, void *stream);

/*
 * Copy-on-write block copy.  "Running Out of Cache" (section "Fragmentation
 * is lost users") and the PagedAttention summary: sequences share physical
 * blocks and copy a block only when one of them writes into it.
 *
 * For each pair c < n of src_dst_pairs (device, int64 [n][2]) and each layer
 * l < num_layers, copies block_bytes bytes from block src to block dst of
 * k_caches[l] and of v_caches[l].  k_caches and v_caches are HOST arrays of
 * num_layers device pointers (each 16-byte aligned); block_bytes must be a
 * multiple of 16.  num_blocks bounds the ids in checked mode.  Pairs must
 * not overlap (no dst is another pair's src).  Bit-exact.
 */
PKV_API pkv_status pkv_block_copy(const int64_t *src_dst_pairs, int64_t n,
                          void *const *k_caches, void *const *v_caches,
                          int32_t num_layers, int64_t num_blocks,
                          int64_t block_bytes, void *stream);

/*
 * Block swap between two pools, for pre-emption.  "Running Out of Cache"
 * (closing paragraph, and the glossary entry "Pre-emption"): when even a
 * paged cache runs out, a server evicts a request's cache and swaps it back
 * in later.  pkv_bm_preempt / pkv_bm_resume (pkv_block_manager.h) give the
 * pairs.
 *
 * For each pair c < n of pairs (int64 [n][2] = (src, dst)) and each layer
 * l < num_layers, copies block_bytes bytes from block src of src_k[l] to
 * block dst of dst_k[l], and from src_v[l] to dst_v[l].  src_k, src_v,
 * dst_k and dst_v are HOST arrays of num_layers pointers.  Each of those
 * pointers, and pairs, must be device memory, managed memory, or page-locked
 * host memory (cudaHostAlloc, cudaHostRegister; the kernel reads and writes
 * it across the CPU-GPU link); ordinary pageable memory, a null or a
 * misaligned pointer (16 bytes; 8 for pairs) gives PKV_ERR_INVALID_ARG.
 * block_bytes must be a multiple of 16.  src_num_blocks / dst_num_blocks
 * bound the ids in checked mode (PKV_DEVERR_COPY_PAIR).  The two sides must
 * not overlap.  Bit-exact.
 */
PKV_API pkv_status pkv_block_swap(const int64_t *pairs, int64_t n,
                          void *const *src_k, void *const *src_v, int64_t src_num_blocks,
                          void *const *dst_k, void *const *dst_v, int64_t dst_num_blocks,
                          int32_t num_layers, int64_t block_bytes, void *stream);

/*
 * Paged decode attention without a caller workspace.  The pages have no
 * counterpart: this exists for callers that cannot allocate device memory,
 * for instance an engine whose allocator owns all of the GPU's memory for its
 * KV-cache pool, or a latency-critical caller that must not call cudaMalloc
 * or cudaFree (they can synchronise the device).
 *
 * Same arguments and result as pkv_paged_decode_attention, minus the
 * workspace.  The split partials go to a fixed device array of
 * PKV_NOALLOC_SCRATCH_BYTES that every GPU loading the library holds until
 * the process exits; nothing is allocated per call.  The call picks its
 * kernel as the regular call does; if that kernel needs more scratch than
 * the maximum (the CUDA-core split kernel on a large batch of long contexts
 * can), the call is rejected before anything is launched, with
 * PKV_ERR_WORKSPACE and a message in pkv_last_error.  The first call in a
 * device's context looks up the array's device address
 * (cudaGetSymbolAddress) and caches it, keyed by the context, under a lock
 * (first calls from several host threads are safe); make that first call
 * before any stream capture.  All calls on a device share the one array:
 * calls whose kernels overlap on the GPU (on different streams, unordered)
 * race and give wrong results.  The array keeps the last call's contents;
 * nothing in it needs to start at zero.
 */
#define PKV_NOALLOC_SCRATCH_BYTES (16u * 1024u * 1024u)
PKV_API pkv_status pkv_paged_decode_attention_noalloc(
    const void *q, const void *k_cache, const void *v_cache,
    const int32_t *block_tables, int32_t max_blocks_per_seq, int32_t num_blocks,
    const int32_t *context_lens, int32_t num_seqs, int32_t max_context,
    int32_t block_size, float scale, pkv_heads heads, void *out, void *stream);

/*
 * Which decode kernel later calls use: 0 automatic (the default: the
 * tensor-core kernel wherever it applies -- contiguous layout, or a paged
 * block size that is a multiple of 16 -- and the batch holds at least 8
 * sixteen-token tiles per SM when every context is max_context long; else
 * the split kernel, which fills the GPU better for small batches), 1 always the
 * split (CUDA-core) kernel, 2 / 3 the tensor-core kernel with 8 warps x 3
 * stages / 12 warps x 2 stages per CTA (the automatic choice uses 12 x 2;
 * PKV_ERR_UNSUPPORTED where the kernel does not apply).  Meant for tests and
 * tuning; every kernel computes the same result.
 */
PKV_API void pkv_set_decode_variant(int variant);
PKV_API int pkv_get_decode_variant(void);

/*
 * Test hook for the bounded waits.  The next tensor-core decode call makes
 * one warp wait for 16 bytes that never arrive: that wait gives up after its
 * time limit (2 s), the call records PKV_DEVERR_TIMEOUT in the device error
 * word, the output of that call is undefined, and the context stays usable.
 */
PKV_API void pkv_debug_stall_next_decode(void);

/*
 * Test hook for the bounded wait of the in-kernel pair merge.  In the next
 * tensor-core decode call, CTA 1 does not write the record of its first
 * piece (a pair whose first tiles belong to CTA 0): CTA 0's merge re-reads
 * the record until its time limit (2 s), the call records
 * PKV_DEVERR_TIMEOUT, that pair's output is undefined, and the context
 * stays usable.
 */
PKV_API void pkv_debug_drop_next_piece_record(void);

/*
 * Test-only gather: out[i][h][pos] (bf16 [num_seqs][Hkv][max_context][128])
 * = the cache row that the decode kernels read for position pos of sequence
 * i and KV head h, zeros for pos >= context_lens[i].  It locates rows with
 * the same address function as the decode and append kernels, so a
 * byte-for-byte comparison with a plain gather pins the block-table
 * indexing ("Running Out of Cache": positions map to (block, offset) as
 * virtual addresses map to frames) and the reqId x S rule of the contiguous
 * layout ("Leveraging Low-Level CUDA APIs for vAttention's Dynamic Memory"
 * 5.2.3).  Arguments as for the decode calls; checked mode reports and
 * zero-fills rows with an out-of-range block id or request id.
 */
PKV_API pkv_status pkv_debug_gather_paged(
    const void *cache, const int32_t *block_tables, int32_t max_blocks_per_seq,
    int32_t num_blocks, const int32_t *context_lens, int32_t num_seqs,
    int32_t max_context, int32_t block_size, int32_t num_kv_heads, void *out,
    void *stream);
PKV_API pkv_status pkv_debug_gather_contig(
    const void *buf, const int32_t *req_ids, int32_t max_reqs,
    const int32_t *context_lens, int32_t num_seqs, int32_t max_context,
    int64_t S, int32_t num_kv_heads, void *out, void *stream);

/* Checked mode on (1) or off (0, the default) for later calls. */
PKV_API void pkv_set_checked(int enable);
PKV_API int pkv_get_checked(void);

/*
 * Tokens-per-split override in units of 16-token tiles (0 restores the
 * automatic rule).  Changes pkv_decode_num_splits/_workspace_size for later
 * calls; meant for tuning and tests.
 */
PKV_API void pkv_set_split_tiles(int32_t tiles);

/*
 * Reads and clears the error word of the current device (synchronises the
 * device).  *code_out receives a PKV_DEVERR_* code.  Returns PKV_OK when the
 * word was clear, PKV_ERR_DEVICE_BOUNDS when it held an error, PKV_ERR_CUDA
 * if the read failed.
 */
PKV_API pkv_status pkv_get_device_error(int *code_out);

/* Static description of a status code. */
PKV_API const char *pkv_status_string(pkv_status status);

/* Detail message of the last failing call on this host thread ("" if none). */
PKV_API const char *pkv_last_error(void);

#ifdef __cplusplus
}
#endif

#endif /* PKV_H */
