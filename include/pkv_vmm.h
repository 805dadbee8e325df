/*
 * pkv_vmm.h -- contiguous per-request KV buffers backed by physical memory on
 * demand (the vAttention layout).
 *
 * "Leveraging Low-Level CUDA APIs for vAttention's Dynamic Memory" (5.2.3):
 * each layer's K (and V) cache is one virtually contiguous tensor; request
 * reqId's sub-tensor starts at offset reqId x S; physical memory is mapped
 * into the virtual range as the request's context grows, through the CUDA
 * virtual memory management calls (reserve an address range, create
 * physical allocations, map them, set access), and unmapped when it ends.
 * "Insights into LLM Serving Systems: KV-Cache Memory Allocation Patterns"
 * (section 4): decode grows every request by one token per iteration, and
 * the allocation rate a layer needs stays within a few hundred MB/s.
 *
 * A buffer holds K and V tensors of shape [max_reqs][Hkv][S][128] bf16 (the
 * layout pkv_contig_decode_attention, pkv_contig_decode_step and
 * pkv_kv_append with block_size = S read and write).  Pages of the
 * allocation granularity (pkv_vmm_stats) are mapped for both tensors at
 * once.  pkv_vmm_ensure(b, r, n) backs rows [0, n rounded up to 16) of every
 * KV head of request r -- the rows a decode call over n positions (and an
 * append at position n - 1) can touch.  Kernels must touch only backed rows:
 * call pkv_vmm_ensure before the calls that grow a request, and never pass a
 * context longer than pkv_vmm_backed_tokens.  pkv_vmm_release and
 * pkv_vmm_destroy synchronise the device before they unmap anything.
 * Unmapped physical pages are kept for reuse until pkv_vmm_destroy.  Not
 * thread-safe.  Host calls only; they return PKV_ERR_CUDA (message in
 * pkv_last_error) when a driver call fails, e.g. out of device memory.
 */
#ifndef PKV_VMM_H_
#define PKV_VMM_H_

#include "pkv.h"

#ifdef __cplusplus
extern "C" {
#endif

typedef struct pkv_vmm_buffer pkv_vmm_buffer;

/* Reserves the two virtual ranges on the current device (no physical memory
 * yet).  S: tokens per request, a positive multiple of 16. */
PKV_API pkv_status pkv_vmm_create(int32_t max_reqs, int32_t num_kv_heads, int64_t S,
                                  pkv_vmm_buffer **out);
PKV_API void pkv_vmm_destroy(pkv_vmm_buffer *b);

/* Device base addresses of the K and V tensors. */
PKV_API void *pkv_vmm_k(const pkv_vmm_buffer *b);
PKV_API void *pkv_vmm_v(const pkv_vmm_buffer *b);

/* Back request req's first `tokens` positions (0 <= tokens <= S); mapping
 * only what is missing.  On failure nothing changed. */
PKV_API pkv_status pkv_vmm_ensure(pkv_vmm_buffer *b, int32_t req, int64_t tokens);
/* Drop request req's rows; pages no other request uses are unmapped. */
PKV_API pkv_status pkv_vmm_release(pkv_vmm_buffer *b, int32_t req);
/* Rows of each KV head of req that are backed (a multiple of 16), -1 if bad. */
PKV_API int64_t pkv_vmm_backed_tokens(const pkv_vmm_buffer *b, int32_t req);

/* Page size; pages mapped now; physical pages created so far; map
 * operations so far; host seconds spent in pkv_vmm_ensure.  Any output may
 * be NULL. */
PKV_API pkv_status pkv_vmm_stats(const pkv_vmm_buffer *b, size_t *page_bytes,
                                 int64_t *mapped_pages, int64_t *created_pages,
                                 int64_t *map_calls, double *map_seconds);

#ifdef __cplusplus
}
#endif

#endif /* PKV_VMM_H_ */
