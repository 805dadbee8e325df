// pkv_noalloc.cu -- paged decode attention for callers that must not allocate
// device memory.
//
// The regular entry point asks the caller for a workspace that holds the
// per-split partial results.  Some callers cannot provide one: a serving
// engine that has handed nearly all of the GPU's memory to its own KV-cache
// pool and allows no other allocation, or a latency-critical caller for
// which cudaMalloc/cudaFree (which may synchronise the device) are off
// limits.  This file gives them a variant whose partials live in a fixed
// array in device memory, declared below; nothing is allocated per call.
#include <cuda_runtime.h>

#include <cstdio>

#include "../../include/pkv.h"

namespace pkv {
void set_last_error_message(const char* msg);
}

// The scratch: PKV_NOALLOC_SCRATCH_BYTES of device memory, reserved on every
// GPU that loads this part of the library and held until the process exits.
static __device__ __align__(256) float g_noalloc_scratch[PKV_NOALLOC_SCRATCH_BYTES / sizeof(float)];

namespace {

constexpr int kMaxDevices = 64;
void* g_scratch_addr[kMaxDevices] = {};

// Device address of the scratch on the current device.  In host code the
// array's name is only a host-side stand-in, so the address is looked up
// once per device (with that device current) and cached.
pkv_status scratch_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) {
    pkv::set_last_error_message("noalloc: cudaGetDevice failed");
    return PKV_ERR_CUDA;
  }
  if (dev < 0 || dev >= kMaxDevices) {
    pkv::set_last_error_message("noalloc: device id out of range");
    return PKV_ERR_UNSUPPORTED;
  }
  if (g_scratch_addr[dev] == nullptr) {
    void* ptr = nullptr;
    e = cudaGetSymbolAddress(&ptr, g_noalloc_scratch);
    if (e != cudaSuccess || ptr == nullptr) {
      char msg[160];
      snprintf(msg, sizeof msg, "noalloc: cudaGetSymbolAddress(scratch) failed: %s",
               cudaGetErrorString(e));
      pkv::set_last_error_message(msg);
      return PKV_ERR_CUDA;
    }
    g_scratch_addr[dev] = ptr;
  }
  *out = g_scratch_addr[dev];
  return PKV_OK;
}

}  // namespace

extern "C" PKV_API pkv_status pkv_paged_decode_attention_noalloc(
    const void* q, const void* k_cache, const void* v_cache, const int32_t* block_tables,
    int32_t max_blocks_per_seq, int32_t num_blocks, const int32_t* context_lens,
    int32_t num_seqs, int32_t max_context, int32_t block_size, float scale, pkv_heads heads,
    void* out, void* stream) {
  // Same split plan as the regular call; its partials must fit the scratch.
  const size_t need = (num_seqs > 0 && max_context >= 0)
                          ? pkv_decode_workspace_size(num_seqs, heads, max_context)
                          : 0;
  if (need > PKV_NOALLOC_SCRATCH_BYTES) {
    char msg[200];
    snprintf(msg, sizeof msg,
             "noalloc: this batch needs %zu bytes of split scratch, above the fixed maximum of "
             "%zu bytes; use pkv_paged_decode_attention with a workspace",
             need, static_cast<size_t>(PKV_NOALLOC_SCRATCH_BYTES));
    pkv::set_last_error_message(msg);
    return PKV_ERR_WORKSPACE;
  }
  void* scratch = nullptr;
  size_t scratch_bytes = 0;
  if (need > 0) {
    const pkv_status st = scratch_address(&scratch);
    if (st != PKV_OK) return st;
    scratch_bytes = PKV_NOALLOC_SCRATCH_BYTES;
  }
  // Every partial the split-combine reads is written by the same call first,
  // so the scratch needs no clearing between calls.
  return pkv_paged_decode_attention(q, k_cache, v_cache, block_tables, max_blocks_per_seq,
                                    num_blocks, context_lens, num_seqs, max_context, block_size,
                                    scale, heads, out, scratch, scratch_bytes, stream);
}
