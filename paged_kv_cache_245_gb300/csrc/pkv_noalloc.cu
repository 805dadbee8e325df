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
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdio>
#include <mutex>

#include "../../include/pkv.h"

namespace pkv {
void set_last_error_message(const char* msg);
}

// The scratch: PKV_NOALLOC_SCRATCH_BYTES of device memory, reserved on every
// GPU that loads this part of the library and held until the process exits.
static __device__ __align__(256) float g_noalloc_scratch[PKV_NOALLOC_SCRATCH_BYTES / sizeof(float)];

namespace {

constexpr int kMaxDevices = 64;

// The array's device address, per device, together with the id of the CUDA
// context it was looked up in.  A device's primary context can be destroyed
// and created anew (cudaDeviceReset); the module, and with it the array, is
// then loaded again at another address, so an entry is only used while its
// context id still matches the current one.  The mutex makes concurrent
// first calls from several host threads safe.
struct ScratchEntry {
  unsigned long long ctx_id = 0;
  void* addr = nullptr;
};
std::mutex g_scratch_mu;
ScratchEntry g_scratch[kMaxDevices];

using CtxGetCurrentFn = CUresult (*)(CUcontext*);
using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long*);

struct CtxIdQuery {
  CtxGetCurrentFn get_current = nullptr;
  CtxGetIdFn get_id = nullptr;
};

const CtxIdQuery& ctx_query() {
  static CtxIdQuery q;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult r = cudaDriverEntryPointSymbolNotFound;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 12000, cudaEnableDefault, &r) ==
            cudaSuccess && r == cudaDriverEntryPointSuccess)
      q.get_current = reinterpret_cast<CtxGetCurrentFn>(f);
    f = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &f, 12000, cudaEnableDefault, &r) ==
            cudaSuccess && r == cudaDriverEntryPointSuccess)
      q.get_id = reinterpret_cast<CtxGetIdFn>(f);
  });
  return q;
}

// Id of the current context, 0 when there is none yet or it cannot be told.
unsigned long long current_ctx_id() {
  const CtxIdQuery& q = ctx_query();
  if (q.get_current == nullptr || q.get_id == nullptr) return 0;
  CUcontext ctx = nullptr;
  if (q.get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr) return 0;
  unsigned long long id = 0;
  if (q.get_id(ctx, &id) != CUDA_SUCCESS) return 0;
  return id;
}

// Device address of the scratch on the current device.  In host code the
// array's name is only a host-side stand-in, so the address is looked up
// (with the device current) on the first call in a context and cached.
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
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  ScratchEntry& ent = g_scratch[dev];
  const unsigned long long id = current_ctx_id();
  if (ent.addr != nullptr && id != 0 && ent.ctx_id == id) {
    *out = ent.addr;
    return PKV_OK;
  }
  void* ptr = nullptr;
  e = cudaGetSymbolAddress(&ptr, g_noalloc_scratch);
  if (e != cudaSuccess || ptr == nullptr) {
    char msg[160];
    snprintf(msg, sizeof msg, "noalloc: cudaGetSymbolAddress(scratch) failed: %s",
             cudaGetErrorString(e));
    pkv::set_last_error_message(msg);
    return PKV_ERR_CUDA;
  }
  // the lookup created the context if there was none: take its id now
  ent.ctx_id = id != 0 ? id : current_ctx_id();
  ent.addr = ptr;
  *out = ptr;
  return PKV_OK;
}

}  // namespace

extern "C" PKV_API pkv_status pkv_paged_decode_attention_noalloc(
    const void* q, const void* k_cache, const void* v_cache, const int32_t* block_tables,
    int32_t max_blocks_per_seq, int32_t num_blocks, const int32_t* context_lens,
    int32_t num_seqs, int32_t max_context, int32_t block_size, float scale, pkv_heads heads,
    void* out, void* stream) {
  void* scratch = nullptr;
  if (num_seqs > 0) {
    const pkv_status st = scratch_address(&scratch);
    if (st != PKV_OK) return st;
  }
  // The whole array is offered as the workspace.  The regular call picks its
  // kernel and checks that kernel's need against the size before anything
  // is launched, so a batch is turned away only when the kernel that would
  // run needs more.  Every partial a kernel reads back is written by the same
  // call first, and the tensor-core kernel leaves each of its flags at 0 (the
  // array starts zeroed), so the scratch needs no clearing between calls.
  const pkv_status st = pkv_paged_decode_attention(
      q, k_cache, v_cache, block_tables, max_blocks_per_seq, num_blocks, context_lens, num_seqs,
      max_context, block_size, scale, heads, out, scratch,
      scratch != nullptr ? static_cast<size_t>(PKV_NOALLOC_SCRATCH_BYTES) : 0, stream);
  if (st == PKV_ERR_WORKSPACE) {
    char msg[320];
    snprintf(msg, sizeof msg,
             "noalloc: the kernel this batch runs needs more split scratch than the fixed maximum "
             "of %zu bytes (%s); use pkv_paged_decode_attention with a workspace",
             static_cast<size_t>(PKV_NOALLOC_SCRATCH_BYTES), pkv_last_error());
    pkv::set_last_error_message(msg);
  }
  return st;
}
