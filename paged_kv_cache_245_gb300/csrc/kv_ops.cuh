// kv_ops.cuh -- parameters and launchers of the KV append and block copy
// kernels.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace pkv {

struct AppendParams {
  const int64_t* slot_mapping;  // [T]
  const uint16_t* k;            // [T][Hkv][128]
  const uint16_t* v;
  uint16_t* k_cache;            // [.][Hkv][bs][128]
  uint16_t* v_cache;
  int64_t num_tokens;
  int64_t num_slots;
  int64_t bs;
  int64_t Hkv;
  int32_t checked;
  int* err;
};

constexpr int kMaxCopyLayers = 64;  // layers per launch (pointers passed by value)

struct CopyParams {
  const int64_t* pairs;  // [n][2] (src, dst)
  void* k[kMaxCopyLayers];   // source pools
  void* v[kMaxCopyLayers];
  void* dk[kMaxCopyLayers];  // destination pools (the sources for a copy on write)
  void* dv[kMaxCopyLayers];
  int32_t num_layers;    // <= kMaxCopyLayers for this launch
  int64_t num_blocks;     // source ids in checked mode
  int64_t dst_num_blocks; // destination ids in checked mode
  int64_t block_bytes;
  int32_t checked;
  int* err;
};

// Test-only gather of the logical rows: out[i][h][pos] = the cache row the
// attention kernels read for position pos of sequence i, KV head h (zeros at
// pos >= context_lens[i]).  Paged: block_tables; contiguous (block_tables
// null): req_ids with bs = S.
struct GatherParams {
  const uint16_t* cache;
  const int32_t* block_tables;  // [num_seqs][max_blocks] (paged)
  const int32_t* req_ids;       // [num_seqs] (contiguous)
  const int32_t* ctx_lens;      // [num_seqs]
  uint16_t* out;                // [num_seqs][Hkv][max_context][128]
  int64_t bs;
  int64_t num_blocks;           // paged pool size / max_reqs (bounds in checked mode)
  int32_t max_blocks, num_seqs, Hkv, max_context;
  int32_t checked;
  int* err;
};

cudaError_t launch_gather(const GatherParams& p, cudaStream_t stream);

// plain: launch in stream order even when PKV_PDL=1 (a decode step's append,
// whose dependent attention kernel reads its inputs before waiting)
cudaError_t launch_kv_append(const AppendParams& p, cudaStream_t stream, bool plain = false);
cudaError_t launch_block_copy(const CopyParams& p, int64_t num_pairs, cudaStream_t stream);

}  // namespace pkv
