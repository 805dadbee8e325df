// cascade.cuh -- parameters and launchers of the shared-prefix decode path
// (cascade.cu): the own-position tables for the tensor-core pass, and the
// merge of the prefix and own (o, m, l) parts.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "decode_tc_launch.h"

namespace pkv {

struct CascadeParams {
  // the caller's batch
  const uint16_t* q;             // [B][Hq][128]
  const int32_t* ctx;            // [B]
  const int32_t* block_tables;   // [B][max_blocks]
  const int32_t* group_start;    // [num_groups + 1], 0 .. B ascending
  const int32_t* shared_blocks;  // [num_groups]: leading table entries the group shares
  uint16_t* out;                 // [B][Hq][128]
  int32_t B, Hq, Hkv, G, max_blocks, num_groups;
  int32_t bs;
  int32_t checked;
  int* err;
  // own positions attended in the merge kernel (own_cap >= 0: at most own_cap
  // of them per sequence), else (-1) by a tensor-core pass into rec_s
  const uint16_t* k_cache;
  const uint16_t* v_cache;
  float qscale;                  // scale * log2(e)
  int32_t own_cap;
  // own positions attended by the prefix kernel as extra key tiles of each
  // group's last chunk: its records hold them, nothing is attended here
  int32_t own_in_prefix;
  // workspace
  int32_t* tables_s;  // [B][max_blocks]
  int32_t* ctx_s;     // [B]
  float* rec_p;       // [num_groups][prefix_chunks][2][Hkv][prefix_rows][kRecStride] (prefix kernel)
  float* rec_s;       // [B][Hq][kRecStride]
  int32_t prefix_rows;        // largest group x G: record rows per (group, chunk, KV head)
  int32_t prefix_chunks;      // chunks of the shared positions per group (bound)
  int32_t prefix_chunk_keys;  // positions per chunk, a multiple of 128
};

cudaError_t launch_cascade_prep(const CascadeParams& c, cudaStream_t stream);
cudaError_t launch_cascade_merge(const CascadeParams& c, cudaStream_t stream);

}  // namespace pkv
