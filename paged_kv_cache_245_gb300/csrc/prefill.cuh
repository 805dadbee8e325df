// prefill.cuh -- parameters and launcher of causal prefill attention over a
// paged KV cache (prefill.cu).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace pkv {

struct PrefillParams {
  const uint16_t* q;             // [T][Hq][128] the chunks' new tokens, packed
  uint16_t* out;                 // [T][Hq][128]
  const int32_t* cu_q;           // [B + 1] chunk boundaries in q
  const int32_t* ctx_lens;       // [B] positions after the chunk (cached + new)
  const int32_t* block_tables;   // [B][max_blocks]
  int64_t bs;                    // block size, a multiple of 16
  int64_t num_blocks;
  int32_t max_blocks, num_seqs, Hq, Hkv, G;
  int32_t max_q;                 // host bound on any chunk's length
  int32_t run_rows;              // rows per TMA box: gcd(bs, 128), one box per block run
  float qscale;                  // scale * log2(e)
  int32_t checked;
  int* err;
  // Shared-prefix mode (prefix != 0): item z is group z of consecutive
  // sequences group_start[z] .. group_start[z+1]-1 (q holds one decode query
  // per sequence, [B][Hq][128]); its rows are (member, query head) pairs and
  // they all attend the group's first shared_blocks[z] blocks (the first
  // member's table), with no causal mask.  Results go to rec_out as fp32
  // records of kPrefillRecStride floats: o / l, m, l (log2 units of
  // scale * log2 e); chunks past a group's shared positions write none.
  int32_t prefix;
  const int32_t* group_start;    // [num_groups + 1]
  const int32_t* shared_blocks;  // [num_groups]
  float* rec_out;
  int32_t prefix_rows;           // max group size x G
  // A group's shared positions split into chunks of prefix_chunk_keys (a
  // multiple of 128): item z is chunk z % prefix_chunks of group
  // z / prefix_chunks; records [num_groups][prefix_chunks][Hkv][prefix_rows].
  int32_t prefix_chunks;
  int32_t prefix_chunk_keys;
};

constexpr int kPrefillRecStride = 132;  // floats per record: o[128], m, l, pad

// The K or V cache ([rows][128] bf16) as a 4-D tensor (64 columns, 8 rows,
// 2 column halves, row groups of 8) whose boxes of run_rows rows land in
// shared memory as 8-row x 128-byte atoms, 128-byte swizzled, ordered
// (row group, half): the layout the prefill MMAs read.  False when the
// driver rejects the map.
bool encode_prefill_runs(CUtensorMap* map, const void* base, int64_t rows, int run_rows);

// One CTA per (256 query rows, KV head, sequence).
cudaError_t launch_prefill(const CUtensorMap& tk, const CUtensorMap& tv, const PrefillParams& p,
                           cudaStream_t stream);

}  // namespace pkv
