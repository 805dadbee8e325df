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
  int32_t tile_rows;             // query rows of a row tile: whole tokens, (128 / G) G
  float qscale;                  // scale * log2(e)
  int32_t out_tma;               // output rows by tensor stores (G divides 32), else plain stores
  int32_t out_v8;                // plain stores of 32 bytes (out 32-byte aligned), else 16
  int32_t checked;
  int* err;
};

// The K or V cache ([rows][128] bf16) as a 4-D tensor (64 columns, 8 rows,
// 2 column halves, row groups of 8) whose boxes of run_rows rows land in
// shared memory as 8-row x 128-byte atoms, 128-byte swizzled, ordered
// (row group, half): the layout the prefill MMAs read.  False when the
// driver rejects the map.
bool encode_prefill_runs(CUtensorMap* map, const void* base, int64_t rows, int run_rows);

// q or out ([num_tokens][Hq][128] bf16) as a 4-D tensor (64 columns, 2
// column halves, Hq heads, tokens) whose box of box_rows / G tokens x G heads
// x 64 columns is one column half of box_rows rows (token major, head
// minor), 128-byte swizzled: a Q tile's half (box_rows 128) or one warp's
// output rows (32).  False when G does not divide box_rows or the driver
// rejects the map.
bool encode_prefill_rows(CUtensorMap* map, const void* base, int64_t num_tokens, int Hq, int G,
                         int box_rows);

// A persistent grid (one CTA per SM) over the (two row tiles of tile_rows
// query rows, KV head, sequence) items.
cudaError_t launch_prefill(const CUtensorMap& tk, const CUtensorMap& tv, const CUtensorMap& tq,
                           const CUtensorMap& to, const PrefillParams& p, cudaStream_t stream);

}  // namespace pkv
