// prefix.cuh -- parameters and launcher of the shared-prefix attention kernel
// (prefix.cu): every group's (member, query head) rows against the group's
// shared blocks, once for all members, as fp32 (o, m, l) records.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace pkv {

constexpr int kPrefixRecStride = 132;  // floats per record: o[128] / l, m, l, pad

struct PrefixParams {
  const uint16_t* q;             // [B][Hq][128]: one decode query per sequence
  const int32_t* group_start;    // [num_groups + 1]: groups of consecutive sequences
  const int32_t* shared_blocks;  // [num_groups]: leading table entries a group shares
  const int32_t* block_tables;   // [B][max_blocks] (a group reads its first member's)
  // [num_groups][chunks][2][Hkv][rows][kPrefixRecStride]: chunk k of a group's
  // shared positions, key tiles split between two halves (even / odd tiles)
  float* rec_out;
  int64_t bs;                    // block size, a multiple of 16
  int64_t num_blocks;
  int32_t max_blocks, num_groups, Hq, Hkv, G;
  int32_t rows;                  // record rows per (group, chunk, half, KV head): max group x G
  int32_t chunks;                // chunks per group (bound)
  int32_t chunk_keys;            // positions per chunk, a multiple of 128
  int32_t run_rows;              // rows per TMA box: gcd(bs, 128)
  float qscale;                  // scale * log2(e)
  // Own positions (a member's positions after its group's shared blocks),
  // attended as extra key tiles of a group's last chunk when own_slots > 0:
  // member k of the row block (k = row / G - first member) owns key slots
  // [k * own_slots, k * own_slots + n_k) of those tiles, n_k = ctx - shared
  // positions (at most own_cap), and its rows see only those slots.
  const int32_t* ctx;            // [B] context lengths (own_slots > 0)
  int32_t own_slots;             // slots per member, a multiple of run_rows; 0: none
  int32_t own_cap;               // host bound on n_k (checked mode reports a larger one)
  // fused (own_slots > 0 and one chunk per group): the CTA merges its two
  // halves and writes the bf16 output [B][Hq][128] here instead of records
  uint16_t* out;
  int32_t checked;
  int* err;
};

// Grid (ceil(rows / 128), Hkv, num_groups * chunks).  The K/V tensor maps come
// from encode_prefill_runs (prefill.cuh).
cudaError_t launch_prefix(const CUtensorMap& tk, const CUtensorMap& tv, const PrefixParams& p,
                          cudaStream_t stream);

}  // namespace pkv
