// decode_tc_launch.h -- host interface of the tensor-core / stream-K decode
// path (decode_tc.cu).
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace pkv {

constexpr int kTcMaxSeqs = 512;  // sequences per launch (larger batches run in chunks)
constexpr int kRecStride = 132;  // floats per head record: o[128], m, l, pad

struct TcParams {
  const uint16_t* q;        // [B][Hq][128]
  uint16_t* out;            // [B][Hq][128]
  const int32_t* ctx_lens;  // [B]
  const int32_t* block_tables;  // paged [B][max_blocks]
  const int32_t* req_ids;       // contig [B]
  float* rec;               // [gridDim.x][2][8][kRecStride]
  int32_t* prefix_out;      // [B + 1] tile prefix per sequence (CTA 0 writes it)
  int64_t bs;               // paged block size (multiple of 16); contig S
  int64_t num_blocks;       // paged pool size (checked mode)
  int32_t max_blocks, max_reqs;
  int32_t num_seqs, Hq, Hkv, G, max_context;
  float qscale;             // scale * log2(e)
  int32_t checked;
  int32_t stall_test;       // test hook: CTA 0's warp 0 expects 16 bytes that never come
  int* err;
};


enum class TcStatus { kOk, kEncodeFailed, kCudaError };

// Static partition of the flattened tile list [0, T) over P CTAs: CTA c owns
// [floor(c*T/P), floor((c+1)*T/P)).
__host__ __device__ inline int64_t tc_range_lo(int64_t c, int64_t T, int64_t P) {
  return c * T / P;
}

// The CTA that owns tile x (the largest c with range_lo(c) <= x).
__host__ __device__ inline int64_t tc_owner(int64_t x, int64_t T, int64_t P) {
  return ((x + 1) * P + T - 1) / T - 1;
}

// Workspace bytes for the per-CTA partial records and the tile prefix.
size_t tc_workspace_bytes(int num_ctas);

// cfg 0: 8 warps x 3 stages per CTA; cfg 1: 12 warps x 2 stages.
TcStatus launch_decode_tc(const TcParams& p, bool contig, const void* k, const void* v,
                          int64_t rows_total, int cfg, int num_ctas, void* workspace,
                          cudaStream_t stream, cudaError_t* cuda_err);

}  // namespace pkv
