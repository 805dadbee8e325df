// kv_ops.cu -- the two data-movement kernels of a decode step: KV append
// (write each new token's K/V row into its cache slot) and the
// copy-on-write block copy.  Both move bytes unchanged (bit-exact) with
// 16-byte vector loads and stores.
#include "kv_ops.cuh"
#include "pkv_device.cuh"

namespace pkv {

// One 16-lane group per 256-byte row; a 256-thread CTA moves 16 rows.
// Rows are numbered (which in {K, V}, token t, KV head h), K first.
__global__ void __launch_bounds__(256) kv_append_kernel(const AppendParams p) {
  grid_dependency_trigger();
  grid_dependency_wait();
  const int64_t row = static_cast<int64_t>(blockIdx.x) * 16 + (threadIdx.x >> 4);
  const int lane16 = threadIdx.x & 15;
  const int64_t per_kind = p.num_tokens * p.Hkv;
  if (row >= 2 * per_kind) return;
  const bool is_v = row >= per_kind;
  const int64_t r = is_v ? row - per_kind : row;
  const int64_t t = r / p.Hkv;
  const int64_t h = r % p.Hkv;
  const int64_t slot = p.slot_mapping[t];
  if (slot < 0) return;  // padding token
  if (slot >= p.num_slots && p.checked) {
    if (lane16 == 0 && !is_v) record_error(p.err, kErrSlot);
    return;
  }
  const int64_t blk = slot / p.bs;
  const int64_t off = slot % p.bs;
  const uint16_t* src = (is_v ? p.v : p.k) + (t * p.Hkv + h) * kHeadDim + lane16 * 8;
  uint16_t* dst = (is_v ? p.v_cache : p.k_cache) + cache_row(blk, h, p.Hkv, p.bs, off) * kHeadDim +
                  lane16 * 8;
  *reinterpret_cast<uint4*>(dst) = ld_global_nc_v4(src);
}

cudaError_t launch_kv_append(const AppendParams& p, cudaStream_t stream, bool plain) {
  const int64_t rows = 2 * p.num_tokens * p.Hkv;
  if (rows == 0) return cudaSuccess;
  const int64_t blocks = (rows + 15) / 16;
  return launch_pdl_if(!plain && pdl_enabled(), kv_append_kernel,
                       dim3(static_cast<unsigned>(blocks)), dim3(256), 0, stream, p);
}

// Gather: one 16-lane group per (sequence, KV head, position) row, as the
// append moves rows; positions past the context are zero-filled.
__global__ void __launch_bounds__(256) gather_kernel(const GatherParams p) {
  grid_dependency_trigger();
  grid_dependency_wait();
  const int64_t row = static_cast<int64_t>(blockIdx.x) * 16 + (threadIdx.x >> 4);
  const int lane16 = threadIdx.x & 15;
  const int64_t rows = static_cast<int64_t>(p.num_seqs) * p.Hkv * p.max_context;
  if (row >= rows) return;
  const int64_t pos = row % p.max_context;
  const int64_t h = (row / p.max_context) % p.Hkv;
  const int64_t i = row / (static_cast<int64_t>(p.max_context) * p.Hkv);
  uint4* dst = reinterpret_cast<uint4*>(p.out + row * kHeadDim) + lane16;
  const int ctx = p.ctx_lens[i];
  if (pos >= ctx) {
    *dst = make_uint4(0u, 0u, 0u, 0u);
    return;
  }
  int64_t block, off;
  if (p.block_tables != nullptr) {
    block = p.block_tables[i * p.max_blocks + pos / p.bs];
    off = pos % p.bs;
  } else {
    block = p.req_ids[i];
    off = pos;
  }
  if (p.checked && (block < 0 || block >= p.num_blocks)) {
    if (lane16 == 0) record_error(p.err, p.block_tables != nullptr ? kErrBlockId : kErrReqId);
    *dst = make_uint4(0u, 0u, 0u, 0u);
    return;
  }
  *dst = ld_global_nc_v4(p.cache + cache_row(block, h, p.Hkv, p.bs, off) * kHeadDim + lane16 * 8);
}

cudaError_t launch_gather(const GatherParams& p, cudaStream_t stream) {
  const int64_t rows = static_cast<int64_t>(p.num_seqs) * p.Hkv * p.max_context;
  if (rows == 0) return cudaSuccess;
  return launch_pdl(gather_kernel, dim3(static_cast<unsigned>((rows + 15) / 16)), dim3(256), 0,
                    stream, p);
}

// Block copy (within one pool) and block swap (between two): blockIdx.x
// strides over the block's 16-byte chunks, blockIdx.y is the pair,
// blockIdx.z = 2 * layer + (0 for K, 1 for V).
__global__ void __launch_bounds__(256) block_copy_kernel(const CopyParams p) {
  grid_dependency_trigger();
  grid_dependency_wait();
  const int64_t pair = blockIdx.y;
  const int layer = blockIdx.z >> 1;
  const bool is_v = blockIdx.z & 1;
  const int64_t src = p.pairs[2 * pair];
  const int64_t dst = p.pairs[2 * pair + 1];
  if (p.checked && (src < 0 || src >= p.num_blocks || dst < 0 || dst >= p.dst_num_blocks)) {
    if (threadIdx.x == 0 && blockIdx.x == 0) record_error(p.err, kErrCopyPair);
    return;
  }
  const unsigned char* sbase = static_cast<const unsigned char*>(is_v ? p.v[layer] : p.k[layer]);
  unsigned char* dbase = static_cast<unsigned char*>(is_v ? p.dv[layer] : p.dk[layer]);
  const uint4* s = reinterpret_cast<const uint4*>(sbase + src * p.block_bytes);
  uint4* d = reinterpret_cast<uint4*>(dbase + dst * p.block_bytes);
  const int64_t n16 = p.block_bytes / 16;
  constexpr int kUnroll = 4;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  for (; i + (kUnroll - 1) * stride < n16; i += kUnroll * stride) {
    uint4 v[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) v[u] = ld_global_nc_v4(s + i + u * stride);
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) d[i + u * stride] = v[u];
  }
  for (; i < n16; i += stride) d[i] = ld_global_nc_v4(s + i);
}

cudaError_t launch_block_copy(const CopyParams& p, int64_t num_pairs, cudaStream_t stream) {
  if (num_pairs == 0 || p.num_layers == 0) return cudaSuccess;
  const int64_t n16 = p.block_bytes / 16;
  int64_t bx = (n16 + 256 * 4 - 1) / (256 * 4);
  if (bx < 1) bx = 1;
  if (bx > 64) bx = 64;
  const dim3 grid(static_cast<unsigned>(bx), static_cast<unsigned>(num_pairs),
                  static_cast<unsigned>(2 * p.num_layers));
  return launch_pdl(block_copy_kernel, grid, dim3(256), 0, stream, p);
}

}  // namespace pkv
