// decode_tc.cu -- host launch of the tensor-core / stream-K decode kernels:
// tensor-map encoding, batch chunking, kernel instantiations.
#include <cudaTypedefs.h>

#include <atomic>
#include <chrono>
#include <cstdlib>
#include <mutex>
#include <random>

#include "decode_tc.cuh"
#include "decode_tc_launch.h"

namespace pkv {

namespace {

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  });
  return fn;
}

}  // namespace

// [rows][128] bf16 viewed as a 2-D tensor; boxes of 16 rows x 64 columns
// (128 bytes), 128-byte swizzle.
bool encode_rows(CUtensorMap* map, const void* base, int64_t rows) {
  auto enc = tensor_map_encoder();
  if (enc == nullptr) return false;
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(kHeadDim), static_cast<cuuint64_t>(rows)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(kRowBytes)};
  const cuuint32_t box[2] = {64u, 16u};
  const cuuint32_t estr[2] = {1u, 1u};
  const CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims,
                         strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                         CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

namespace {

// Record tags of the launches: a counter from a per-process random start, so
// that consecutive launches differ and words left in reused memory (by
// another process or any other data) rarely carry a launch's tag.  Never 0
// (the value of a consumed record).
uint32_t next_launch_tag() {
  static std::atomic<uint32_t> counter{[] {
    std::random_device rd;
    uint64_t x = (static_cast<uint64_t>(rd()) << 32) ^ rd();
    x ^= static_cast<uint64_t>(std::chrono::steady_clock::now().time_since_epoch().count()) *
         0x9E3779B97F4A7C15ull;
    return static_cast<uint32_t>(x ^ (x >> 32));
  }()};
  uint32_t t;
  do t = counter.fetch_add(1, std::memory_order_relaxed); while (t == 0);
  return t;
}

}  // namespace

// Batches above kTcMaxSeqs run as consecutive chunks reusing the workspace;
// a chunk's tile prefix (int32) must hold chunk * ceil(max_context / 16).
int tc_chunk_seqs(int max_context) {
  const int64_t max_tiles = (static_cast<int64_t>(max_context) + 15) / 16;
  int chunk = kTcMaxSeqs;
  if (max_tiles > 0 && static_cast<int64_t>(chunk) * max_tiles > 0x7fffffffLL)
    chunk = static_cast<int>(0x7fffffffLL / max_tiles);
  return chunk < 1 ? 1 : chunk;
}

namespace {

template <bool kContig, int W, int S, bool kFuse, int MH = kTcMergeHeads, int NT = 1>
cudaError_t launch_cfg(const CUtensorMap& tk, const CUtensorMap& tv, const TcParams& p0,
                       int num_ctas, cudaStream_t stream) {
  using L = TcSmem<W, S, NT, MH>;
  static unsigned long long done_mask = 0;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const unsigned long long bit = 1ull << (dev & 63);
  auto kernel = decode_tc_kernel<kContig, W, S, NT, kFuse, MH>;
  if (!(__atomic_load_n(&done_mask, __ATOMIC_ACQUIRE) & bit)) {
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, L::kTotal);
    if (e != cudaSuccess) return e;
    __atomic_fetch_or(&done_mask, bit, __ATOMIC_ACQ_REL);
  }
  const int chunk = tc_chunk_seqs(p0.max_context);
  for (int s0 = 0; s0 < p0.num_seqs; s0 += chunk) {
    TcParams p = p0;
    p.num_seqs = (p0.num_seqs - s0) < chunk ? (p0.num_seqs - s0) : chunk;
    p.q += static_cast<int64_t>(s0) * p.Hq * kHeadDim;
    p.out += static_cast<int64_t>(s0) * p.Hq * kHeadDim;
    if (p.rec_out != nullptr) p.rec_out += static_cast<int64_t>(s0) * p.Hq * kRecStride;
    p.ctx_lens += s0;
    if (p.slot_mapping != nullptr) {
      p.slot_mapping += s0;
      p.k_new += static_cast<int64_t>(s0) * p.Hkv * kHeadDim;
      p.v_new += static_cast<int64_t>(s0) * p.Hkv * kHeadDim;
    }
    if (kContig) p.req_ids += s0;
    else p.block_tables += static_cast<int64_t>(s0) * p.max_blocks;
    p.tag = next_launch_tag();  // every launch writes its piece records under a fresh tag
    e = launch_pdl_if(pdl_decode_enabled(), kernel, dim3(num_ctas), dim3(W * 32),
                      L::kTotal, stream, tk, tv, p);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace

// Per CTA: one piece record (its first segment, when that is part of a pair
// that an earlier CTA's range began) of kTcRecHeads heads, kRecStride tagged
// 64-bit words each.
size_t tc_workspace_bytes(int num_ctas) {
  return static_cast<size_t>(num_ctas) * kTcRecHeads * kRecStride * sizeof(uint64_t);
}

TcStatus launch_decode_tc(const TcParams& p_in, bool contig, const void* k, const void* v,
                          int64_t rows_total, int cfg, int num_ctas, void* workspace,
                          cudaStream_t stream, cudaError_t* cuda_err) {
  *cuda_err = cudaSuccess;
  alignas(64) CUtensorMap tk;
  alignas(64) CUtensorMap tv;
  if (!encode_rows(&tk, k, rows_total) || !encode_rows(&tv, v, rows_total))
    return TcStatus::kEncodeFailed;
  TcParams p = p_in;
  // The cost of a segment in tiles, per pass of the segment merge (4 query
  // heads a pass, or 8 with cfg 2).  Per-CTA timelines grow by about 2-3 us
  // per extra segment; sweeps of 16..48 on GB300 were fastest at 24 for one
  // pass (the ragged batch: 24 -> 16 or 32 costs 3-4 %, the Llama-3-8B shape
  // moves by 0.6 %; the Yi-6B shape in one pass of 8 heads: 29.0 / 28.8 /
  // 29.0 us at 16 / 24 / 32) and at 48 for two.  PKV_TC_SEG_COST overrides
  // the per-pass cost (0: an even split of the tiles alone).
  static const int seg_cost = [] {
    const char* v = getenv("PKV_TC_SEG_COST");
    const int x = v != nullptr ? atoi(v) : 24;
    return x < 0 ? 0 : (x > 2048 ? 2048 : x);
  }();
  // cfg 2 (groups of more than 4 query heads): 10 warps x 2 stages, whose
  // shared memory holds every warp's partials of all 8 heads: one merge pass
  const int mh = cfg == 2 && p.G > kTcMergeHeads ? 8 : kTcMergeHeads;
  p.seg_cost = seg_cost * ((p.G + mh - 1) / mh);
  p.rec = static_cast<uint64_t*>(workspace);
  cudaError_t e;
  const bool fuse = p.slot_mapping != nullptr;  // the decode step with its append
#define PKV_TC_LAUNCH(C, W, S, F, M) launch_cfg<C, W, S, F, M>(tk, tv, p, num_ctas, stream)
#define PKV_TC_PICK(C, F)                                                             \
  (mh == 8 ? PKV_TC_LAUNCH(C, 10, 2, F, 8)                                            \
           : (cfg == 0 ? PKV_TC_LAUNCH(C, 8, 3, F, 4) : PKV_TC_LAUNCH(C, 12, 2, F, 4)))
  if (p.G > kTcHeads) {  // one n-tile of 8 query heads per KV head (the API allows G <= 8)
    e = cudaErrorInvalidValue;
  } else if (fuse) {
    e = contig ? PKV_TC_PICK(true, true) : PKV_TC_PICK(false, true);
  } else {
    e = contig ? PKV_TC_PICK(true, false) : PKV_TC_PICK(false, false);
  }
#undef PKV_TC_PICK
#undef PKV_TC_LAUNCH
  *cuda_err = e;
  return e == cudaSuccess ? TcStatus::kOk : TcStatus::kCudaError;
}

}  // namespace pkv
