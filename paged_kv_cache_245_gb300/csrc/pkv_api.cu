// pkv_api.cu -- the C ABI declared in include/pkv.h: host-side validation,
// split policy, launches, checked mode and the per-device error word.
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <vector>

#include "../../include/pkv.h"
#include "decode_launch.cuh"
#include "cascade.cuh"
#include "prefill.cuh"
#include "prefix.cuh"
#include "decode_tc_launch.h"
#include "kv_ops.cuh"

namespace {

std::atomic<int> g_checked{0};
std::atomic<int> g_split_tiles{0};
// 0 automatic, 1 CUDA-core split kernel, 2 tensor-core 8x3, 3 tensor-core 12x2
std::atomic<int> g_variant{0};
std::atomic<int> g_stall_test{0};
std::atomic<int> g_drop_record_test{0};
thread_local char g_last_error[256] = "";

// The device error word: one int per device (module-scope __device__).
__device__ int g_device_error = 0;

constexpr int kMaxDevices = 64;
int* g_err_ptr[kMaxDevices] = {};
int g_num_sms[kMaxDevices] = {};

pkv_status fail(pkv_status s, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_last_error, sizeof g_last_error, fmt, ap);
  va_end(ap);
  return s;
}

pkv_status cuda_fail(cudaError_t e, const char* what) {
  return fail(PKV_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// Device id, its error-word address and SM count (cached per device).
pkv_status device_info(int* dev_out, int** err_out, int* sms_out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev < 0 || dev >= kMaxDevices) return fail(PKV_ERR_UNSUPPORTED, "device id %d", dev);
  if (g_err_ptr[dev] == nullptr) {
    void* ptr = nullptr;
    e = cudaGetSymbolAddress(&ptr, g_device_error);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(error word)");
    int sms = 0;
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceGetAttribute(SM count)");
    g_num_sms[dev] = sms;
    g_err_ptr[dev] = static_cast<int*>(ptr);
  }
  if (dev_out) *dev_out = dev;
  if (err_out) *err_out = g_err_ptr[dev];
  if (sms_out) *sms_out = g_num_sms[dev];
  return PKV_OK;
}

pkv_status check_heads(const pkv_heads& h) {
  if (h.num_q_heads <= 0 || h.num_kv_heads <= 0 || h.head_dim <= 0)
    return fail(PKV_ERR_INVALID_ARG, "head counts must be positive");
  if (h.head_dim != pkv::kHeadDim)
    return fail(PKV_ERR_UNSUPPORTED, "head_dim %d (only 128 is built)", h.head_dim);
  if (h.num_q_heads % h.num_kv_heads != 0)
    return fail(PKV_ERR_INVALID_ARG, "num_q_heads %d not a multiple of num_kv_heads %d",
                h.num_q_heads, h.num_kv_heads);
  const int g = h.num_q_heads / h.num_kv_heads;
  if (g > 8) return fail(PKV_ERR_UNSUPPORTED, "query heads per KV head %d > 8", g);
  if (h.num_kv_heads > 65535) return fail(PKV_ERR_UNSUPPORTED, "num_kv_heads > 65535");
  return PKV_OK;
}

// Split rule.  A split is a run of `chunk` 16-token tiles of one (sequence,
// KV head); a CTA handles one split.  The rule picks the chunk (a multiple
// of the warp count) that minimises a simple makespan model: waves of
// resident CTAs x (tiles per CTA + a fixed per-CTA overhead of 2 tiles),
// capped at 64 tiles so that one long context cannot dominate a batch.
int32_t choose_chunk_tiles(int32_t num_seqs, int32_t num_kv_heads, int32_t max_context,
                           int num_sms) {
  const int64_t ntiles = max_context > 0 ? (static_cast<int64_t>(max_context) + 15) / 16 : 0;
  const int forced = g_split_tiles.load();
  if (forced > 0) return forced;
  if (ntiles <= pkv::kDecodeWarps) return pkv::kDecodeWarps;
  const int64_t pairs = static_cast<int64_t>(num_seqs) * num_kv_heads;
  const int64_t slots = static_cast<int64_t>(num_sms > 0 ? num_sms : 1) * 2;
  int64_t best_chunk = pkv::kDecodeWarps;
  double best_cost = 1e300;
  const int64_t cap = 64;
  for (int64_t chunk = pkv::kDecodeWarps; chunk <= cap; chunk += pkv::kDecodeWarps) {
    const int64_t nsplit = (ntiles + chunk - 1) / chunk;
    const int64_t ctas = pairs * nsplit;
    const int64_t waves = (ctas + slots - 1) / slots;
    const int64_t used = chunk < ntiles ? chunk : ntiles;
    const double cost = static_cast<double>(waves) * static_cast<double>(used + 2);
    if (cost < best_cost - 1e-9) {
      best_cost = cost;
      best_chunk = chunk;
    }
    if (chunk >= ntiles) break;
  }
  return static_cast<int32_t>(best_chunk);
}

struct SplitPlan {
  int32_t chunk_tiles;
  int32_t nsplit;
  size_t workspace_bytes;
};

SplitPlan plan_splits(int32_t num_seqs, const pkv_heads& h, int32_t max_context, int num_sms) {
  SplitPlan s;
  s.chunk_tiles = choose_chunk_tiles(num_seqs, h.num_kv_heads, max_context, num_sms);
  const int64_t ntiles = max_context > 0 ? (static_cast<int64_t>(max_context) + 15) / 16 : 0;
  int64_t n = (ntiles + s.chunk_tiles - 1) / s.chunk_tiles;
  if (n < 1) n = 1;
  s.nsplit = static_cast<int32_t>(n);
  s.workspace_bytes = s.nsplit > 1 ? static_cast<size_t>(num_seqs) * h.num_q_heads *
                                         static_cast<size_t>(s.nsplit) *
                                         (pkv::kHeadDim + 2) * sizeof(float)
                                   : 0;
  return s;
}

// Persistent tensor-core kernel: one CTA per SM.
int tc_ctas(int num_sms) { return num_sms > 0 ? num_sms : 1; }

// Workspace the decode calls may need: the larger of the two kernels'
// requirements (the query does not know the layout or block size).
size_t decode_workspace_need(int32_t num_seqs, const pkv_heads& h, int32_t max_context,
                             int num_sms) {
  const size_t split = plan_splits(num_seqs, h, max_context, num_sms).workspace_bytes;
  const size_t tc = pkv::tc_workspace_bytes(tc_ctas(num_sms));
  return split > tc ? split : tc;
}

// A decode step's append, for the tensor-core kernel to do itself.
struct FusedAppend {
  const int64_t* slot_mapping;
  const void* k_new;
  const void* v_new;
  int64_t num_slots;
};

// Validates a decode call and, unless dry_run, launches it.  fused (the
// tensor-core kernel only): the step's append done by the attention kernel.
// *tc_out: whether the tensor-core kernel is (or would be) the one launched.
// Automatic choice: the persistent tensor-core kernel needs enough tiles to
// spread over one CTA per SM; for batches whose upper-bound tile count (all
// contexts at max_context) is under 8 tiles per SM the many-CTA split kernel
// finishes sooner.  Llama-3-8B shape, context 1024, on GB300: batch 1 (3.4
// tiles per SM) 10.6 us split / 14.4 tensor-core, batch 2 (6.7) 11.9 / 11.4,
// batch 4 (13.5) 12.8 / 11.1, batch 8 15.9 / 13.8.
bool tc_enough_tiles(int32_t num_seqs, const pkv_heads& h, int32_t max_context, int sms) {
  const int64_t tile_bound = static_cast<int64_t>(num_seqs) * h.num_kv_heads *
                             ((static_cast<int64_t>(max_context) + 15) / 16);
  return tile_bound >= 8LL * tc_ctas(sms);
}

pkv_status decode_common(bool contig, const void* q, const void* k, const void* v,
                         const int32_t* block_tables, int32_t max_blocks, int64_t num_blocks,
                         const int32_t* req_ids, int32_t max_reqs, const int32_t* context_lens,
                         int32_t num_seqs, int32_t max_context, int64_t bs_or_S, float scale,
                         pkv_heads h, void* out, void* workspace, size_t workspace_bytes,
                         void* stream, bool dry_run = false, bool* tc_out = nullptr,
                         const FusedAppend* fused = nullptr) {
  if (tc_out) *tc_out = false;
  pkv_status st = check_heads(h);
  if (st != PKV_OK) return st;
  if (num_seqs < 0 || max_context < 0) return fail(PKV_ERR_INVALID_ARG, "negative size");
  if (num_seqs == 0) return PKV_OK;
  if (num_seqs > 65535) return fail(PKV_ERR_UNSUPPORTED, "num_seqs > 65535");
  if (!q || !k || !v || !out || !context_lens)
    return fail(PKV_ERR_INVALID_ARG, "null pointer argument");
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(out, 16))
    return fail(PKV_ERR_INVALID_ARG, "bf16 tensors must be 16-byte aligned");
  if (!aligned(context_lens, 4)) return fail(PKV_ERR_INVALID_ARG, "context_lens misaligned");
  if (!std::isfinite(scale)) return fail(PKV_ERR_INVALID_ARG, "scale is not finite");
  if (bs_or_S <= 0) return fail(PKV_ERR_INVALID_ARG, contig ? "S must be >= 1" : "block_size must be >= 1");
  if (contig) {
    if (!req_ids || !aligned(req_ids, 4)) return fail(PKV_ERR_INVALID_ARG, "req_ids null or misaligned");
    if (max_reqs <= 0) return fail(PKV_ERR_INVALID_ARG, "max_reqs must be >= 1");
    if (max_context > bs_or_S) return fail(PKV_ERR_INVALID_ARG, "max_context %d > S %lld",
                                            max_context, static_cast<long long>(bs_or_S));
  } else {
    if (!block_tables || !aligned(block_tables, 4))
      return fail(PKV_ERR_INVALID_ARG, "block_tables null or misaligned");
    if (max_blocks <= 0 || num_blocks <= 0) return fail(PKV_ERR_INVALID_ARG, "empty block table or pool");
    if (static_cast<int64_t>(max_blocks) * bs_or_S < max_context)
      return fail(PKV_ERR_INVALID_ARG, "max_blocks_per_seq * block_size < max_context");
    if (static_cast<int64_t>(num_blocks) * h.num_kv_heads * bs_or_S > (int64_t{1} << 40))
      return fail(PKV_ERR_UNSUPPORTED, "cache too large");
  }
  int dev = 0, sms = 0;
  int* err = nullptr;
  st = device_info(&dev, &err, &sms);
  if (st != PKV_OK) return st;
  const int group = h.num_q_heads / h.num_kv_heads;
  const int64_t rows_total = contig ? static_cast<int64_t>(max_reqs) * h.num_kv_heads * bs_or_S
                                    : static_cast<int64_t>(num_blocks) * h.num_kv_heads * bs_or_S;
  const bool tc_ok = (contig || bs_or_S % 16 == 0) && rows_total <= 0x7fffffffLL;
  const int variant = g_variant.load();
  if (variant >= 2 && !tc_ok)
    return fail(PKV_ERR_UNSUPPORTED, "tensor-core kernel needs block_size %% 16 == 0 and < 2^31 rows");
  const bool tc_pick = variant >= 2 || (variant == 0 && tc_enough_tiles(num_seqs, h, max_context, sms));
  if (tc_pick && tc_ok) {
    if (tc_out) *tc_out = true;
    const size_t need = pkv::tc_workspace_bytes(tc_ctas(sms));
    if (!workspace || workspace_bytes < need)
      return fail(PKV_ERR_WORKSPACE, "workspace needs %zu bytes, got %zu", need,
                  workspace ? workspace_bytes : size_t{0});
    if (!aligned(workspace, 16)) return fail(PKV_ERR_WORKSPACE, "workspace must be 16-byte aligned");
    if (dry_run) return PKV_OK;
    pkv::TcParams t;
    std::memset(&t, 0, sizeof t);
    t.q = static_cast<const uint16_t*>(q);
    t.out = static_cast<uint16_t*>(out);
    t.ctx_lens = context_lens;
    t.block_tables = block_tables;
    t.req_ids = req_ids;
    t.bs = bs_or_S;
    t.num_blocks = num_blocks;
    t.max_blocks = max_blocks;
    t.max_reqs = max_reqs;
    t.num_seqs = num_seqs;
    t.Hq = h.num_q_heads;
    t.Hkv = h.num_kv_heads;
    t.G = group;
    t.max_context = max_context;
    t.qscale = scale * 1.4426950408889634f;  // log2(e)
    t.checked = g_checked.load();
    t.stall_test = g_stall_test.exchange(0);
    t.drop_record_test = g_drop_record_test.exchange(0);
    if (fused != nullptr) {
      t.slot_mapping = fused->slot_mapping;
      t.k_new = static_cast<const uint16_t*>(fused->k_new);
      t.v_new = static_cast<const uint16_t*>(fused->v_new);
      t.k_cache = static_cast<uint16_t*>(const_cast<void*>(k));
      t.v_cache = static_cast<uint16_t*>(const_cast<void*>(v));
      t.num_slots = fused->num_slots;
    }
    t.err = err;
    cudaError_t ce = cudaSuccess;
    // 8 x 3 when forced; 12 x 2 when forced or for up to 4 query heads per KV
    // head, else 10 x 2 (one merge pass for all 8 heads)
    const int cfg = variant == 2 ? 0 : (variant == 0 && group > 4 ? 2 : 1);
    const pkv::TcStatus ts = pkv::launch_decode_tc(t, contig, k, v, rows_total, cfg,
                                                   tc_ctas(sms), workspace,
                                                   static_cast<cudaStream_t>(stream), &ce);
    if (ts == pkv::TcStatus::kEncodeFailed)
      return fail(PKV_ERR_CUDA, "cuTensorMapEncodeTiled failed for the K/V cache");
    if (ts != pkv::TcStatus::kOk) return cuda_fail(ce, "decode launch");
    return PKV_OK;
  }
  const SplitPlan plan = plan_splits(num_seqs, h, max_context, sms);
  if (plan.nsplit > 65535) return fail(PKV_ERR_UNSUPPORTED, "too many splits");
  if (plan.workspace_bytes > 0) {
    if (!workspace || workspace_bytes < plan.workspace_bytes)
      return fail(PKV_ERR_WORKSPACE, "workspace needs %zu bytes, got %zu", plan.workspace_bytes,
                  workspace ? workspace_bytes : size_t{0});
    if (!aligned(workspace, 16)) return fail(PKV_ERR_WORKSPACE, "workspace must be 16-byte aligned");
  }
  if (dry_run) return PKV_OK;

  pkv::DecodeParams p;
  std::memset(&p, 0, sizeof p);
  p.q = static_cast<const uint16_t*>(q);
  p.k = static_cast<const uint16_t*>(k);
  p.v = static_cast<const uint16_t*>(v);
  p.out = static_cast<uint16_t*>(out);
  if (plan.nsplit > 1) {
    p.part_o = static_cast<float*>(workspace);
    p.part_ml = p.part_o + static_cast<size_t>(num_seqs) * h.num_q_heads * plan.nsplit * pkv::kHeadDim;
  }
  p.ctx_lens = context_lens;
  p.block_tables = block_tables;
  p.req_ids = req_ids;
  p.bs = bs_or_S;
  p.num_blocks = num_blocks;
  p.max_blocks = max_blocks;
  p.max_reqs = max_reqs;
  p.num_seqs = num_seqs;
  p.Hq = h.num_q_heads;
  p.Hkv = h.num_kv_heads;
  p.max_context = max_context;
  p.chunk_tiles = plan.chunk_tiles;
  p.nsplit = plan.nsplit;
  p.qscale = scale * 1.4426950408889634f;  // log2(e)
  p.checked = g_checked.load();
  p.err = err;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const cudaError_t e = contig ? pkv::launch_decode_contig(p, group, s)
                               : pkv::launch_decode_paged(p, group, s);
  if (e != cudaSuccess) return cuda_fail(e, "decode launch");
  return PKV_OK;
}

// Validates and launches an append.  plain: launch in stream order whatever
// PKV_PDL says (the append of a decode step).
pkv_status append_common(const int64_t* slot_mapping, int64_t num_tokens, const void* k,
                         const void* v, void* k_cache, void* v_cache, int64_t num_slots,
                         int64_t block_size, pkv_heads heads, void* stream, bool plain,
                         bool dry_run = false) {
  if (heads.num_kv_heads <= 0) return fail(PKV_ERR_INVALID_ARG, "num_kv_heads must be positive");
  if (heads.head_dim != pkv::kHeadDim)
    return fail(PKV_ERR_UNSUPPORTED, "head_dim %d (only 128 is built)", heads.head_dim);
  if (num_tokens < 0 || num_slots < 0) return fail(PKV_ERR_INVALID_ARG, "negative size");
  if (num_tokens == 0) return PKV_OK;
  if (block_size <= 0) return fail(PKV_ERR_INVALID_ARG, "block_size must be >= 1");
  if (!slot_mapping || !k || !v || !k_cache || !v_cache)
    return fail(PKV_ERR_INVALID_ARG, "null pointer argument");
  if (!aligned(slot_mapping, 8)) return fail(PKV_ERR_INVALID_ARG, "slot_mapping misaligned");
  if (!aligned(k, 16) || !aligned(v, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16))
    return fail(PKV_ERR_INVALID_ARG, "bf16 tensors must be 16-byte aligned");
  int* err = nullptr;
  pkv_status st = device_info(nullptr, &err, nullptr);
  if (st != PKV_OK) return st;
  pkv::AppendParams p;
  p.slot_mapping = slot_mapping;
  p.k = static_cast<const uint16_t*>(k);
  p.v = static_cast<const uint16_t*>(v);
  p.k_cache = static_cast<uint16_t*>(k_cache);
  p.v_cache = static_cast<uint16_t*>(v_cache);
  p.num_tokens = num_tokens;
  p.num_slots = num_slots;
  p.bs = block_size;
  p.Hkv = heads.num_kv_heads;
  p.checked = g_checked.load();
  p.err = err;
  const int64_t rows = 2 * num_tokens * heads.num_kv_heads;
  if ((rows + 15) / 16 > 0x7fffffff) return fail(PKV_ERR_UNSUPPORTED, "too many tokens");
  if (dry_run) return PKV_OK;
  const cudaError_t e = pkv::launch_kv_append(p, static_cast<cudaStream_t>(stream), plain);
  if (e != cudaSuccess) return cuda_fail(e, "kv_append launch");
  return PKV_OK;
}

// Own parts of at most this many positions are attended in the merge kernel.
constexpr int32_t kInlineOwnMax = 256;
constexpr int64_t kPrefixRowTile = 128;  // rows of a prefix-kernel row block
constexpr int64_t kOwnTileSlots = 512;   // own key slots per prefix row block (4 key tiles)

// Shared-prefix plan: prefix entries stack the heads of m sequences (m * G
// <= 16 query heads per KV head); workspace regions, 256-byte aligned.
static_assert(pkv::kPrefixRecStride == pkv::kRecStride, "one record layout for every kernel");

// Workspace of the shared-prefix call: the prefix records (one per group,
// KV head and (member, query head) row), and for own parts attended by the
// tensor-core decode pass, their tables, lengths and records.
constexpr int kMaxPrefixChunks = 8;  // chunks of a group's shared positions (bound)

// Chunk of the shared positions for the prefix kernel: whole blocks, a
// multiple of 128 positions, at most kMaxPrefixChunks chunks per group.  A
// CTA's start and drain are paid once per chunk, so chunks are as long as
// possible, up to kMaxChunk positions, while there are still about 1.5 chunks
// per SM, counting every group at the table's full length.  On the Yi-34B
// sharing workload (32 groups x 8 KV heads, 1 K - 8 K shared positions, 152
// SMs), chunks of 2048, 3072, 4096, 5120, 6144, 7168 and 8192 positions gave
// 129.9, 122.1, 114.2, 114.2, 111.9, 109.9 and 109.0 us per call.
// PKV_PREFIX_CHUNK (positions, 1024 .. 65536) fixes the length instead.
int32_t prefix_chunk_blocks(int32_t max_blocks, int32_t block_size, int32_t num_groups,
                            int32_t num_kv_heads, int sms) {
  constexpr int64_t kMinChunk = 1024, kMaxChunk = 8192;
  static const int64_t fixed = [] {
    const char* v = getenv("PKV_PREFIX_CHUNK");
    const long x = v != nullptr ? strtol(v, nullptr, 10) : 0;
    return x >= 1024 && x <= 65536 ? static_cast<int64_t>(x) : int64_t{0};
  }();
  int64_t chunk = fixed;
  if (chunk == 0) {
    const int64_t slots = static_cast<int64_t>(num_groups) * num_kv_heads;  // CTAs per chunk
    const int64_t want = (3 * static_cast<int64_t>(sms > 0 ? sms : 1) + 1) / 2;
    const int64_t per_group = (want + slots - 1) / slots;
    chunk = (static_cast<int64_t>(max_blocks) * block_size + per_group - 1) / per_group;
    chunk = chunk < kMinChunk ? kMinChunk : (chunk > kMaxChunk ? kMaxChunk : chunk);
  }
  auto up8 = [](int64_t x) { return static_cast<int32_t>((x + 7) / 8 * 8); };
  const int32_t a = up8((max_blocks + kMaxPrefixChunks - 1) / kMaxPrefixChunks);
  const int32_t b = up8((chunk + block_size - 1) / block_size);
  return a > b ? a : b;
}

struct SharedPlan {
  int32_t rows = 0;  // largest group x G
  size_t tables_s = 0, ctx_s = 0, rec_p = 0, rec_s = 0, tc = 0;
  size_t total = 0;
};

SharedPlan shared_plan(int32_t B, int32_t num_groups, int32_t max_group_size, int32_t max_blocks,
                       const pkv_heads& h, int sms) {
  SharedPlan s;
  const int32_t G = h.num_q_heads / h.num_kv_heads;
  s.rows = max_group_size * G;
  size_t at = 0;
  auto take = [&](size_t bytes) {
    const size_t here = at;
    at += (bytes + 255) / 256 * 256;
    return here;
  };
  s.rec_p = take(static_cast<size_t>(num_groups) * kMaxPrefixChunks * 2 * h.num_kv_heads *
                 s.rows * pkv::kRecStride * 4);
  s.tables_s = take(static_cast<size_t>(B) * max_blocks * 4);
  s.ctx_s = take(static_cast<size_t>(B) * 4);
  s.rec_s = take(static_cast<size_t>(B) * h.num_q_heads * pkv::kRecStride * 4);
  s.tc = take(pkv::tc_workspace_bytes(tc_ctas(sms)));
  s.total = at;
  return s;
}

// How a shared-prefix call runs: the chunks of the shared positions and
// where the own positions (after a group's shared blocks) are attended.
struct SharedModes {
  int32_t chunk_blocks = 0, prefix_chunks = 0;
  int32_t run_rows = 0;    // rows per TMA box of the prefix kernel: gcd(block_size, 128)
  int32_t own_cap = -1;    // a host bound of at most kInlineOwnMax own positions, else -1
  int32_t own_slots = 0;   // > 0: own positions as masked key tiles of the prefix kernel
  bool fused = false;      // the prefix kernel writes the output: the call is one launch
};

SharedModes shared_modes(int32_t max_blocks, int32_t block_size, int32_t num_groups,
                         int32_t max_group_size, int32_t max_own_tokens, const pkv_heads& h,
                         int sms) {
  SharedModes m;
  const int32_t G = h.num_q_heads / h.num_kv_heads;
  m.chunk_blocks = prefix_chunk_blocks(max_blocks, block_size, num_groups, h.num_kv_heads, sms);
  m.prefix_chunks = (max_blocks + m.chunk_blocks - 1) / m.chunk_blocks;
  m.run_rows = 128;
  while (block_size % m.run_rows != 0) m.run_rows >>= 1;
  // short own parts are attended without a second tensor-core pass
  m.own_cap = max_own_tokens >= 0 && max_own_tokens <= kInlineOwnMax ? max_own_tokens : -1;
  // Own parts of at most kOwnTileSlots slots per row block (slots: the bound
  // rounded up to whole boxes, times the members a row block can hold) ride
  // as masked key tiles of the prefix kernel; with one chunk per group that
  // kernel then writes the output itself and the merge is not launched.
  // Otherwise the merge kernel attends them on CUDA cores.
  if (m.own_cap >= 0) {
    const int64_t slots = (static_cast<int64_t>(m.own_cap) + m.run_rows - 1) / m.run_rows * m.run_rows;
    const int64_t members = std::min<int64_t>(max_group_size, kPrefixRowTile / G + 2);
    if (slots > 0 && members * slots <= kOwnTileSlots) m.own_slots = static_cast<int32_t>(slots);
  }
  m.fused = m.own_slots > 0 && m.prefix_chunks == 1;
  return m;
}

pkv_status gather_common(const void* cache, const int32_t* block_tables, int32_t max_blocks,
                         int32_t num_blocks, const int32_t* req_ids, int32_t max_reqs,
                         const int32_t* context_lens, int32_t num_seqs, int32_t max_context,
                         int64_t bs_or_S, int32_t num_kv_heads, void* out, void* stream) {
  const bool contig = block_tables == nullptr;
  if (num_seqs < 0 || max_context < 0 || num_kv_heads <= 0)
    return fail(PKV_ERR_INVALID_ARG, "negative size or no KV heads");
  if (num_seqs == 0 || max_context == 0) return PKV_OK;
  if (!cache || !context_lens || !out || (contig && !req_ids))
    return fail(PKV_ERR_INVALID_ARG, "null pointer argument");
  if (!aligned(cache, 16) || !aligned(out, 16)) return fail(PKV_ERR_INVALID_ARG, "misaligned rows");
  if (bs_or_S <= 0) return fail(PKV_ERR_INVALID_ARG, "block_size / S must be >= 1");
  if (contig) {
    if (max_reqs <= 0 || max_context > bs_or_S)
      return fail(PKV_ERR_INVALID_ARG, "max_reqs < 1 or max_context > S");
  } else if (max_blocks <= 0 || num_blocks <= 0 ||
             static_cast<int64_t>(max_blocks) * bs_or_S < max_context) {
    return fail(PKV_ERR_INVALID_ARG, "block table shorter than max_context");
  }
  const int64_t rows = static_cast<int64_t>(num_seqs) * num_kv_heads * max_context;
  if ((rows + 15) / 16 > 0x7fffffffLL) return fail(PKV_ERR_UNSUPPORTED, "gather too large");
  int* err = nullptr;
  pkv_status st = device_info(nullptr, &err, nullptr);
  if (st != PKV_OK) return st;
  pkv::GatherParams p;
  std::memset(&p, 0, sizeof p);
  p.cache = static_cast<const uint16_t*>(cache);
  p.block_tables = block_tables;
  p.req_ids = req_ids;
  p.ctx_lens = context_lens;
  p.out = static_cast<uint16_t*>(out);
  p.bs = bs_or_S;
  p.num_blocks = contig ? max_reqs : num_blocks;
  p.max_blocks = max_blocks;
  p.num_seqs = num_seqs;
  p.Hkv = num_kv_heads;
  p.max_context = max_context;
  p.checked = g_checked.load();
  p.err = err;
  const cudaError_t e = pkv::launch_gather(p, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "gather launch");
  return PKV_OK;
}

}  // namespace

extern "C" {

pkv_status pkv_kv_append(const int64_t* slot_mapping, int64_t num_tokens, const void* k,
                         const void* v, void* k_cache, void* v_cache, int64_t num_slots,
                         int64_t block_size, pkv_heads heads, void* stream) {
  return append_common(slot_mapping, num_tokens, k, v, k_cache, v_cache, num_slots, block_size,
                       heads, stream, false);
}

// A decode step: the attention call is checked first, so that a bad argument
// launches nothing; then the append (plain launch) and the attention.
pkv_status pkv_paged_decode_step(const int64_t* slot_mapping, const void* k_new,
                                 const void* v_new, const void* q, void* k_cache, void* v_cache,
                                 const int32_t* block_tables, int32_t max_blocks_per_seq,
                                 int32_t num_blocks, const int32_t* context_lens,
                                 int32_t num_seqs, int32_t max_context, int32_t block_size,
                                 float scale, pkv_heads heads, void* out, void* workspace,
                                 size_t workspace_bytes, void* stream) {
  bool tc = false;
  pkv_status st = decode_common(false, q, k_cache, v_cache, block_tables, max_blocks_per_seq,
                                num_blocks, nullptr, 0, context_lens, num_seqs, max_context,
                                block_size, scale, heads, out, workspace, workspace_bytes, stream,
                                true, &tc);
  if (st != PKV_OK || num_seqs == 0) return st;
  const int64_t num_slots = static_cast<int64_t>(num_blocks) * block_size;
  if (tc) {  // one launch: the tensor-core kernel does the append too
    st = append_common(slot_mapping, num_seqs, k_new, v_new, k_cache, v_cache, num_slots,
                       block_size, heads, stream, true, true);
    if (st != PKV_OK) return st;
    const FusedAppend fa{slot_mapping, k_new, v_new, num_slots};
    return decode_common(false, q, k_cache, v_cache, block_tables, max_blocks_per_seq,
                         num_blocks, nullptr, 0, context_lens, num_seqs, max_context, block_size,
                         scale, heads, out, workspace, workspace_bytes, stream, false, nullptr,
                         &fa);
  }
  st = append_common(slot_mapping, num_seqs, k_new, v_new, k_cache, v_cache, num_slots,
                     block_size, heads, stream, true);
  if (st != PKV_OK) return st;
  return decode_common(false, q, k_cache, v_cache, block_tables, max_blocks_per_seq, num_blocks,
                       nullptr, 0, context_lens, num_seqs, max_context, block_size, scale, heads,
                       out, workspace, workspace_bytes, stream);
}

pkv_status pkv_contig_decode_step(const int64_t* slot_mapping, const void* k_new,
                                  const void* v_new, const void* q, void* k_buf, void* v_buf,
                                  const int32_t* req_ids, int32_t max_reqs,
                                  const int32_t* context_lens, int32_t num_seqs,
                                  int32_t max_context, int64_t S, float scale, pkv_heads heads,
                                  void* out, void* workspace, size_t workspace_bytes,
                                  void* stream) {
  bool tc = false;
  pkv_status st = decode_common(true, q, k_buf, v_buf, nullptr, 0, 0, req_ids, max_reqs,
                                context_lens, num_seqs, max_context, S, scale, heads, out,
                                workspace, workspace_bytes, stream, true, &tc);
  if (st != PKV_OK || num_seqs == 0) return st;
  const int64_t num_slots = static_cast<int64_t>(max_reqs) * S;
  if (tc) {  // one launch: the tensor-core kernel does the append too
    st = append_common(slot_mapping, num_seqs, k_new, v_new, k_buf, v_buf, num_slots, S, heads,
                       stream, true, true);
    if (st != PKV_OK) return st;
    const FusedAppend fa{slot_mapping, k_new, v_new, num_slots};
    return decode_common(true, q, k_buf, v_buf, nullptr, 0, 0, req_ids, max_reqs, context_lens,
                         num_seqs, max_context, S, scale, heads, out, workspace, workspace_bytes,
                         stream, false, nullptr, &fa);
  }
  st = append_common(slot_mapping, num_seqs, k_new, v_new, k_buf, v_buf, num_slots, S, heads,
                     stream, true);
  if (st != PKV_OK) return st;
  return decode_common(true, q, k_buf, v_buf, nullptr, 0, 0, req_ids, max_reqs, context_lens,
                       num_seqs, max_context, S, scale, heads, out, workspace, workspace_bytes,
                       stream);
}

int32_t pkv_decode_num_splits(int32_t num_seqs, pkv_heads heads, int32_t max_context) {
  int sms = 0;
  if (device_info(nullptr, nullptr, &sms) != PKV_OK) return -1;
  if (check_heads(heads) != PKV_OK || num_seqs < 0 || max_context < 0) return -1;
  return plan_splits(num_seqs, heads, max_context, sms).nsplit;
}

int32_t pkv_decode_uses_tensor_cores(int32_t num_seqs, pkv_heads heads, int32_t max_context,
                                     int32_t block_size) {
  int sms = 0;
  if (device_info(nullptr, nullptr, &sms) != PKV_OK) return -1;
  if (check_heads(heads) != PKV_OK || num_seqs < 0 || max_context < 0) return -1;
  const int variant = g_variant.load();
  if (variant == 1 || (block_size > 0 && block_size % 16 != 0)) return 0;
  if (variant >= 2) return 1;
  return tc_enough_tiles(num_seqs, heads, max_context, sms) ? 1 : 0;
}

size_t pkv_decode_workspace_size(int32_t num_seqs, pkv_heads heads, int32_t max_context) {
  int sms = 0;
  if (device_info(nullptr, nullptr, &sms) != PKV_OK) return 0;
  if (check_heads(heads) != PKV_OK || num_seqs <= 0 || max_context < 0) return 0;
  return decode_workspace_need(num_seqs, heads, max_context, sms);
}

pkv_status pkv_paged_decode_attention(const void* q, const void* k_cache, const void* v_cache,
                                      const int32_t* block_tables, int32_t max_blocks_per_seq,
                                      int32_t num_blocks, const int32_t* context_lens,
                                      int32_t num_seqs, int32_t max_context, int32_t block_size,
                                      float scale, pkv_heads heads, void* out, void* workspace,
                                      size_t workspace_bytes, void* stream) {
  return decode_common(false, q, k_cache, v_cache, block_tables, max_blocks_per_seq, num_blocks,
                       nullptr, 0, context_lens, num_seqs, max_context, block_size, scale, heads,
                       out, workspace, workspace_bytes, stream);
}

pkv_status pkv_contig_decode_attention(const void* q, const void* k_buf, const void* v_buf,
                                       const int32_t* req_ids, int32_t max_reqs,
                                       const int32_t* context_lens, int32_t num_seqs,
                                       int32_t max_context, int64_t S, float scale,
                                       pkv_heads heads, void* out, void* workspace,
                                       size_t workspace_bytes, void* stream) {
  return decode_common(true, q, k_buf, v_buf, nullptr, 0, 0, req_ids, max_reqs, context_lens,
                       num_seqs, max_context, S, scale, heads, out, workspace, workspace_bytes,
                       stream);
}

int32_t pkv_shared_decode_launches(int32_t num_seqs, int32_t num_groups, int32_t max_group_size,
                                   int32_t max_blocks_per_seq, int32_t max_context,
                                   int32_t block_size, int32_t max_own_tokens, pkv_heads heads) {
  int sms = 0;
  if (device_info(nullptr, nullptr, &sms) != PKV_OK) return -1;
  if (check_heads(heads) != PKV_OK || num_seqs <= 0 || num_groups <= 0 || max_group_size <= 0 ||
      max_blocks_per_seq <= 0 || max_context < 0 || block_size <= 0 || block_size % 16 != 0)
    return -1;
  const SharedModes m = shared_modes(max_blocks_per_seq, block_size, num_groups, max_group_size,
                                     max_own_tokens, heads, sms);
  if (m.fused) return 1;          // the prefix kernel
  if (m.own_cap >= 0) return 2;   // the prefix kernel, the merge
  // the prep, the prefix kernel, the tensor-core pass (one launch per chunk of
  // sequences), the merge
  const int chunk = pkv::tc_chunk_seqs(max_context);
  return 3 + (num_seqs + chunk - 1) / chunk;
}

size_t pkv_shared_decode_workspace_size(int32_t num_seqs, int32_t num_groups,
                                        int32_t max_group_size, int32_t max_blocks_per_seq,
                                        pkv_heads heads) {
  int sms = 0;
  if (device_info(nullptr, nullptr, &sms) != PKV_OK) return 0;
  if (check_heads(heads) != PKV_OK || num_seqs <= 0 || num_groups <= 0 || max_group_size <= 0 ||
      max_blocks_per_seq <= 0)
    return 0;
  return shared_plan(num_seqs, num_groups, max_group_size, max_blocks_per_seq, heads, sms).total;
}

pkv_status pkv_paged_decode_attention_shared(
    const void* q, const void* k_cache, const void* v_cache, const int32_t* block_tables,
    int32_t max_blocks_per_seq, int32_t num_blocks, const int32_t* context_lens, int32_t num_seqs,
    int32_t max_context, int32_t block_size, const int32_t* group_start,
    const int32_t* shared_blocks, int32_t num_groups, int32_t max_group_size,
    int32_t max_own_tokens, float scale, pkv_heads heads, void* out, void* workspace,
    size_t workspace_bytes, void* stream) {
  pkv_status st = check_heads(heads);
  if (st != PKV_OK) return st;
  if (num_seqs < 0 || max_context < 0 || num_groups < 0) return fail(PKV_ERR_INVALID_ARG, "negative size");
  if (num_seqs == 0) return PKV_OK;
  if (num_seqs > 65535) return fail(PKV_ERR_UNSUPPORTED, "num_seqs > 65535");
  if (num_groups < 1 || num_groups > num_seqs || max_group_size < 1 || max_group_size > num_seqs)
    return fail(PKV_ERR_INVALID_ARG, "need 1 <= num_groups <= num_seqs and 1 <= max_group_size <= num_seqs");
  if (!q || !k_cache || !v_cache || !out || !context_lens || !block_tables || !group_start ||
      !shared_blocks)
    return fail(PKV_ERR_INVALID_ARG, "null pointer argument");
  if (!aligned(q, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) || !aligned(out, 16))
    return fail(PKV_ERR_INVALID_ARG, "bf16 tensors must be 16-byte aligned");
  if (!aligned(context_lens, 4) || !aligned(block_tables, 4) || !aligned(group_start, 4) ||
      !aligned(shared_blocks, 4))
    return fail(PKV_ERR_INVALID_ARG, "int32 arrays misaligned");
  if (!std::isfinite(scale)) return fail(PKV_ERR_INVALID_ARG, "scale is not finite");
  if (block_size <= 0 || block_size % 16 != 0)
    return fail(PKV_ERR_UNSUPPORTED, "the shared-prefix path needs block_size %% 16 == 0");
  if (max_blocks_per_seq <= 0 || num_blocks <= 0 ||
      static_cast<int64_t>(max_blocks_per_seq) * block_size < max_context)
    return fail(PKV_ERR_INVALID_ARG, "max_blocks_per_seq * block_size < max_context");
  const int64_t rows_total = static_cast<int64_t>(num_blocks) * heads.num_kv_heads * block_size;
  if (rows_total > 0x7fffffffLL) return fail(PKV_ERR_UNSUPPORTED, "cache of 2^31 rows or more");
  if (static_cast<int64_t>(max_blocks_per_seq) * block_size > 0x7fffffffLL)
    return fail(PKV_ERR_UNSUPPORTED, "block table longer than 2^31 positions");
  int dev = 0, sms = 0;
  int* err = nullptr;
  st = device_info(&dev, &err, &sms);
  if (st != PKV_OK) return st;
  const SharedPlan sp = shared_plan(num_seqs, num_groups, max_group_size, max_blocks_per_seq,
                                    heads, sms);
  if (!workspace || workspace_bytes < sp.total)
    return fail(PKV_ERR_WORKSPACE, "workspace needs %zu bytes, got %zu", sp.total,
                workspace ? workspace_bytes : size_t{0});
  if (!aligned(workspace, 256)) return fail(PKV_ERR_WORKSPACE, "workspace must be 256-byte aligned");
  unsigned char* ws = static_cast<unsigned char*>(workspace);
  pkv::CascadeParams c;
  std::memset(&c, 0, sizeof c);
  c.q = static_cast<const uint16_t*>(q);
  c.ctx = context_lens;
  c.block_tables = block_tables;
  c.group_start = group_start;
  c.shared_blocks = shared_blocks;
  c.out = static_cast<uint16_t*>(out);
  c.B = num_seqs;
  c.Hq = heads.num_q_heads;
  c.Hkv = heads.num_kv_heads;
  c.G = heads.num_q_heads / heads.num_kv_heads;
  c.max_blocks = max_blocks_per_seq;
  c.num_groups = num_groups;
  c.bs = block_size;
  c.prefix_rows = sp.rows;
  const SharedModes sm = shared_modes(max_blocks_per_seq, block_size, num_groups, max_group_size,
                                      max_own_tokens, heads, sms);
  c.prefix_chunks = sm.prefix_chunks;
  c.prefix_chunk_keys = sm.chunk_blocks * block_size;
  if (static_cast<int64_t>(num_groups) * c.prefix_chunks > 65535)
    return fail(PKV_ERR_UNSUPPORTED, "too many groups");
  c.checked = g_checked.load();
  c.err = err;
  c.k_cache = static_cast<const uint16_t*>(k_cache);
  c.v_cache = static_cast<const uint16_t*>(v_cache);
  c.qscale = scale * 1.4426950408889634f;  // log2(e)
  c.own_cap = sm.own_cap;
  c.own_in_prefix = sm.own_slots > 0;
  const int32_t own_slots = sm.own_slots;
  const int run_rows = sm.run_rows;
  const bool fused = sm.fused;
  c.tables_s = reinterpret_cast<int32_t*>(ws + sp.tables_s);
  c.ctx_s = reinterpret_cast<int32_t*>(ws + sp.ctx_s);
  c.rec_p = reinterpret_cast<float*>(ws + sp.rec_p);
  c.rec_s = reinterpret_cast<float*>(ws + sp.rec_s);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t ce = cudaSuccess;
  if (c.own_cap < 0) {  // own parts by the tensor-core decode pass: their tables
    ce = pkv::launch_cascade_prep(c, s);
    if (ce != cudaSuccess) return cuda_fail(ce, "prefix-sharing prep launch");
  }
  // The shared positions, once per group: every (member, query head) row of
  // a group against its shared blocks on the tcgen05 prefill kernel (no
  // causal mask), records out.
  {
    alignas(64) CUtensorMap tk;
    alignas(64) CUtensorMap tv;
    if (!pkv::encode_prefill_runs(&tk, k_cache, rows_total, run_rows) ||
        !pkv::encode_prefill_runs(&tv, v_cache, rows_total, run_rows))
      return fail(PKV_ERR_CUDA, "cuTensorMapEncodeTiled failed for the K/V cache");
    pkv::PrefixParams pf;
    std::memset(&pf, 0, sizeof pf);
    pf.q = c.q;
    pf.group_start = group_start;
    pf.shared_blocks = shared_blocks;
    pf.block_tables = block_tables;
    pf.rec_out = c.rec_p;
    pf.bs = block_size;
    pf.num_blocks = num_blocks;
    pf.max_blocks = max_blocks_per_seq;
    pf.num_groups = num_groups;
    pf.Hq = heads.num_q_heads;
    pf.Hkv = heads.num_kv_heads;
    pf.G = c.G;
    pf.rows = sp.rows;
    pf.chunks = c.prefix_chunks;
    pf.chunk_keys = c.prefix_chunk_keys;
    pf.run_rows = run_rows;
    pf.qscale = c.qscale;
    pf.ctx = context_lens;
    pf.own_slots = own_slots;
    pf.own_cap = c.own_cap;
    pf.out = fused ? c.out : nullptr;
    pf.checked = c.checked;
    pf.err = err;
    ce = pkv::launch_prefix(tk, tv, pf, s);
    if (ce != cudaSuccess) return cuda_fail(ce, "prefix-sharing prefix launch");
  }
  if (c.own_cap < 0) {  // every sequence's own positions: tensor-core decode, records
    pkv::TcParams t;
    std::memset(&t, 0, sizeof t);
    t.q = c.q;
    t.out = c.out;  // unused: record mode
    t.rec_out = c.rec_s;
    t.ctx_lens = c.ctx_s;
    t.block_tables = c.tables_s;
    t.bs = block_size;
    t.num_blocks = num_blocks;
    t.max_blocks = max_blocks_per_seq;
    t.num_seqs = num_seqs;
    t.Hkv = heads.num_kv_heads;
    t.G = c.G;
    t.Hq = t.Hkv * t.G;
    t.max_context = max_context;
    t.qscale = c.qscale;
    t.checked = c.checked;
    t.err = err;
    const pkv::TcStatus ts = pkv::launch_decode_tc(t, false, k_cache, v_cache, rows_total, 1,
                                                   tc_ctas(sms), ws + sp.tc, s, &ce);
    if (ts == pkv::TcStatus::kEncodeFailed)
      return fail(PKV_ERR_CUDA, "cuTensorMapEncodeTiled failed for the K/V cache");
    if (ts != pkv::TcStatus::kOk) return cuda_fail(ce, "prefix-sharing decode launch");
  }
  if (fused) return PKV_OK;  // the prefix kernel wrote the output
  ce = pkv::launch_cascade_merge(c, s);
  if (ce != cudaSuccess) return cuda_fail(ce, "prefix-sharing merge launch");
  return PKV_OK;
}

}  // extern "C"

namespace {

// Causal prefill over rows addressed as block (or request) x block_size; a
// TMA box covers run_rows rows of one block.
pkv_status prefill_common(const void* q, const int32_t* cu_seqlens_q, int32_t num_tokens,
                          const void* k_cache, const void* v_cache, const int32_t* block_tables,
                          int32_t max_blocks_per_seq, int32_t num_blocks,
                          const int32_t* context_lens, int32_t num_seqs, int32_t max_q_tokens,
                          int32_t block_size, int run_rows, float scale, pkv_heads heads,
                          void* out, void* stream) {
  pkv_status st = check_heads(heads);
  if (st != PKV_OK) return st;
  if (num_seqs < 0 || num_tokens < 0 || max_q_tokens < 0) return fail(PKV_ERR_INVALID_ARG, "negative size");
  if (num_seqs == 0 || num_tokens == 0 || max_q_tokens == 0) return PKV_OK;
  if (num_seqs > 65535) return fail(PKV_ERR_UNSUPPORTED, "num_seqs > 65535");
  if (!q || !cu_seqlens_q || !k_cache || !v_cache || !block_tables || !context_lens || !out)
    return fail(PKV_ERR_INVALID_ARG, "null pointer argument");
  if (!aligned(q, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) || !aligned(out, 16))
    return fail(PKV_ERR_INVALID_ARG, "bf16 tensors must be 16-byte aligned");
  if (!aligned(cu_seqlens_q, 4) || !aligned(block_tables, 4) || !aligned(context_lens, 4))
    return fail(PKV_ERR_INVALID_ARG, "int32 arrays misaligned");
  if (!std::isfinite(scale)) return fail(PKV_ERR_INVALID_ARG, "scale is not finite");
  if (block_size <= 0 || block_size % 16 != 0)
    return fail(PKV_ERR_UNSUPPORTED, "prefill needs block_size %% 16 == 0");
  if (max_blocks_per_seq <= 0 || num_blocks <= 0)
    return fail(PKV_ERR_INVALID_ARG, "empty block table or pool");
  const int64_t rows_total = static_cast<int64_t>(num_blocks) * heads.num_kv_heads * block_size;
  if (rows_total > 0x7fffffffLL) return fail(PKV_ERR_UNSUPPORTED, "cache of 2^31 rows or more");
  if (static_cast<int64_t>(max_blocks_per_seq) * block_size > 0x7fffffffLL)
    return fail(PKV_ERR_UNSUPPORTED, "block table longer than 2^31 positions");
  const int32_t G = heads.num_q_heads / heads.num_kv_heads;
  if ((static_cast<int64_t>(max_q_tokens) * G + 255) / 256 > 0x7fffffffLL)
    return fail(PKV_ERR_UNSUPPORTED, "chunk too long");
  int dev = 0;
  int* err = nullptr;
  st = device_info(&dev, &err, nullptr);
  if (st != PKV_OK) return st;
  alignas(64) CUtensorMap tk;
  alignas(64) CUtensorMap tv;
  if (!pkv::encode_prefill_runs(&tk, k_cache, rows_total, run_rows) ||
      !pkv::encode_prefill_runs(&tv, v_cache, rows_total, run_rows))
    return fail(PKV_ERR_CUDA, "cuTensorMapEncodeTiled failed for the K/V cache");
  pkv::PrefillParams p;
  std::memset(&p, 0, sizeof p);
  p.q = static_cast<const uint16_t*>(q);
  p.out = static_cast<uint16_t*>(out);
  p.cu_q = cu_seqlens_q;
  p.ctx_lens = context_lens;
  p.block_tables = block_tables;
  p.bs = block_size;
  p.num_blocks = num_blocks;
  p.max_blocks = max_blocks_per_seq;
  p.num_seqs = num_seqs;
  p.Hq = heads.num_q_heads;
  p.Hkv = heads.num_kv_heads;
  p.G = G;
  p.max_q = max_q_tokens;
  p.run_rows = run_rows;
  p.qscale = scale * 1.4426950408889634f;  // log2(e)
  p.checked = g_checked.load();
  p.err = err;
  // Q tiles by TMA (boxes of whole tokens), and the output by tensor stores
  // when G divides 32 (else plain stores)
  alignas(64) CUtensorMap tq;
  alignas(64) CUtensorMap to;
  std::memset(&tq, 0, sizeof tq);
  std::memset(&to, 0, sizeof to);
  p.tile_rows = (128 / G) * G;  // a row tile holds whole tokens
  if (!pkv::encode_prefill_rows(&tq, q, num_tokens, heads.num_q_heads, G, p.tile_rows))
    return fail(PKV_ERR_CUDA, "cuTensorMapEncodeTiled failed for q");
  p.out_tma = pkv::encode_prefill_rows(&to, out, num_tokens, heads.num_q_heads, G, 32) ? 1 : 0;
  p.out_v8 = aligned(out, 32) ? 1 : 0;
  const cudaError_t e =
      pkv::launch_prefill(tk, tv, tq, to, p, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "prefill launch");
  return PKV_OK;
}

}  // namespace

extern "C" {

pkv_status pkv_paged_prefill_attention(const void* q, const int32_t* cu_seqlens_q,
                                       int32_t num_tokens, const void* k_cache,
                                       const void* v_cache, const int32_t* block_tables,
                                       int32_t max_blocks_per_seq, int32_t num_blocks,
                                       const int32_t* context_lens, int32_t num_seqs,
                                       int32_t max_q_tokens, int32_t block_size, float scale,
                                       pkv_heads heads, void* out, void* stream) {
  int run_rows = 128;  // gcd(block_size, 128): a run of rows inside one block
  while (block_size > 0 && block_size % run_rows != 0) run_rows >>= 1;
  return prefill_common(q, cu_seqlens_q, num_tokens, k_cache, v_cache, block_tables,
                        max_blocks_per_seq, num_blocks, context_lens, num_seqs, max_q_tokens,
                        block_size, run_rows, scale, heads, out, stream);
}

pkv_status pkv_contig_prefill_attention(const void* q, const int32_t* cu_seqlens_q,
                                        int32_t num_tokens, const void* k_buf, const void* v_buf,
                                        const int32_t* req_ids, int32_t max_reqs,
                                        const int32_t* context_lens, int32_t num_seqs,
                                        int32_t max_q_tokens, int64_t S, float scale,
                                        pkv_heads heads, void* out, void* stream) {
  if (S <= 0 || S > 0x7fffffffLL) return fail(PKV_ERR_UNSUPPORTED, "S out of range");
  // The contiguous layout is the paged one with block_size S and a one-entry
  // table [reqId].  Boxes of 16 rows never read past round_up(ctx, 16) rows,
  // so buffers whose pages are mapped on demand stay within their backing.
  return prefill_common(q, cu_seqlens_q, num_tokens, k_buf, v_buf, req_ids, 1, max_reqs,
                        context_lens, num_seqs, max_q_tokens, static_cast<int32_t>(S), 16, scale,
                        heads, out, stream);
}

pkv_status pkv_debug_gather_paged(const void* cache, const int32_t* block_tables,
                                  int32_t max_blocks_per_seq, int32_t num_blocks,
                                  const int32_t* context_lens, int32_t num_seqs,
                                  int32_t max_context, int32_t block_size, int32_t num_kv_heads,
                                  void* out, void* stream) {
  return gather_common(cache, block_tables, max_blocks_per_seq, num_blocks, nullptr, 0,
                       context_lens, num_seqs, max_context, block_size, num_kv_heads, out, stream);
}

pkv_status pkv_debug_gather_contig(const void* buf, const int32_t* req_ids, int32_t max_reqs,
                                   const int32_t* context_lens, int32_t num_seqs,
                                   int32_t max_context, int64_t S, int32_t num_kv_heads,
                                   void* out, void* stream) {
  return gather_common(buf, nullptr, 0, 0, req_ids, max_reqs, context_lens, num_seqs,
                       max_context, S, num_kv_heads, out, stream);
}

}  // extern "C"

namespace {

// Launches the block copy kernel over n pairs and num_layers layers in
// slices of at most 65535 pairs (grid y) and kMaxCopyLayers layers.
pkv_status copy_blocks(const int64_t* pairs, int64_t n, void* const* sk, void* const* sv,
                       int64_t src_blocks, void* const* dk, void* const* dv, int64_t dst_blocks,
                       int32_t num_layers, int64_t block_bytes, void* stream) {
  int* err = nullptr;
  pkv_status st = device_info(nullptr, &err, nullptr);
  if (st != PKV_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  for (int64_t p0 = 0; p0 < n; p0 += 65535) {
    const int64_t np = (n - p0) < 65535 ? (n - p0) : 65535;
    for (int32_t l0 = 0; l0 < num_layers; l0 += pkv::kMaxCopyLayers) {
      pkv::CopyParams p;
      std::memset(&p, 0, sizeof p);
      p.pairs = pairs + 2 * p0;
      p.num_layers = (num_layers - l0) < pkv::kMaxCopyLayers ? (num_layers - l0) : pkv::kMaxCopyLayers;
      for (int32_t l = 0; l < p.num_layers; ++l) {
        p.k[l] = sk[l0 + l];
        p.v[l] = sv[l0 + l];
        p.dk[l] = dk[l0 + l];
        p.dv[l] = dv[l0 + l];
      }
      p.num_blocks = src_blocks;
      p.dst_num_blocks = dst_blocks;
      p.block_bytes = block_bytes;
      p.checked = g_checked.load();
      p.err = err;
      const cudaError_t e = pkv::launch_block_copy(p, np, s);
      if (e != cudaSuccess) return cuda_fail(e, "block copy launch");
    }
  }
  return PKV_OK;
}

// The address the kernels on `dev` use for p: p itself for device memory of
// `dev` or managed memory, the device alias of page-locked host memory;
// null for pageable host memory, another device's memory or an unknown
// pointer.
void* device_view(void* p, int dev) {
  if (p == nullptr) return nullptr;
  cudaPointerAttributes a;
  if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
    (void)cudaGetLastError();
    return nullptr;
  }
  switch (a.type) {
    case cudaMemoryTypeDevice:
      return a.device == dev ? a.devicePointer : nullptr;
    case cudaMemoryTypeManaged:
    case cudaMemoryTypeHost:
      return a.devicePointer;
    default:
      return nullptr;
  }
}

}  // namespace

extern "C" {

pkv_status pkv_block_copy(const int64_t* src_dst_pairs, int64_t n, void* const* k_caches,
                          void* const* v_caches, int32_t num_layers, int64_t num_blocks,
                          int64_t block_bytes, void* stream) {
  if (n < 0 || num_layers < 0) return fail(PKV_ERR_INVALID_ARG, "negative size");
  if (n == 0 || num_layers == 0) return PKV_OK;
  if (!src_dst_pairs || !aligned(src_dst_pairs, 8))
    return fail(PKV_ERR_INVALID_ARG, "src_dst_pairs null or misaligned");
  if (!k_caches || !v_caches) return fail(PKV_ERR_INVALID_ARG, "null cache pointer array");
  if (block_bytes <= 0 || block_bytes % 16 != 0)
    return fail(PKV_ERR_INVALID_ARG, "block_bytes must be a positive multiple of 16");
  if (num_blocks <= 0) return fail(PKV_ERR_INVALID_ARG, "num_blocks must be >= 1");
  for (int32_t l = 0; l < num_layers; ++l) {
    if (!k_caches[l] || !v_caches[l] || !aligned(k_caches[l], 16) || !aligned(v_caches[l], 16))
      return fail(PKV_ERR_INVALID_ARG, "cache pointer of layer %d null or misaligned", l);
  }
  return copy_blocks(src_dst_pairs, n, k_caches, v_caches, num_blocks, k_caches, v_caches,
                     num_blocks, num_layers, block_bytes, stream);
}

pkv_status pkv_block_swap(const int64_t* pairs, int64_t n, void* const* src_k,
                          void* const* src_v, int64_t src_num_blocks, void* const* dst_k,
                          void* const* dst_v, int64_t dst_num_blocks, int32_t num_layers,
                          int64_t block_bytes, void* stream) {
  if (n < 0 || num_layers < 0) return fail(PKV_ERR_INVALID_ARG, "negative size");
  if (n == 0 || num_layers == 0) return PKV_OK;
  if (!src_k || !src_v || !dst_k || !dst_v)
    return fail(PKV_ERR_INVALID_ARG, "null pool pointer array");
  if (block_bytes <= 0 || block_bytes % 16 != 0)
    return fail(PKV_ERR_INVALID_ARG, "block_bytes must be a positive multiple of 16");
  if (src_num_blocks <= 0 || dst_num_blocks <= 0)
    return fail(PKV_ERR_INVALID_ARG, "pool sizes must be >= 1");
  if (num_layers > 4096) return fail(PKV_ERR_INVALID_ARG, "more than 4096 layers");
  int dev = 0;
  pkv_status st = device_info(&dev, nullptr, nullptr);
  if (st != PKV_OK) return st;
  const int64_t* pv =
      static_cast<const int64_t*>(device_view(const_cast<int64_t*>(pairs), dev));
  if (pv == nullptr || !aligned(pv, 8))
    return fail(PKV_ERR_INVALID_ARG,
                "pairs must be device, managed or page-locked host memory, 8-byte aligned");
  std::vector<void*> view(4 * static_cast<size_t>(num_layers));
  void* const* in[4] = {src_k, src_v, dst_k, dst_v};
  static const char* const kName[4] = {"src_k", "src_v", "dst_k", "dst_v"};
  for (int a = 0; a < 4; ++a)
    for (int32_t l = 0; l < num_layers; ++l) {
      void* d = device_view(in[a][l], dev);
      if (d == nullptr || !aligned(d, 16))
        return fail(PKV_ERR_INVALID_ARG,
                    "%s[%d] must be device, managed or page-locked host memory, 16-byte aligned",
                    kName[a], l);
      view[a * num_layers + l] = d;
    }
  return copy_blocks(pv, n, view.data(), view.data() + num_layers, src_num_blocks,
                     view.data() + 2 * num_layers, view.data() + 3 * num_layers, dst_num_blocks,
                     num_layers, block_bytes, stream);
}

void pkv_set_checked(int enable) { g_checked.store(enable ? 1 : 0); }
void pkv_debug_stall_next_decode(void) { g_stall_test.store(1); }
void pkv_debug_drop_next_piece_record(void) { g_drop_record_test.store(1); }
void pkv_set_decode_variant(int variant) { g_variant.store(variant >= 0 && variant <= 3 ? variant : 0); }
int pkv_get_decode_variant(void) { return g_variant.load(); }
int pkv_get_checked(void) { return g_checked.load(); }
void pkv_set_split_tiles(int32_t tiles) {
  if (tiles > 0) tiles = (tiles + pkv::kDecodeWarps - 1) / pkv::kDecodeWarps * pkv::kDecodeWarps;
  g_split_tiles.store(tiles > 0 ? tiles : 0);
}

pkv_status pkv_get_device_error(int* code_out) {
  if (!code_out) return fail(PKV_ERR_INVALID_ARG, "code_out is null");
  int* err = nullptr;
  pkv_status st = device_info(nullptr, &err, nullptr);
  if (st != PKV_OK) return st;
  cudaError_t e = cudaDeviceSynchronize();
  if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceSynchronize");
  int code = 0;
  e = cudaMemcpy(&code, err, sizeof code, cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_fail(e, "read error word");
  const int zero = 0;
  e = cudaMemcpy(err, &zero, sizeof zero, cudaMemcpyHostToDevice);
  if (e != cudaSuccess) return cuda_fail(e, "clear error word");
  *code_out = code;
  return code == 0 ? PKV_OK : PKV_ERR_DEVICE_BOUNDS;
}

const char* pkv_status_string(pkv_status s) {
  switch (s) {
    case PKV_OK: return "ok";
    case PKV_ERR_INVALID_ARG: return "invalid argument";
    case PKV_ERR_UNSUPPORTED: return "unsupported configuration";
    case PKV_ERR_WORKSPACE: return "workspace missing or too small";
    case PKV_ERR_CUDA: return "CUDA runtime error";
    case PKV_ERR_DEVICE_BOUNDS: return "device-side bounds error recorded";
    case PKV_ERR_OUT_OF_BLOCKS: return "not enough free blocks";
  }
  return "unknown status";
}

const char* pkv_last_error(void) { return g_last_error; }

}  // extern "C"

namespace pkv {

// Lets other translation units of the library report a failure through
// pkv_last_error().
void set_last_error_message(const char* msg) {
  snprintf(g_last_error, sizeof g_last_error, "%s", msg);
}

}  // namespace pkv
