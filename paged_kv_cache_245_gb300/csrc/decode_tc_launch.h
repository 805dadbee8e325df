// decode_tc_launch.h -- host interface of the tensor-core / stream-K decode
// path (decode_tc.cu).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace pkv {

constexpr int kTcMaxSeqs = 512;  // sequences per launch (larger batches run in chunks)
constexpr int kRecStride = 132;  // floats per head record: o[128], m, l, pad
constexpr int kTcRecHeads = 16;  // head slots per piece record (up to two n-tiles)

struct TcParams {
  const uint16_t* q;        // [B][Hq][128]
  uint16_t* out;            // [B][Hq][128]
  const int32_t* ctx_lens;  // [B]
  const int32_t* block_tables;  // paged [B][max_blocks]
  const int32_t* req_ids;       // contig [B]
  uint64_t* rec;            // piece records [gridDim.x][kTcRecHeads][kRecStride] tagged words
  uint32_t tag;             // this launch's record tag (never 0)
  float* rec_out;           // null: bf16 out; else [B][Hq][kRecStride] (o, m, l) records
  int32_t seg_cost;         // schedule weight of one segment, in tiles (alpha below)
  int64_t bs;               // paged block size (multiple of 16); contig S
  int64_t num_blocks;       // paged pool size (checked mode)
  int32_t max_blocks, max_reqs;
  int32_t num_seqs, Hq, Hkv, G, max_context;
  float qscale;             // scale * log2(e)
  int32_t checked;
  int32_t stall_test;       // test hook: CTA 0's warp 0 expects 16 bytes that never come
  int32_t drop_record_test; // test hook: CTA 1 writes no piece record
  // The decode step's append, fused (slot_mapping non-null): sequence i's
  // new K/V rows k_new / v_new [B][Hkv][128] go to slot slot_mapping[i]
  // (negative: none) of the caches, and its attention reads them for
  // position ctx_i - 1 from the inputs rather than from the cache -- the same
  // bytes, so the same result as the append followed by the attention, as
  // long as the slot is that position's (checked mode verifies it).
  const int64_t* slot_mapping;
  const uint16_t* k_new;
  const uint16_t* v_new;
  uint16_t* k_cache;        // the caches (written: the new rows only)
  uint16_t* v_cache;
  int64_t num_slots;        // checked mode: slots in [0, num_slots)
  int* err;
};


enum class TcStatus { kOk, kEncodeFailed, kCudaError };

// The helpers below divide in 32 bits whenever every operand fits (the
// same quotients as in 64 bits; a 64-bit division costs several times more).
__host__ __device__ inline bool tc_small(int64_t V, int64_t P) {
  return V < (int64_t{1} << 22) && P < (int64_t{1} << 10);  // (V + 1) * P < 2^32
}

// Even partition of [0, V) over P CTAs: CTA c owns [floor(c*V/P), floor((c+1)*V/P)).
__host__ __device__ inline int64_t tc_range_lo(int64_t c, int64_t V, int64_t P) {
  if (tc_small(V, P))
    return static_cast<uint32_t>(c * V) / static_cast<uint32_t>(P);
  return c * V / P;
}

// The CTA whose range holds position u (the largest c with range_lo(c) <= u).
__host__ __device__ inline int64_t tc_owner(int64_t u, int64_t V, int64_t P) {
  if (tc_small(V, P))
    return static_cast<int64_t>(static_cast<uint32_t>((u + 1) * P + V - 1) /
                                static_cast<uint32_t>(V)) - 1;
  return ((u + 1) * P + V - 1) / V - 1;
}

// Cost-weighted schedule.  A CTA's time grows with its tiles and, about as
// much as alpha more tiles would, with each (sequence, KV head) segment it
// walks (the per-segment merge, Q load and table lookups).  So the partition
// is even over "virtual units": pair (i, h) spans n_i + alpha units, alpha
// units of padding followed by its n_i tiles, pairs in order.  Sequence i's
// pairs start at unit Hkv * (prefix[i] + alpha * i) (prefix[i] = tiles of
// sequences before i; an empty sequence is padding only).  Tile j of pair
// (i, h) is unit tc_vseq(i) + h * (n_i + alpha) + alpha + j.  A CTA's units
// hold a contiguous run of tiles; a range that falls inside padding holds
// none, and a cut inside padding leaves the next pair whole.
__host__ __device__ inline int64_t tc_vseq(const int32_t* prefix, int i, int Hkv, int alpha) {
  return static_cast<int64_t>(Hkv) * (static_cast<int64_t>(prefix[i]) + static_cast<int64_t>(alpha) * i);
}

// First tile whose unit is >= u (u in [0, V]; u == V gives T).
__host__ __device__ inline int64_t tc_unit_to_tile(int64_t u, const int32_t* prefix, int B, int Hkv,
                                                   int alpha) {
  if (u >= tc_vseq(prefix, B, Hkv, alpha)) return static_cast<int64_t>(Hkv) * prefix[B];
  int a = 0, b = B - 1;  // largest i with tc_vseq(i) <= u
  while (a < b) {
    const int mid = (a + b + 1) >> 1;
    if (tc_vseq(prefix, mid, Hkv, alpha) <= u) a = mid; else b = mid - 1;
  }
  const int64_t n = prefix[a + 1] - prefix[a];
  if (n + alpha <= 0) return static_cast<int64_t>(Hkv) * prefix[a];  // (not reached: see above)
  const int64_t r = u - tc_vseq(prefix, a, Hkv, alpha);  // < Hkv * (n + alpha)
  int64_t h, o;
  if (r < (int64_t{1} << 31)) {
    const uint32_t q = static_cast<uint32_t>(r) / static_cast<uint32_t>(n + alpha);
    h = q;
    o = r - static_cast<int64_t>(q) * (n + alpha) - alpha;
  } else {
    h = r / (n + alpha);
    o = r % (n + alpha) - alpha;
  }
  return static_cast<int64_t>(Hkv) * prefix[a] + h * n + (o > 0 ? o : 0);
}

// A run of tiles of one pair inside a CTA's range.
struct TcSeg {
  int64_t x0, x1;        // tiles [x0, x1) of the flattened list
  int64_t pstart, pend;  // the whole pair's tiles
  int seq, kvh;
};

// Segment starting at tile x (x < hi <= T) of sequence a (the one whose
// tiles hold x).  prefix[i] = tiles of sequences before i; pair (i, h) holds
// tiles [Hkv*prefix[i] + h*n_i, + n_i).
__host__ __device__ inline TcSeg tc_seg_at(int64_t x, int64_t hi, int a, const int32_t* prefix,
                                           int Hkv) {
  const int64_t base = static_cast<int64_t>(Hkv) * prefix[a];
  const int n = prefix[a + 1] - prefix[a];  // > 0 because x < Hkv*prefix[a+1]
  TcSeg s;
  s.seq = a;
  const int64_t dx = x - base;  // < Hkv * n
  s.kvh = dx < (int64_t{1} << 31) ? static_cast<int>(static_cast<uint32_t>(dx) / static_cast<uint32_t>(n))
                                  : static_cast<int>(dx / n);
  s.pstart = base + static_cast<int64_t>(s.kvh) * n;
  s.pend = s.pstart + n;
  s.x0 = x;
  s.x1 = s.pend < hi ? s.pend : hi;
  return s;
}

// Segment starting at tile x (x < hi <= T): finds x's sequence first (the
// last sequence whose tiles start at or before x).
__host__ __device__ inline TcSeg tc_find_seg(int64_t x, int64_t hi, const int32_t* prefix,
                                             int B, int Hkv) {
  int a = 0, b = B - 1;
  while (a < b) {
    const int mid = (a + b + 1) >> 1;
    if (static_cast<int64_t>(Hkv) * prefix[mid] <= x) a = mid; else b = mid - 1;
  }
  return tc_seg_at(x, hi, a, prefix, Hkv);
}

// The CTAs cf .. cl whose ranges hold tiles of the pair that segment `seg`
// belongs to (cf holds the pair's first tile, cl its last).  A CTA strictly
// between them with a non-empty range holds tiles of the pair only.
__host__ __device__ inline void tc_pair_ctas(const TcSeg& seg, const int32_t* prefix, int Hkv,
                                             int alpha, int64_t V, int64_t P, int* cf, int* cl) {
  const int64_t n = seg.pend - seg.pstart;
  const int64_t u0 = tc_vseq(prefix, seg.seq, Hkv, alpha) + seg.kvh * (n + alpha) + alpha;
  *cf = static_cast<int>(tc_owner(u0, V, P));
  *cl = static_cast<int>(tc_owner(u0 + n - 1, V, P));
}

// A TMA tensor map over a K or V cache viewed as [rows][128] bf16: boxes of
// 16 rows x 64 columns, 128-byte swizzle.  False if the driver refuses it.
bool encode_rows(CUtensorMap* map, const void* base, int64_t rows);

// Workspace bytes for the per-CTA partial records.
size_t tc_workspace_bytes(int num_ctas);

// Sequences per launch (a larger batch runs as consecutive launches).
int tc_chunk_seqs(int max_context);

// cfg 0: 8 warps x 3 stages per CTA; cfg 1: 12 warps x 2 stages; cfg 2:
// 10 warps x 2 stages with one merge pass for groups of 5..8 query heads
// (else as cfg 1).
TcStatus launch_decode_tc(const TcParams& p, bool contig, const void* k, const void* v,
                          int64_t rows_total, int cfg, int num_ctas, void* workspace,
                          cudaStream_t stream, cudaError_t* cuda_err);

}  // namespace pkv
