// decode_tc.cuh -- decode attention over a paged (block size a multiple of 16)
// or contiguous KV cache with warp-level tensor-core math and a persistent,
// evenly balanced ("stream-K") schedule.  sm_103a.
//
// Same result as decode_attention.cuh: for sequence i, query head h, KV head
// h / G, out[i][h] = sum_j softmax_j(scale * q . K_j) V_j over j < ctx_i
// ("Running Out of Cache": block tables map positions to blocks;
// "Leveraging Low-Level CUDA APIs for vAttention's Dynamic Memory" 5.2.3:
// request sub-tensor at reqId x S).
//
// Schedule.  The work is the flattened list of 16-token tiles of every
// (sequence, KV head) pair, pair p = seq * Hkv + kvh in order.  The grid has
// one CTA per SM, and each CTA takes a contiguous run of tiles.  The runs are
// cut so that every CTA gets the same cost, counting a tile as 1 and each
// pair it touches as seg_cost more (tc_unit_to_tile), whatever the context
// lengths.  A CTA walks its run pair by pair ("segments"); its warps take
// the segment's tiles round-robin.  A segment that covers a whole pair writes
// the bf16 output directly.  The at most two partial segments of a CTA (its
// first and its last: "pieces" of a pair cut by the ranges) are merged inside
// the kernel: the CTA holding a pair's first tiles (its last segment)
// merges the others' records, which their CTAs wrote as their first
// segments, usually long before; the records validate themselves (a launch
// tag in every word), and a record not yet complete is read again, for a
// bounded time (tc_merge_pieces).
//
// Data movement.  K and V tiles (16 rows x 256 B) come in through the TMA
// engine from a 2-D tensor map over the cache's rows, as two 64-column boxes
// with 128-byte swizzling (so ldmatrix reads are free of bank conflicts),
// into a per-warp ring of shared-memory stages completed by mbarriers.  The
// group's query rows ride along with a warp's first tile of each segment.
//
// Math per tile (one warp): S^T[16 tokens x 8 heads] = K . Q^T with 8
// mma.m16n8k16 (bf16 in, fp32 accumulate); fp32 online softmax in base 2 on
// the accumulator fragment; P is packed to bf16 and transposed in registers
// (movmatrix) into the B operand of O^T[128 x 8] += V^T . P^T (8 more mma,
// V^T fetched with ldmatrix.trans).  Query heads beyond G are zero padding.
#pragma once

#include <cuda.h>
#include <math.h>

#include "decode_tc_launch.h"
#include "pkv_device.cuh"

namespace pkv {

constexpr int kTcHeads = 8;           // mma N of one n-tile: query heads of one KV head, padded
constexpr int kTcMergeHeads = 4;      // heads merged per pass through shared memory (or 8: MH)
constexpr int kTcStageBytes = 8192;   // K tile 4 KiB, V tile 4 KiB
constexpr int kBoxBytes = 2048;       // 16 rows x 128 B: half a head_dim row


template <int W, int S, int NT = 1, int MH = kTcMergeHeads>
struct TcSmem {
  static constexpr int kStagesOff = 0;
  static constexpr int kBarsOff = W * S * kTcStageBytes;
  static constexpr int kMergeOff = kBarsOff + W * S * 8;
  static constexpr int kMLOff = kMergeOff + W * MH * kRecStride * 4;
  static constexpr int kCtxOff = kMLOff + W * kTcHeads * NT * 2 * 4;
  static constexpr int kReqOff = kCtxOff + kTcMaxSeqs * 4;
  static constexpr int kPrefixOff = kReqOff + kTcMaxSeqs * 4;
  static constexpr int kRangeOff = (kPrefixOff + (kTcMaxSeqs + 1) * 4 + 7) / 8 * 8;
  static constexpr int kEnd = kRangeOff + 3 * 8;
  static constexpr int kTotal = kEnd + 1024;  // slack to align the base to 1 KiB
  static_assert(kTotal <= 232448, "shared memory per CTA exceeds 227 KiB");
};

// Context length as the kernels use it (checked mode: clamp and report).
__device__ __forceinline__ int tc_context(const TcParams& p, int i, bool contig, bool report) {
  int ctx = p.ctx_lens[i];
  if (ctx < 0) ctx = 0;
  if (p.checked) {
    int64_t cap = contig ? p.bs : static_cast<int64_t>(p.max_blocks) * p.bs;
    if (cap > p.max_context) cap = p.max_context;
    if (ctx > cap) {
      if (report) record_error(p.err, kErrContext);
      ctx = static_cast<int>(cap);
    }
    if (contig) {
      const int r = p.req_ids[i];
      if (r < 0 || r >= p.max_reqs) {
        if (report) record_error(p.err, kErrReqId);
        ctx = 0;
      }
    }
  }
  return ctx;
}

__device__ __forceinline__ bool tc_range_nonempty(int cc, int64_t V, int64_t P) {
  return tc_range_lo(cc, V, P) < tc_range_lo(cc + 1, V, P);
}

// Asynchronous global -> shared copies (cp.async, generic proxy): 16, 8 and
// 4 bytes, aligned to their size; wait_all waits for this thread's own.
__device__ __forceinline__ void cp_async_16(void* dst, const void* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 16;" ::"r"(smem_addr(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_8(void* dst, const void* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 8;" ::"r"(smem_addr(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_4(void* dst, const void* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(smem_addr(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

// One query head's result, from lane's four output elements: bf16 output,
// or an (o, m, l) record in record mode.
__device__ __forceinline__ void tc_write_out(const TcParams& p, int seq, int qh, int lane,
                                             float4 o4, float M, float L) {
  if (p.rec_out != nullptr) {
    float* r = p.rec_out + (static_cast<int64_t>(seq) * p.Hq + qh) * kRecStride;
    *reinterpret_cast<float4*>(r + lane * 4) = o4;
    if (lane == 0) {
      r[128] = M;
      r[129] = L;
    }
    return;
  }
  const uint32_t lo16 = f32_to_bf16_bits(o4.x) | (uint32_t(f32_to_bf16_bits(o4.y)) << 16);
  const uint32_t hi16 = f32_to_bf16_bits(o4.z) | (uint32_t(f32_to_bf16_bits(o4.w)) << 16);
  *reinterpret_cast<uint2*>(p.out + (static_cast<int64_t>(seq) * p.Hq + qh) * kHeadDim + lane * 4) =
      make_uint2(lo16, hi16);
}

// Piece records.  Every 64-bit word of a record holds one fp32 value in its
// low half and the launch's tag in its high half; naturally aligned 64-bit
// stores and loads are single-copy atomic, so a reader that finds the tag in
// every word of a record has read the whole record of this launch, with no
// fence on either side.  The reader zeroes the tags once it has merged, so
// every record is stale again when the launch ends: a launch replayed with
// the same tag (a CUDA graph) never meets a word of an earlier replay, and a
// word of any other origin matches a tag only by a 2^-32 accident per word.
// Words 0..127: o (lane l owns 4l .. 4l + 3); 128: m; 129: l.
__device__ __forceinline__ uint64_t tc_tagged(float x, uint32_t tag) {
  return (static_cast<uint64_t>(tag) << 32) | __float_as_uint(x);
}

__device__ __forceinline__ void tc_store_piece(uint64_t* w, uint32_t tag, int lane, float4 o4, float M,
                                               float L) {
  asm volatile("st.relaxed.gpu.global.v2.u64 [%0], {%1, %2};" ::"l"(w + lane * 4),
               "l"(tc_tagged(o4.x, tag)), "l"(tc_tagged(o4.y, tag))
               : "memory");
  asm volatile("st.relaxed.gpu.global.v2.u64 [%0], {%1, %2};" ::"l"(w + lane * 4 + 2),
               "l"(tc_tagged(o4.z, tag)), "l"(tc_tagged(o4.w, tag))
               : "memory");
  if (lane == 0)
    asm volatile("st.relaxed.gpu.global.v2.u64 [%0], {%1, %2};" ::"l"(w + 128),
                 "l"(tc_tagged(M, tag)), "l"(tc_tagged(L, tag))
                 : "memory");
}

// Lane's part of a piece record as read (o words, then m and l; the (m, l)
// words are read by every lane).
struct TcPieceWords {
  uint64_t w[6];
};

__device__ __forceinline__ void tc_issue_piece(const uint64_t* w, int lane, TcPieceWords& pw) {
  asm volatile("ld.relaxed.gpu.global.v2.u64 {%0, %1}, [%2];"
               : "=l"(pw.w[0]), "=l"(pw.w[1])
               : "l"(w + lane * 4)
               : "memory");
  asm volatile("ld.relaxed.gpu.global.v2.u64 {%0, %1}, [%2];"
               : "=l"(pw.w[2]), "=l"(pw.w[3])
               : "l"(w + lane * 4 + 2)
               : "memory");
  asm volatile("ld.relaxed.gpu.global.v2.u64 {%0, %1}, [%2];"
               : "=l"(pw.w[4]), "=l"(pw.w[5])
               : "l"(w + 128)
               : "memory");
}

// True if every word read carries `tag`; the values in o, m, l.
__device__ __forceinline__ bool tc_parse_piece(const TcPieceWords& pw, uint32_t tag, float4* o4,
                                               float* M, float* L) {
  *o4 = make_float4(__uint_as_float(static_cast<uint32_t>(pw.w[0])),
                    __uint_as_float(static_cast<uint32_t>(pw.w[1])),
                    __uint_as_float(static_cast<uint32_t>(pw.w[2])),
                    __uint_as_float(static_cast<uint32_t>(pw.w[3])));
  *M = __uint_as_float(static_cast<uint32_t>(pw.w[4]));
  *L = __uint_as_float(static_cast<uint32_t>(pw.w[5]));
  bool ok = true;
#pragma unroll
  for (int k = 0; k < 6; ++k) ok = ok && static_cast<uint32_t>(pw.w[k] >> 32) == tag;
  return ok;
}

__device__ __forceinline__ void tc_clear_piece(uint64_t* w, int lane) {
  asm volatile("st.relaxed.gpu.global.v2.u64 [%0], {%1, %1};" ::"l"(w + lane * 4), "l"(0ull)
               : "memory");
  asm volatile("st.relaxed.gpu.global.v2.u64 [%0], {%1, %1};" ::"l"(w + lane * 4 + 2), "l"(0ull)
               : "memory");
  if (lane == 0)
    asm volatile("st.relaxed.gpu.global.v2.u64 [%0], {%1, %1};" ::"l"(w + 128), "l"(0ull) : "memory");
}

// Merge the pieces of a pair cut by the CTA ranges (CTAs cf .. cl) for query
// head hh of the group and write the result; called by the CTA of the head
// piece (cf), whose own piece comes from the caller's registers.  Every piece
// is a normalised partial result (o, m, l) over its positions; softmax over
// their union is
//   M = max m_k,  w_k = l_k 2^(m_k - M),  o = sum w_k o_k / sum w_k,
// folded here in CTA order with a running maximum.  A record not yet complete
// (its CTA is still on that piece: rare, the head piece is the CTA's last
// segment and the others are earlier segments of theirs) is read again until
// it is, for at most kWaitLimitNs.  Every CTA of the grid is resident or
// finishes without waiting (waits point only to higher CTAs, and the last
// CTA's last segment is never a head piece), so the wait ends.  Returns
// false if it gave up.
__device__ __forceinline__ bool tc_merge_pieces(const TcParams& p, int seq, int qh, int hh, int cf,
                                                int cl, int64_t V, int64_t P, int lane,
                                                float4 o_own, float m_own, float l_own,
                                                const TcPieceWords& next) {
  constexpr unsigned kFull = 0xffffffffu;
  const uint32_t tag = p.tag;
  float Mr = -INFINITY, Wr = 0.f;
  float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
  auto fold = [&](float m, float l, float4 o) {
    if (!(l > 0.f)) return;
    if (m > Mr) {
      const float s = fast_exp2(Mr - m);  // 0 while Mr is -inf
      Wr *= s;
      a.x *= s; a.y *= s; a.z *= s; a.w *= s;
      Mr = m;
    }
    const float w = l * fast_exp2(m - Mr);
    a.x = fmaf(w, o.x, a.x);
    a.y = fmaf(w, o.y, a.y);
    a.z = fmaf(w, o.z, a.z);
    a.w = fmaf(w, o.w, a.w);
    Wr += w;
  };
  fold(m_own, l_own, o_own);
  bool ok = true;
  for (int cc = cf + 1; cc <= cl; ++cc) {
    if (!tc_range_nonempty(cc, V, P)) continue;
    uint64_t* rec = p.rec + (static_cast<int64_t>(cc) * kTcRecHeads + hh) * kRecStride;
    float m, l;
    float4 o;
    TcPieceWords pw;
    if (cc == cf + 1) pw = next;  // read by the caller while the CTA merged its warps
    else tc_issue_piece(rec, lane, pw);
    if (!__all_sync(kFull, tc_parse_piece(pw, tag, &o, &m, &l))) {
      const unsigned long long t0 = global_timer_ns();
      bool have;
      do {
        __nanosleep(256);
        tc_issue_piece(rec, lane, pw);
        have = __all_sync(kFull, tc_parse_piece(pw, tag, &o, &m, &l));
      } while (!have && global_timer_ns() - t0 < kWaitLimitNs);
      if (!have) ok = false;
    }
    fold(m, l, o);
    tc_clear_piece(rec, lane);
  }
  const float inv = Wr > 0.f ? 1.f / Wr : 0.f;
  tc_write_out(p, seq, qh, lane, make_float4(a.x * inv, a.y * inv, a.z * inv, a.w * inv),
               Wr > 0.f ? Mr : -INFINITY, Wr);
  return ok;
}

// NT n-tiles of 8 query heads per KV head (instantiated with NT = 1: GQA
// groups of up to 8 query heads).  kFuse: the decode step's append is done
// here too (p.slot_mapping).  MH: query heads merged per pass (4, or 8 when
// the shared memory holds every warp's 8 partials: one pass at G = 8).
template <bool kContig, int W, int S, int NT, bool kFuse, int MH>
__global__ void __launch_bounds__(W * 32, 1)
    decode_tc_kernel(const __grid_constant__ CUtensorMap tmk,
                     const __grid_constant__ CUtensorMap tmv, const TcParams p) {
  using L = TcSmem<W, S, NT, MH>;
  constexpr int H = kTcHeads * NT;  // padded query heads per KV head
  constexpr unsigned kFull = 0xffffffffu;
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem = smem_raw + ((1024 - (smem_addr(smem_raw) & 1023)) & 1023);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int tid = threadIdx.x;
  const int c = blockIdx.x;
  const int P = gridDim.x;
  const int B = p.num_seqs;
  const int G = p.G;

  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::kBarsOff) + warp * S;
  float* merge = reinterpret_cast<float*>(smem + L::kMergeOff);
  float* ml = reinterpret_cast<float*>(smem + L::kMLOff);
  int32_t* ctx_s = reinterpret_cast<int32_t*>(smem + L::kCtxOff);
  int32_t* req_s = reinterpret_cast<int32_t*>(smem + L::kReqOff);
  int32_t* prefix = reinterpret_cast<int32_t*>(smem + L::kPrefixOff);
  // this CTA's tiles [range[0], range[1]), and the sequence of its first tile
  int64_t* range = reinterpret_cast<int64_t*>(smem + L::kRangeOff);

  if (lane == 0) {
    for (int s = 0; s < S; ++s) mbar_init(&bars[s], 1);
    fence_barrier_init();
    prefetch_tensormap(&tmk);
    prefetch_tensormap(&tmv);
  }
  // Programmatic dependent launch (no-ops without the launch attribute):
  // wait for the previous kernel in the stream to finish before reading any
  // input, then let the next kernel get scheduled.
  grid_dependency_wait();
  grid_dependency_trigger();

  // ---- tile counts and their prefix over sequences (every CTA, once)
  for (int i = tid; i < B; i += W * 32) {
    const int ctx = tc_context(p, i, kContig, c == 0);
    ctx_s[i] = ctx;
    if (kContig) req_s[i] = ctx > 0 ? p.req_ids[i] : 0;
  }
  __syncthreads();
  if (warp == 0) {
    const int per = (B + 31) / 32;
    const int i0 = lane * per;
    int sum = 0;
    for (int i = i0; i < i0 + per && i < B; ++i) sum += (ctx_s[i] + 15) >> 4;
    int incl = sum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(kFull, incl, o);
      if (lane >= o) incl += v;
    }
    int run = incl - sum;
    for (int i = i0; i < i0 + per && i < B; ++i) {
      prefix[i] = run;
      run += (ctx_s[i] + 15) >> 4;
    }
    if (lane == 31) prefix[B] = incl;
    // This CTA's run of tiles [range[0], range[1]) (tc_unit_to_tile of its
    // first and past-the-end units) and the sequence holding its first tile
    // (range[2]).  In 32-bit arithmetic, when the partition has fewer than
    // 2^30 units (always, short of a million sequences of 128 K positions),
    // the warp finds each sequence with one max-reduction over the lanes'
    // own sequences instead of a serial search.
    const int total = __shfl_sync(kFull, incl, 31);
    const int64_t V64 = static_cast<int64_t>(p.Hkv) * (static_cast<int64_t>(total) +
                                                      static_cast<int64_t>(p.seg_cost) * B);
    if (V64 < (int64_t{1} << 30) && P < 1024) {
      const uint32_t V = static_cast<uint32_t>(V64), hkv = static_cast<uint32_t>(p.Hkv);
      const uint32_t alpha = static_cast<uint32_t>(p.seg_cost);
      uint32_t u[2];
#pragma unroll
      for (int k = 0; k < 2; ++k) u[k] = static_cast<uint32_t>(tc_range_lo(c + k, V, P));
      // per unit: the last sequence whose units start at or before it
      int best[2] = {-1, -1};
      run = incl - sum;
      for (int i = i0; i < i0 + per && i < B; ++i) {
        const uint32_t vi = hkv * (static_cast<uint32_t>(run) + alpha * static_cast<uint32_t>(i));
#pragma unroll
        for (int k = 0; k < 2; ++k)
          if (vi <= u[k]) best[k] = i;
        run += (ctx_s[i] + 15) >> 4;
      }
      int64_t tile[2];
#pragma unroll
      for (int k = 0; k < 2; ++k) {
        const int a = __reduce_max_sync(kFull, best[k]);
        if (u[k] >= V || a < 0) {
          tile[k] = static_cast<int64_t>(hkv) * total;
        } else {
          // the owner lane of sequence a holds its prefix; every lane reads
          // it from shared memory (written above by that lane)
          __syncwarp();
          const uint32_t pa = static_cast<uint32_t>(prefix[a]);
          const uint32_t n = static_cast<uint32_t>((ctx_s[a] + 15) >> 4);
          const uint32_t r = u[k] - hkv * (pa + alpha * static_cast<uint32_t>(a));
          const uint32_t h = r / (n + alpha);
          const int32_t o = static_cast<int32_t>(r - h * (n + alpha)) - static_cast<int32_t>(alpha);
          tile[k] = static_cast<int64_t>(hkv) * pa + h * n + (o > 0 ? o : 0);
        }
      }
      // the sequence whose tiles hold tile[0]: the last with hkv * prefix <= tile[0]
      int seq = -1;
      run = incl - sum;
      for (int i = i0; i < i0 + per && i < B; ++i) {
        if (static_cast<int64_t>(hkv) * run <= tile[0]) seq = i;
        run += (ctx_s[i] + 15) >> 4;
      }
      seq = __reduce_max_sync(kFull, seq);
      if (lane == 0) {
        range[0] = tile[0];
        range[1] = tile[1];
        range[2] = seq < 0 ? 0 : seq;
      }
    } else {
      __syncwarp();
      if (lane < 2) {
        const int64_t V = tc_vseq(prefix, B, p.Hkv, p.seg_cost);
        range[lane] = tc_unit_to_tile(tc_range_lo(c + lane, V, P), prefix, B, p.Hkv, p.seg_cost);
      }
      __syncwarp();
      if (lane == 0) {  // the sequence holding the first tile
        int a = 0, b = B - 1;
        while (a < b) {
          const int mid = (a + b + 1) >> 1;
          if (static_cast<int64_t>(p.Hkv) * prefix[mid] <= range[0]) a = mid; else b = mid - 1;
        }
        range[2] = a;
      }
    }
  }
  __syncthreads();
  // outputs of empty contexts are zeros (sequences c, c + P, ... of this CTA)
  for (int i = c; i < B; i += P) {
    if (ctx_s[i] != 0) continue;
    if (p.rec_out != nullptr) {  // empty records: o = 0, m = -inf, l = 0
      float* r = p.rec_out + static_cast<int64_t>(i) * p.Hq * kRecStride;
      for (int k = tid; k < p.Hq * kRecStride; k += W * 32) {
        const int e = k % kRecStride;
        r[k] = e == 128 ? -INFINITY : 0.f;
      }
    } else {
      uint4* o = reinterpret_cast<uint4*>(p.out + static_cast<int64_t>(i) * p.Hq * kHeadDim);
      for (int k = tid; k < p.Hq * kHeadDim / 8; k += W * 32) o[k] = make_uint4(0u, 0u, 0u, 0u);
    }
    if (kFuse) {  // the fused append of a sequence with no tile to take it
      const int64_t slot = p.slot_mapping[i];
      if (slot >= 0 && p.checked && slot >= p.num_slots) {
        if (tid == 0) record_error(p.err, kErrSlot);
      } else if (slot >= 0) {
        for (int k = tid; k < p.Hkv * 32; k += W * 32) {  // (KV head, tensor, 16-byte chunk)
          const int h = k >> 5, ch = k & 15;
          const bool is_v = (k & 16) != 0;
          *reinterpret_cast<uint4*>((is_v ? p.v_cache : p.k_cache) +
                                    cache_row(slot / p.bs, h, p.Hkv, p.bs, slot % p.bs) * kHeadDim +
                                    ch * 8) =
              ld_global_nc_v4((is_v ? p.v_new : p.k_new) +
                              (static_cast<int64_t>(i) * p.Hkv + h) * kHeadDim + ch * 8);
        }
      }
    }
  }
  const int64_t lo = range[0];
  const int64_t hi = range[1];
  const int64_t V = tc_vseq(prefix, B, p.Hkv, p.seg_cost);  // units of the whole partition
  if (lo >= hi) return;  // uniform across the CTA

  const uint64_t policy = l2_policy_evict_first();
  unsigned char* stage0 = smem + L::kStagesOff + warp * S * kTcStageBytes;
  const int g = lane >> 2;   // accumulator row group
  const int tq = lane & 3;   // accumulator column pair

  // Q^T fragments of one segment straight from global memory, n-tile t:
  // b0 = Q[8t+g][16ks + 2tq, +1], b1 = Q[8t+g][16ks + 2tq + 8, +9] (heads >= G are 0).
  auto load_q = [&](uint32_t (&qf)[NT][8][2], int seq, int kvh) {
#pragma unroll
    for (int t = 0; t < NT; ++t) {
      const int hq = 8 * t + g;
      const uint32_t* qrow = reinterpret_cast<const uint32_t*>(
          p.q + (static_cast<int64_t>(seq) * p.Hq + kvh * G + (hq < G ? hq : 0)) * kHeadDim);
#pragma unroll
      for (int ks = 0; ks < 8; ++ks) {
        qf[t][ks][0] = hq < G ? __ldg(qrow + ks * 8 + tq) : 0u;
        qf[t][ks][1] = hq < G ? __ldg(qrow + ks * 8 + 4 + tq) : 0u;
      }
    }
  };

  // ---- this warp's tile stream: segment by segment, tiles x0 + warp, + W, ...
  const int seq_lo = static_cast<int>(range[2]);
  TcSeg iseg = tc_seg_at(lo, hi, seq_lo, prefix, p.Hkv);
  int64_t ix = iseg.x0 + warp;
  bool ivalid = true;
  auto settle = [&]() {
    while (ix >= iseg.x1) {
      if (iseg.x1 >= hi) {
        ivalid = false;
        return;
      }
      iseg = tc_find_seg(iseg.x1, hi, prefix, B, p.Hkv);
      ix = iseg.x0 + warp;
    }
  };
  settle();

  // The next segment's Q fragments are fetched into qn when the stream first
  // reaches it (if qn is free), so the segment start does not wait on them.
  uint32_t qn[NT][8][2];
  int64_t qn_pair = -1;

  // block-table entry of the tile at the issue cursor (lane 0 only)
  auto load_entry = [&]() -> int32_t {
    if (kContig || lane != 0 || !ivalid) return 0;
    const int64_t pos = (ix - iseg.pstart) * 16;
    return __ldg(p.block_tables + static_cast<int64_t>(iseg.seq) * p.max_blocks + pos / p.bs);
  };

  int issued = 0;  // tiles issued by this warp so far
  auto issue = [&](int stage, int32_t entry) {
    if (ix == iseg.x0 + warp && qn_pair < 0) {  // whole warp
      load_q(qn, iseg.seq, iseg.kvh);
      qn_pair = iseg.pstart;
    }
    if (lane == 0) {
      unsigned char* st = stage0 + stage * kTcStageBytes;
      const int64_t pos = (ix - iseg.pstart) * 16;
      bool kv_ok = true;
      int64_t row;
      if (kContig) {
        row = cache_row(req_s[iseg.seq], iseg.kvh, p.Hkv, p.bs, pos);
      } else {
        if (p.checked && (entry < 0 || entry >= p.num_blocks)) {
          record_error(p.err, kErrBlockId);
          kv_ok = false;  // skip the copy: stale rows, undefined output, no fault
        }
        row = cache_row(entry, iseg.kvh, p.Hkv, p.bs, pos % p.bs);
      }
      // (test hook: on its first tile, CTA 0's warp 0 announces 16 more bytes
      // than its copies bring, so that wait runs into its time limit)
      const uint32_t extra = (p.stall_test && c == 0 && warp == 0 && issued == 0) ? 16u : 0u;
      mbar_arrive_expect_tx(&bars[stage], (kv_ok ? 4u * kBoxBytes : 0u) + extra);
      if (kv_ok) {
        const int32_t y = static_cast<int32_t>(row);
        tma_load_2d(st, &tmk, 0, y, &bars[stage], policy);
        tma_load_2d(st + kBoxBytes, &tmk, 64, y, &bars[stage], policy);
        tma_load_2d(st + 2 * kBoxBytes, &tmv, 0, y, &bars[stage], policy);
        tma_load_2d(st + 3 * kBoxBytes, &tmv, 64, y, &bars[stage], policy);
      }
    }
  };

  // Prologue: walk the stream S tiles ahead so that lane s fetches the block
  // table entry of tile s (one memory latency for all of them), then fill
  // the stages.
  int32_t pre_entry = 0;
  if (!kContig) {
    TcSeg cs = iseg;
    int64_t cx = ix;
    bool cv = ivalid;
    for (int s = 0; s < S && cv; ++s) {
      if (lane == s) {
        const int64_t pos = (cx - cs.pstart) * 16;
        pre_entry = __ldg(p.block_tables + static_cast<int64_t>(cs.seq) * p.max_blocks + pos / p.bs);
      }
      cx += W;
      while (cx >= cs.x1) {
        if (cs.x1 >= hi) {
          cv = false;
          break;
        }
        cs = tc_find_seg(cs.x1, hi, prefix, B, p.Hkv);
        cx = cs.x0 + warp;
      }
    }
  }
  for (int s = 0; s < S && ivalid; ++s) {
    issue(s, __shfl_sync(kFull, pre_entry, s));
    ++issued;
    ix += W;
    settle();
  }
  int32_t next_entry = load_entry();

  // ---- per-lane ldmatrix offsets inside a 128-byte-swizzled 16 x 128 B box
  uint32_t koff[4], voff[4];
  {
    const int rk = (lane & 7) + 8 * ((lane >> 3) & 1), hk = lane >> 4;
    const int rv = (lane & 7) + 8 * (lane >> 4), hv = (lane >> 3) & 1;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      koff[j] = rk * 128 + ((((2 * j + hk) ^ (rk & 7))) << 4);
      voff[j] = rv * 128 + ((((2 * j + hv) ^ (rv & 7))) << 4);
    }
  }

  uint32_t qb[NT][8][2];
  float acc[8][NT][4];
  float m0[NT], m1[NT], l0[NT], l1[NT];
  int consumed = 0;
  bool dead = false;

  TcSeg seg = tc_seg_at(lo, hi, seq_lo, prefix, p.Hkv);
  while (true) {
#pragma unroll
    for (int t = 0; t < NT; ++t) {
      m0[t] = m1[t] = -INFINITY;
      l0[t] = l1[t] = 0.f;
#pragma unroll
      for (int i = 0; i < 8; ++i) acc[i][t][0] = acc[i][t][1] = acc[i][t][2] = acc[i][t][3] = 0.f;
    }
    const int ctx = ctx_s[seg.seq];
    // A segment that is only part of its pair (the CTA ranges cut the pair)
    // is a "piece"; the pair's CTAs are cf .. cl.  The piece of cf (the
    // pair's first tiles, this CTA's last segment) usually finishes last:
    // its CTA merges the pair (the head piece).
    const bool whole = seg.x0 == seg.pstart && seg.x1 == seg.pend;
    int cf = c, cl = c;
    if (!whole) tc_pair_ctas(seg, prefix, p.Hkv, p.seg_cost, V, P, &cf, &cl);
    const bool head_piece = !whole && cf == c;

    // The fused append (slot_mapping): the warp that takes the pair's last
    // tile (position ctx - 1) brings the new rows into its merge slot, idle
    // until the segment's end (lanes 0-15 K, 16-31 V, 16 bytes each; then the
    // slot and, checked, the table entry of position ctx - 1), writes them to
    // the cache and over that row of the tile.
    const int64_t x_last = seg.pend - 1;
    const bool own_last = kFuse && x_last >= seg.x0 && x_last < seg.x1 &&
                          (x_last - seg.x0) % W == warp;
    unsigned char* fuse_s = reinterpret_cast<unsigned char*>(merge + warp * MH * kRecStride);
    if (own_last) {
      const int64_t pr = static_cast<int64_t>(seg.seq) * p.Hkv + seg.kvh;
      cp_async_16(fuse_s + lane * 16,
                  (lane < 16 ? p.k_new : p.v_new) + pr * kHeadDim + (lane & 15) * 8);
      if (lane == 0) cp_async_8(fuse_s + 512, p.slot_mapping + seg.seq);
      if (lane == 1 && p.checked && !kContig)
        cp_async_4(fuse_s + 520,
                   p.block_tables + static_cast<int64_t>(seg.seq) * p.max_blocks + (ctx - 1) / p.bs);
    }

    for (int64_t x = seg.x0 + warp; x < seg.x1 && !dead; x += W) {
      if (x == seg.x0 + warp) {  // this warp's first tile of the segment
        if (qn_pair == seg.pstart) {
#pragma unroll
          for (int t = 0; t < NT; ++t)
#pragma unroll
            for (int ks = 0; ks < 8; ++ks) {
              qb[t][ks][0] = qn[t][ks][0];
              qb[t][ks][1] = qn[t][ks][1];
            }
          qn_pair = -1;
        } else {
          load_q(qb, seg.seq, seg.kvh);
        }
      }
      const int stage = consumed % S;
      const uint32_t parity = static_cast<uint32_t>(consumed / S) & 1u;
      if (!__all_sync(kFull, mbar_wait_bounded(&bars[stage], parity))) {
        dead = true;
        if (lane == 0) record_error(p.err, kErrTimeout);
        break;
      }
      ++consumed;
      unsigned char* st = stage0 + stage * kTcStageBytes;
      const uint32_t kaddr = smem_addr(st);
      const uint32_t vaddr = kaddr + 2 * kBoxBytes;
      const int nvalid = min(16, ctx - static_cast<int>((x - seg.pstart) * 16));
      if (own_last && x == x_last) {  // the new rows: into the cache and over row nvalid - 1
        cp_async_wait_all();
        __syncwarp();
        const int64_t slot = *reinterpret_cast<const int64_t*>(fuse_s + 512);
        bool ok = slot >= 0;
        if (ok && p.checked) {
          int64_t want;  // the slot of position ctx - 1
          if (kContig) {
            want = static_cast<int64_t>(req_s[seg.seq]) * p.bs + ctx - 1;
          } else {
            want = static_cast<int64_t>(*reinterpret_cast<const int32_t*>(fuse_s + 520)) * p.bs +
                   (ctx - 1) % p.bs;
          }
          if (slot >= p.num_slots || slot != want) {
            if (lane == 0) record_error(p.err, kErrSlot);
            ok = false;
          }
        }
        if (ok) {
          const uint4 v = *reinterpret_cast<const uint4*>(fuse_s + lane * 16);
          const int r = nvalid - 1, ch = lane & 15;
          *reinterpret_cast<uint4*>((lane < 16 ? p.k_cache : p.v_cache) +
                                    cache_row(slot / p.bs, seg.kvh, p.Hkv, p.bs, slot % p.bs) *
                                        kHeadDim + ch * 8) = v;
          *reinterpret_cast<uint4*>(st + (lane < 16 ? 0 : 2 * kBoxBytes) + (ch >> 3) * kBoxBytes +
                                    r * 128 + (((ch & 7) ^ (r & 7)) << 4)) = v;
        }
        __syncwarp();
      }

      if (nvalid < 16) {  // rows past the context must not feed p.V (0 * NaN)
        for (int idx = lane; idx < (16 - nvalid) * 16; idx += 32) {
          const int r = nvalid + (idx >> 4);
          const int ch = idx & 15;
          *reinterpret_cast<uint4*>(st + 2 * kBoxBytes + (ch >> 3) * kBoxBytes + r * 128 +
                                    (ch & 7) * 16) = make_uint4(0u, 0u, 0u, 0u);
        }
        __syncwarp();
      }

      // ---- S^T = K . Q^T  (two accumulation chains per n-tile)
      float sa[NT][4], sb[NT][4];
#pragma unroll
      for (int t = 0; t < NT; ++t)
#pragma unroll
        for (int e = 0; e < 4; ++e) sa[t][e] = sb[t][e] = 0.f;
#pragma unroll
      for (int ks = 0; ks < 8; ++ks) {
        uint32_t a[4];
        ldmatrix_x4(a, kaddr + (ks >> 2) * kBoxBytes + koff[ks & 3]);
#pragma unroll
        for (int t = 0; t < NT; ++t) {
          if (ks & 1) mma_bf16_16816(sb[t], a, qb[t][ks][0], qb[t][ks][1]);
          else mma_bf16_16816(sa[t], a, qb[t][ks][0], qb[t][ks][1]);
        }
      }
      const bool v0 = g < nvalid, v1 = g + 8 < nvalid;
      uint32_t b0[NT], b1[NT];
#pragma unroll
      for (int t = 0; t < NT; ++t) {
        const float s0 = v0 ? (sa[t][0] + sb[t][0]) * p.qscale : -INFINITY;  // token g,   head 2tq
        const float s1 = v0 ? (sa[t][1] + sb[t][1]) * p.qscale : -INFINITY;  // token g,   head 2tq+1
        const float s2 = v1 ? (sa[t][2] + sb[t][2]) * p.qscale : -INFINITY;  // token g+8, head 2tq
        const float s3 = v1 ? (sa[t][3] + sb[t][3]) * p.qscale : -INFINITY;  // token g+8, head 2tq+1

        // ---- online softmax, per head column
        float mx0 = fmaxf(s0, s2), mx1 = fmaxf(s1, s3);
#pragma unroll
        for (int o = 4; o < 32; o <<= 1) {
          mx0 = fmaxf(mx0, __shfl_xor_sync(kFull, mx0, o));
          mx1 = fmaxf(mx1, __shfl_xor_sync(kFull, mx1, o));
        }
        const float n0 = fmaxf(m0[t], mx0), n1 = fmaxf(m1[t], mx1);
        if (n0 > m0[t]) {
          const float a = fast_exp2(m0[t] - n0);
          l0[t] *= a;
#pragma unroll
          for (int i = 0; i < 8; ++i) { acc[i][t][0] *= a; acc[i][t][2] *= a; }
          m0[t] = n0;
        }
        if (n1 > m1[t]) {
          const float a = fast_exp2(m1[t] - n1);
          l1[t] *= a;
#pragma unroll
          for (int i = 0; i < 8; ++i) { acc[i][t][1] *= a; acc[i][t][3] *= a; }
          m1[t] = n1;
        }
        const float p0 = fast_exp2(s0 - m0[t]), p2 = fast_exp2(s2 - m0[t]);
        const float p1 = fast_exp2(s1 - m1[t]), p3 = fast_exp2(s3 - m1[t]);
        l0[t] += p0 + p2;
        l1[t] += p1 + p3;
        b0[t] = movmatrix_trans(pack_bf16x2(p0, p1));  // P^T rows: tokens 0..7
        b1[t] = movmatrix_trans(pack_bf16x2(p2, p3));  // tokens 8..15
      }

      // ---- O^T += V^T . P^T  (each V^T fragment serves every n-tile)
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        uint32_t a[4];
        ldmatrix_x4_trans(a, vaddr + (i >> 2) * kBoxBytes + voff[i & 3]);
#pragma unroll
        for (int t = 0; t < NT; ++t) mma_bf16_16816(acc[i][t], a, b0[t], b1[t]);
      }
      __syncwarp();

      // ---- refill this stage with the next tile of the stream
      if (ivalid) {
        fence_proxy_async_smem();
        issue(stage, next_entry);
        ++issued;
        ix += W;
        settle();
        next_entry = load_entry();
      }
    }

    // ---- the head piece's merge warps request the next CTA's piece record
    // of their heads now, so that it arrives while the warps are merged
    constexpr int kPasses = (NT * 8 + MH - 1) / MH;  // merge passes that can hold heads
    TcPieceWords nxt[kPasses];
    if (head_piece && warp < MH && cf + 1 <= cl && tc_range_nonempty(cf + 1, V, P)) {
#pragma unroll
      for (int k = 0; k < kPasses; ++k)
        if (warp + MH * k < G)
          tc_issue_piece(p.rec + (static_cast<int64_t>(cf + 1) * kTcRecHeads + warp + MH * k) *
                                     kRecStride,
                         lane, nxt[k]);
    }

    // ---- merge the warps' partial results for this segment (4 heads a pass)
#pragma unroll
    for (int t = 0; t < NT; ++t) {
#pragma unroll
      for (int o = 4; o < 32; o <<= 1) {
        l0[t] += __shfl_xor_sync(kFull, l0[t], o);
        l1[t] += __shfl_xor_sync(kFull, l1[t], o);
      }
      if (g == 0) {
        const int h = 8 * t + 2 * tq;
        ml[(warp * H + h) * 2] = m0[t];
        ml[(warp * H + h) * 2 + 1] = l0[t];
        ml[(warp * H + h + 1) * 2] = m1[t];
        ml[(warp * H + h + 1) * 2 + 1] = l1[t];
      }
    }
#pragma unroll
    for (int pass = 0; pass < kPasses; ++pass) {
      const int h0 = pass * MH;
      if (h0 >= G) break;
      // lanes whose head pair (8t + 2tq, + 1) falls in [h0, h0 + 4) write it
#pragma unroll
      for (int t = 0; t < NT; ++t) {
        const int h = 8 * t + 2 * tq;
        if (h >= h0 && h < h0 + MH) {
          float* mb = merge + (warp * MH + (h - h0)) * kRecStride;
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            mb[16 * i + g] = acc[i][t][0];
            mb[kRecStride + 16 * i + g] = acc[i][t][1];
            mb[16 * i + g + 8] = acc[i][t][2];
            mb[kRecStride + 16 * i + g + 8] = acc[i][t][3];
          }
        }
      }
      __syncthreads();
      // warp hl merges head h0 + hl: lane j < W derives warp j's weight
      // 2^(m_j - M) / sum_k l_k 2^(m_k - M) once, then every lane sums its four
      // output elements over the W partials
      const int nh = min(MH, G - h0);
      if (warp < nh) {
        const int hh = h0 + warp;
        const float mj = lane < W ? ml[(lane * H + hh) * 2] : -INFINITY;
        const float lj = lane < W ? ml[(lane * H + hh) * 2 + 1] : 0.f;
        float M = mj;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(kFull, M, o));
        const float fj = mj == -INFINITY ? 0.f : fast_exp2(mj - M);
        float Ls = lj * fj;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) Ls += __shfl_xor_sync(kFull, Ls, o);
        const float wj = Ls > 0.f ? fj / Ls : 0.f;
        float4 o4 = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int w = 0; w < W; ++w) {
          const float ww = __shfl_sync(kFull, wj, w);
          const float4 v =
              *reinterpret_cast<const float4*>(merge + (w * MH + warp) * kRecStride + lane * 4);
          o4.x = fmaf(v.x, ww, o4.x);
          o4.y = fmaf(v.y, ww, o4.y);
          o4.z = fmaf(v.z, ww, o4.z);
          o4.w = fmaf(v.w, ww, o4.w);
        }
        const float Mr = Ls > 0.f ? M : -INFINITY;
        if (whole) {
          tc_write_out(p, seg.seq, seg.kvh * G + hh, lane, o4, Mr, Ls);
        } else if (head_piece) {
          // this piece first, then the other pieces' records in CTA order
          if (!tc_merge_pieces(p, seg.seq, seg.kvh * G + hh, hh, cf, cl, V, P, lane, o4, Mr, Ls,
                               nxt[pass]) &&
              lane == 0)
            record_error(p.err, kErrTimeout);
        } else if (!(p.drop_record_test && c == 1)) {
          tc_store_piece(p.rec + (static_cast<int64_t>(c) * kTcRecHeads + hh) * kRecStride,
                         p.tag, lane, o4, Mr, Ls);
        }
      }
      __syncthreads();
    }
    if (seg.x1 >= hi) break;
    seg = tc_find_seg(seg.x1, hi, prefix, B, p.Hkv);
  }

  if (dead) {
    // give the copies still in flight a bounded chance to land before exit
    for (int k = consumed; k < issued; ++k)
      mbar_wait_bounded(&bars[k % S], static_cast<uint32_t>(k / S) & 1u);
  }
}

}  // namespace pkv
