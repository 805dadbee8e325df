// decode_attention.cuh -- single-query decode attention over a paged or a
// contiguous KV cache, for sm_103a.
//
// What it computes ("Running Out of Cache": block tables map a sequence's
// positions to physical blocks; "Leveraging Low-Level CUDA APIs for
// vAttention's Dynamic Memory", section 5.2.3: request sub-tensor at
// reqId x S): for sequence i and query head h with KV head h / G,
//     out[i][h] = sum_j softmax_j(scale * q . K_j) V_j,   j < ctx_i,
// with K_j, V_j the rows at logical position j.
//
// Work decomposition: one CTA per (split of the context, KV head, sequence).
// The CTA's four warps take the split's 16-token tiles round-robin; each
// warp streams its tiles through its own ring of shared-memory stages filled
// by 1-D bulk copies (the TMA engine) that complete on per-stage mbarriers,
// so no warp ever waits on another inside the loop.  All G query heads of a
// KV head are served from one read of each K/V tile.  Each warp keeps an
// fp32 online softmax (running max m, running sum l, unnormalised output);
// the warps are merged through shared memory at the end and the CTA writes
// either the bf16 output (one split) or its (o, m, l) partial for the
// split-combine kernel.
//
// Lane roles inside a warp: lane = 16*half + j.  For q.K, lane j owns
// head_dim elements [8j, 8j+8) and, in round r, token 2*(r ^ (j>>1)) + half
// of the tile; the XOR order lets the 16-lane reduction of the 8 partial
// dot products run as a transpose-reduce with no selects (8 shuffles per
// head per tile), ending with lane j holding the score of token
// 2*(j>>1) + half.  For p.V, lane j owns output elements [8j, 8j+8) of the
// tokens of parity `half`; probabilities are broadcast through shared memory.
#pragma once

#include <math.h>

#include "pkv_device.cuh"

namespace pkv {

struct DecodeParams {
  const uint16_t* q;             // [B][Hq][128] bf16
  const uint16_t* k;             // paged [NB][Hkv][bs][128]; contig [R][Hkv][S][128]
  const uint16_t* v;
  uint16_t* out;                 // [B][Hq][128] bf16
  float* part_o;                 // [B][Hq][nsplit][128]     (nsplit > 1)
  float* part_ml;                // [B][Hq][nsplit][2] (m, l) (nsplit > 1)
  const int32_t* ctx_lens;       // [B]
  const int32_t* block_tables;   // paged: [B][max_blocks]
  const int32_t* req_ids;        // contig: [B]
  int64_t bs;                    // paged: block size; contig: S
  int64_t num_blocks;            // paged: pool size (checked mode)
  int32_t max_blocks;            // paged: table row length
  int32_t max_reqs;              // contig: buffer rows (checked mode)
  int32_t num_seqs, Hq, Hkv;
  int32_t max_context;
  int32_t chunk_tiles;           // 16-token tiles per split
  int32_t nsplit;
  float qscale;                  // scale * log2(e): scores in base-2 units
  int32_t checked;
  int* err;
};

constexpr int kDecodeWarps = 4;
constexpr int kDecodeThreads = kDecodeWarps * 32;

template <int G>
struct GroupPad {
  static constexpr int value = (G + 3) & ~3;
};

template <int G, int kStages>
struct DecodeSmemLayout {
  static constexpr int kPad = GroupPad<G>::value;
  static constexpr int kStageBytes = 2 * kTileBytes;  // K tile, then V tile
  static constexpr int kStagesBytes = kDecodeWarps * kStages * kStageBytes;
  static constexpr int kProbBytes = kDecodeWarps * kTileTokens * kPad * 4;
  static constexpr int kBarBytes = kDecodeWarps * kStages * 8;
  static constexpr int kTotal = kStagesBytes + kProbBytes + kBarBytes;
  // end-of-CTA merge reuses the stage region
  static constexpr int kMergeBytes = kDecodeWarps * G * (kHeadDim + 2) * 4;
  static_assert(kMergeBytes <= kStagesBytes, "merge buffer must fit");
};

// Context length of sequence `seq` as the kernels use it: in checked mode a
// length beyond what the grid, the block table or S can hold is reported and
// clamped; a bad request id reports and yields 0.
__device__ __forceinline__ int effective_context(const DecodeParams& p, int seq,
                                                 bool contig, bool report) {
  int ctx = p.ctx_lens[seq];
  if (p.checked) {
    int64_t cap = contig ? p.bs : static_cast<int64_t>(p.max_blocks) * p.bs;
    if (cap > p.max_context) cap = p.max_context;
    if (ctx > cap) {
      if (report) record_error(p.err, kErrContext);
      ctx = static_cast<int>(cap);
    }
    if (contig) {
      const int r = p.req_ids[seq];
      if (r < 0 || r >= p.max_reqs) {
        if (report) record_error(p.err, kErrReqId);
        ctx = 0;
      }
    }
  }
  return ctx;
}

template <int G, bool kContig, int kStages>
__global__ void __launch_bounds__(kDecodeThreads)
    decode_attention_kernel(const DecodeParams p) {
  using L = DecodeSmemLayout<G, kStages>;
  constexpr int GP = L::kPad;
  constexpr unsigned kFull = 0xffffffffu;
  extern __shared__ __align__(128) unsigned char smem[];

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int half = lane >> 4;
  const int j = lane & 15;
  const int c = j >> 1;
  const int split = blockIdx.x;
  const int kvh = blockIdx.y;
  const int seq = blockIdx.z;

  grid_dependency_trigger();
  grid_dependency_wait();
  const int ctx = effective_context(p, seq, kContig, threadIdx.x == 0 && split == 0);
  const int ntiles = ctx > 0 ? (ctx + kTileTokens - 1) / kTileTokens : 0;
  const int t_begin = split * p.chunk_tiles;
  const int t_end = min(t_begin + p.chunk_tiles, ntiles);
  if (p.nsplit > 1 && t_begin >= t_end) return;  // empty split: the combine skips it

  unsigned char* stage_base = smem + (warp * kStages) * L::kStageBytes;
  float* pbuf = reinterpret_cast<float*>(smem + L::kStagesBytes) + warp * kTileTokens * GP;
  uint64_t* bars =
      reinterpret_cast<uint64_t*>(smem + L::kStagesBytes + L::kProbBytes) + warp * kStages;

  if (lane == 0) {
    for (int s = 0; s < kStages; ++s) mbar_init(&bars[s], 1);
    fence_barrier_init();
  }
  __syncwarp();

  // Source rows.  Paged: block table row of this sequence.  Contig: the
  // request's sub-tensor for this KV head.
  const int32_t* bt_row = nullptr;
  const uint16_t* kbase = p.k;
  const uint16_t* vbase = p.v;
  if (kContig) {
    const int64_t req = ctx > 0 ? p.req_ids[seq] : 0;
    const int64_t off = cache_row(req, kvh, p.Hkv, p.bs, 0) * kHeadDim;
    kbase += off;
    vbase += off;
  } else {
    bt_row = p.block_tables + static_cast<int64_t>(seq) * p.max_blocks;
  }

  // Query rows of the group, pre-scaled so that scores are in log2 units.
  float qf[G][8];
#pragma unroll
  for (int g = 0; g < G; ++g) {
    const uint4 w = ld_global_nc_v4(p.q + (static_cast<int64_t>(seq) * p.Hq + kvh * G + g) *
                                              kHeadDim + j * 8);
    const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      qf[g][2 * e] = bf16_lo(ws[e]) * p.qscale;
      qf[g][2 * e + 1] = bf16_hi(ws[e]) * p.qscale;
    }
  }

  // This warp's tiles: t_begin + warp + k * kDecodeWarps.
  const int first = t_begin + warp;
  const int n_my = (t_end > first) ? (t_end - first + kDecodeWarps - 1) / kDecodeWarps : 0;
  const uint64_t policy = l2_policy_evict_first();

  // Block-table entry for row `lane` of local tile k (paged only).
  auto load_entry = [&](int k) -> int32_t {
    if (kContig) return 0;
    const int pos = (first + k * kDecodeWarps) * kTileTokens + lane;
    // positions are below 2^31: divide in 32 bits
    return (lane < kTileTokens && pos < ctx)
               ? __ldg(bt_row + static_cast<uint32_t>(pos) / static_cast<uint32_t>(p.bs))
               : 0;
  };

  // Fill stage k % kStages with local tile k.  Whole warp.
  auto issue = [&](int k, int32_t entry) {
    const int tile = first + k * kDecodeWarps;
    const int s = k % kStages;
    const int row0 = tile * kTileTokens;
    const int nvalid = min(kTileTokens, ctx - row0);
    unsigned char* kdst = stage_base + s * L::kStageBytes;
    unsigned char* vdst = kdst + kTileBytes;
    if (kContig) {
      if (lane == 0) {
        const uint32_t bytes = static_cast<uint32_t>(nvalid) * kRowBytes;
        mbar_arrive_expect_tx(&bars[s], 2 * bytes);
        bulk_copy_g2s(kdst, kbase + static_cast<int64_t>(row0) * kHeadDim, bytes, &bars[s], policy);
        bulk_copy_g2s(vdst, vbase + static_cast<int64_t>(row0) * kHeadDim, bytes, &bars[s], policy);
      }
    } else {
      // Lane r < nvalid holds position row0 + r; a run of rows that share a
      // physical block starts where the in-block offset is 0 (or at r = 0).
      const int64_t pos = row0 + lane;
      const int64_t off = static_cast<uint32_t>(pos) % static_cast<uint32_t>(p.bs);
      const bool start = lane < nvalid && (lane == 0 || off == 0);
      int len = 0;
      if (start) {
        const int64_t rest = p.bs - off;
        len = static_cast<int>(rest < static_cast<int64_t>(nvalid - lane) ? rest : static_cast<int64_t>(nvalid - lane));
        if (p.checked && (entry < 0 || entry >= p.num_blocks)) {
          record_error(p.err, kErrBlockId);
          len = 0;  // skip the copy; rows stay stale, output is undefined
        }
      }
      const uint32_t bytes = static_cast<uint32_t>(len) * kRowBytes;
      const uint32_t total = __reduce_add_sync(kFull, 2 * bytes);
      if (lane == 0) mbar_arrive_expect_tx(&bars[s], total);
      __syncwarp();
      if (bytes != 0) {
        const int64_t row = cache_row(entry, kvh, p.Hkv, p.bs, off);
        bulk_copy_g2s(kdst + lane * kRowBytes, p.k + row * kHeadDim, bytes, &bars[s], policy);
        bulk_copy_g2s(vdst + lane * kRowBytes, p.v + row * kHeadDim, bytes, &bars[s], policy);
      }
    }
  };

  // Prologue: fill every stage we can.
  for (int k = 0; k < kStages && k < n_my; ++k) issue(k, load_entry(k));
  int32_t next_entry = (kStages < n_my) ? load_entry(kStages) : 0;

  float m[G], l[G], acc[G][8];
#pragma unroll
  for (int g = 0; g < G; ++g) {
    m[g] = -INFINITY;
    l[g] = 0.f;
#pragma unroll
    for (int e = 0; e < 8; ++e) acc[g][e] = 0.f;
  }

  int k_done = 0;
  bool timed_out = false;
  for (int k = 0; k < n_my; ++k) {
    const int s = k % kStages;
    const uint32_t parity = static_cast<uint32_t>(k / kStages) & 1u;
    const bool ok = __all_sync(kFull, mbar_wait_bounded(&bars[s], parity));
    if (!ok) {
      timed_out = true;
      k_done = k;
      break;
    }
    const unsigned char* ks = stage_base + s * L::kStageBytes;
    const unsigned char* vs = ks + kTileBytes;
    const int nvalid = min(kTileTokens, ctx - (first + k * kDecodeWarps) * kTileTokens);

    // ---- scores: 8 rounds of partial dot products, then transpose-reduce
    float sc[G];
    {
      float part[8][G];
#pragma unroll
      for (int r = 0; r < 8; ++r) {
        const int t = 2 * (r ^ c) + half;
        const uint4 w = *reinterpret_cast<const uint4*>(ks + t * kRowBytes + j * 16);
        const float kf[8] = {bf16_lo(w.x), bf16_hi(w.x), bf16_lo(w.y), bf16_hi(w.y),
                             bf16_lo(w.z), bf16_hi(w.z), bf16_lo(w.w), bf16_hi(w.w)};
#pragma unroll
        for (int g = 0; g < G; ++g) {
          float a = qf[g][0] * kf[0];
#pragma unroll
          for (int e = 1; e < 8; ++e) a = fmaf(qf[g][e], kf[e], a);
          part[r][g] = a;
        }
      }
#pragma unroll
      for (int g = 0; g < G; ++g) {
        float a0 = part[0][g] + __shfl_xor_sync(kFull, part[4][g], 8);
        float a1 = part[1][g] + __shfl_xor_sync(kFull, part[5][g], 8);
        float a2 = part[2][g] + __shfl_xor_sync(kFull, part[6][g], 8);
        float a3 = part[3][g] + __shfl_xor_sync(kFull, part[7][g], 8);
        a0 += __shfl_xor_sync(kFull, a2, 4);
        a1 += __shfl_xor_sync(kFull, a3, 4);
        a0 += __shfl_xor_sync(kFull, a1, 2);
        a0 += __shfl_xor_sync(kFull, a0, 1);
        sc[g] = a0;  // score of token 2*c + half
      }
    }

    // ---- online softmax update (m, l warp-uniform; p to shared memory)
    const int my_t = 2 * c + half;
    const bool valid = my_t < nvalid;
    float pr[GP];
#pragma unroll
    for (int g = 0; g < G; ++g) {
      const float s_val = valid ? sc[g] : -INFINITY;
      float mx = s_val;
      mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, 2));
      mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, 4));
      mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, 8));
      mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, 16));
      const float m_new = fmaxf(m[g], mx);
      if (m_new > m[g]) {
        const float alpha = fast_exp2(m[g] - m_new);
        l[g] *= alpha;
#pragma unroll
        for (int e = 0; e < 8; ++e) acc[g][e] *= alpha;
        m[g] = m_new;
      }
      pr[g] = fast_exp2(s_val - m[g]);
      l[g] += pr[g];
    }
#pragma unroll
    for (int g = G; g < GP; ++g) pr[g] = 0.f;
    if ((j & 1) == 0) {
#pragma unroll
      for (int g4 = 0; g4 < GP; g4 += 4)
        *reinterpret_cast<float4*>(pbuf + my_t * GP + g4) =
            make_float4(pr[g4], pr[g4 + 1], pr[g4 + 2], pr[g4 + 3]);
    }
    __syncwarp();

    // ---- o += p . V over the tokens of parity `half`
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int t = 2 * u + half;
      if (nvalid == kTileTokens || t < nvalid) {
        const uint4 w = *reinterpret_cast<const uint4*>(vs + t * kRowBytes + j * 16);
        const float vf[8] = {bf16_lo(w.x), bf16_hi(w.x), bf16_lo(w.y), bf16_hi(w.y),
                             bf16_lo(w.z), bf16_hi(w.z), bf16_lo(w.w), bf16_hi(w.w)};
        float pt[GP];
#pragma unroll
        for (int g4 = 0; g4 < GP; g4 += 4) {
          const float4 f = *reinterpret_cast<const float4*>(pbuf + t * GP + g4);
          pt[g4] = f.x;
          pt[g4 + 1] = f.y;
          pt[g4 + 2] = f.z;
          pt[g4 + 3] = f.w;
        }
#pragma unroll
        for (int g = 0; g < G; ++g)
#pragma unroll
          for (int e = 0; e < 8; ++e) acc[g][e] = fmaf(pt[g], vf[e], acc[g][e]);
      }
    }
    __syncwarp();

    // ---- refill this stage with the tile kStages ahead
    if (k + kStages < n_my) {
      fence_proxy_async_smem();
      issue(k + kStages, next_entry);
      next_entry = (k + kStages + 1 < n_my) ? load_entry(k + kStages + 1) : 0;
    }
  }

  if (timed_out) {
    // A copy never completed: report, then give the copies still in flight
    // a bounded chance to land before this CTA's shared memory goes away.
    if (lane == 0) record_error(p.err, kErrTimeout);
    for (int k = k_done; k < n_my && k < k_done + kStages; ++k)
      mbar_wait_bounded(&bars[k % kStages], static_cast<uint32_t>(k / kStages) & 1u);
#pragma unroll
    for (int g = 0; g < G; ++g) {
      m[g] = -INFINITY;
      l[g] = 0.f;
#pragma unroll
      for (int e = 0; e < 8; ++e) acc[g][e] = 0.f;
    }
  }

  // ---- warp totals: both halves hold output d in [8j, 8j+8); l counted twice
#pragma unroll
  for (int g = 0; g < G; ++g) {
#pragma unroll
    for (int e = 0; e < 8; ++e) acc[g][e] += __shfl_xor_sync(kFull, acc[g][e], 16);
    float s = l[g];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) s += __shfl_xor_sync(kFull, s, o);
    l[g] = 0.5f * s;
  }

  // ---- merge the warps through shared memory (stage region reused)
  __syncthreads();
  float* red_acc = reinterpret_cast<float*>(smem);                // [W][G][128]
  float* red_ml = red_acc + kDecodeWarps * G * kHeadDim;          // [W][G][2]
  if (half == 0) {
#pragma unroll
    for (int g = 0; g < G; ++g) {
      float* dst = red_acc + (warp * G + g) * kHeadDim + j * 8;
      *reinterpret_cast<float4*>(dst) = make_float4(acc[g][0], acc[g][1], acc[g][2], acc[g][3]);
      *reinterpret_cast<float4*>(dst + 4) =
          make_float4(acc[g][4], acc[g][5], acc[g][6], acc[g][7]);
    }
  }
  if (lane == 0) {
#pragma unroll
    for (int g = 0; g < G; ++g) {
      red_ml[(warp * G + g) * 2] = m[g];
      red_ml[(warp * G + g) * 2 + 1] = l[g];
    }
  }
  __syncthreads();

  const int d = threadIdx.x;  // 0 .. 127
#pragma unroll
  for (int g = 0; g < G; ++g) {
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kDecodeWarps; ++w) M = fmaxf(M, red_ml[(w * G + g) * 2]);
    float Lsum = 0.f, O = 0.f;
    if (M != -INFINITY) {
#pragma unroll
      for (int w = 0; w < kDecodeWarps; ++w) {
        const float sc_w = fast_exp2(red_ml[(w * G + g) * 2] - M);
        Lsum = fmaf(red_ml[(w * G + g) * 2 + 1], sc_w, Lsum);
        O = fmaf(red_acc[(w * G + g) * kHeadDim + d], sc_w, O);
      }
    }
    const int64_t row = static_cast<int64_t>(seq) * p.Hq + kvh * G + g;
    const float o = Lsum > 0.f ? O / Lsum : 0.f;
    if (p.nsplit == 1) {
      p.out[row * kHeadDim + d] = f32_to_bf16_bits(o);
    } else {
      const int64_t slot = row * p.nsplit + split;
      p.part_o[slot * kHeadDim + d] = o;
      if (d == 0) {
        p.part_ml[slot * 2] = Lsum > 0.f ? M : -INFINITY;
        p.part_ml[slot * 2 + 1] = Lsum;
      }
    }
  }
}

// Merge the splits of one (sequence, query head) per warp:
//   M = max_s m_s,  w_s = l_s 2^(m_s - M),  out = sum_s w_s o_s / sum_s w_s.
template <bool kContig>
__global__ void __launch_bounds__(128) decode_combine_kernel(const DecodeParams p) {
  grid_dependency_trigger();
  grid_dependency_wait();
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int64_t idx = static_cast<int64_t>(blockIdx.x) * 4 + warp;
  if (idx >= static_cast<int64_t>(p.num_seqs) * p.Hq) return;
  const int seq = static_cast<int>(idx / p.Hq);
  const int ctx = effective_context(p, seq, kContig, false);
  const int ntiles = ctx > 0 ? (ctx + kTileTokens - 1) / kTileTokens : 0;
  const int n = min(p.nsplit, (ntiles + p.chunk_tiles - 1) / p.chunk_tiles);
  const float* ml = p.part_ml + idx * p.nsplit * 2;
  const float* po = p.part_o + idx * p.nsplit * kHeadDim;

  float M = -INFINITY;
  for (int s = lane; s < n; s += 32) M = fmaxf(M, ml[2 * s]);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));

  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  float W = 0.f;
  if (M != -INFINITY) {
    for (int s = 0; s < n; ++s) {
      const float ls = ml[2 * s + 1];
      if (ls > 0.f) {
        const float w = ls * fast_exp2(ml[2 * s] - M);
        const float4 o = *reinterpret_cast<const float4*>(po + s * kHeadDim + lane * 4);
        acc.x = fmaf(w, o.x, acc.x);
        acc.y = fmaf(w, o.y, acc.y);
        acc.z = fmaf(w, o.z, acc.z);
        acc.w = fmaf(w, o.w, acc.w);
        W += w;
      }
    }
  }
  const float inv = W > 0.f ? 1.f / W : 0.f;
  const uint32_t lo = f32_to_bf16_bits(acc.x * inv) | (uint32_t(f32_to_bf16_bits(acc.y * inv)) << 16);
  const uint32_t hi = f32_to_bf16_bits(acc.z * inv) | (uint32_t(f32_to_bf16_bits(acc.w * inv)) << 16);
  *reinterpret_cast<uint2*>(p.out + idx * kHeadDim + lane * 4) = make_uint2(lo, hi);
}

}  // namespace pkv
