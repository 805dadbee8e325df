// cascade.cu -- decode attention for sequences that share prompt blocks
// ("Running Out of Cache", "Fragmentation is lost users": sequences sampled
// from one prompt share its blocks until one writes into them).  The shared
// positions are attended once for all members of a group instead of once
// per sequence: softmax over a concatenation splits into per-part partial
// results (o, m, l) merged as
//   M = max(m_a, m_b),  w_x = l_x 2^(m_x - M),  o = (w_a o_a + w_b o_b) / (w_a + w_b).
//
// The shared part of every group goes through the tcgen05 prefix kernel
// (prefix.cu): the group's (member, query head) rows against its shared
// blocks, fp32 records out (per chunk of the shared positions, two halves).  The own part after the shared blocks
// is attended here, inside the merge (a host bound of at most 256 own
// positions), or by the tensor-core decode kernel in record mode over a
// virtual batch the prep kernel builds (entry i: sequence i's own positions).
// cascade_merge_kernel merges the two records of every (sequence, head).
#include "cascade.cuh"
#include "pkv_device.cuh"

namespace pkv {

namespace {

// The group holding sequence i (group_start is ascending, group_start[0] = 0).
__device__ __forceinline__ int group_of(const int32_t* group_start, int num_groups, int i) {
  int a = 0, b = num_groups - 1;
  while (a < b) {
    const int mid = (a + b + 1) >> 1;
    if (group_start[mid] <= i) a = mid; else b = mid - 1;
  }
  return a;
}

}  // namespace

// One block per sequence: the table and length of its own positions (after
// the group's shared blocks), for the tensor-core decode pass.
__global__ void __launch_bounds__(256) cascade_prep_kernel(const CascadeParams c) {
  grid_dependency_wait();
  grid_dependency_trigger();
  const int tid = threadIdx.x;
  const int i = blockIdx.x;
  if (i >= c.B) return;
  const int g = group_of(c.group_start, c.num_groups, i);
  const int sb_in = c.shared_blocks[g];
  const int sb = sb_in < 0 ? 0 : (sb_in > c.max_blocks ? c.max_blocks : sb_in);
  const int ctx = c.ctx[i];
  const int rest = ctx - sb * c.bs;
  if (tid == 0) c.ctx_s[i] = rest > 0 ? rest : 0;
  const int n = rest > 0 ? (rest + c.bs - 1) / c.bs : 0;
  for (int j = tid; j < n; j += blockDim.x)
    c.tables_s[static_cast<int64_t>(i) * c.max_blocks + j] =
        c.block_tables[static_cast<int64_t>(i) * c.max_blocks + sb + j];
}

// The own positions [s0, s0 + n) of sequence i for query head h, on CUDA
// cores: lane j holds dimensions 4j .. 4j+3; the block-table entries are
// loaded first (lane j: entry j), then 8 positions at a time with all their
// K and V loads in flight.  Returns (o over this lane's dims, m, l) with o
// not yet normalised (o / l is the attention over these positions).
__device__ void own_attention(const CascadeParams& c, int i, int h, int sb, int n, float4& o,
                              float& m, float& l) {
  constexpr unsigned kFull = 0xffffffffu;
  constexpr int U = 8;
  const int lane = threadIdx.x & 31;
  const int kvh = h / c.G;
  const int nblk = (n + c.bs - 1) / c.bs;  // <= 32: own_cap <= 256 and bs >= 16
  const int32_t ent =
      lane < nblk ? c.block_tables[static_cast<int64_t>(i) * c.max_blocks + sb + lane] : 0;
  const uint2 qraw = __ldg(reinterpret_cast<const uint2*>(c.q + (static_cast<int64_t>(i) * c.Hq + h) *
                                                                  kHeadDim) + lane);
  const float q0 = bf16_lo(qraw.x) * c.qscale, q1 = bf16_hi(qraw.x) * c.qscale;
  const float q2 = bf16_lo(qraw.y) * c.qscale, q3 = bf16_hi(qraw.y) * c.qscale;
  o = make_float4(0.f, 0.f, 0.f, 0.f);
  m = -INFINITY;
  l = 0.f;
  for (int t0 = 0; t0 < n; t0 += U) {
    uint2 kr[U], vr[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int t = t0 + u < n ? t0 + u : n - 1;
      const int32_t blk = __shfl_sync(kFull, ent, t / c.bs);
      const int64_t row = cache_row(blk, kvh, c.Hkv, c.bs, t % c.bs);
      kr[u] = __ldg(reinterpret_cast<const uint2*>(c.k_cache + row * kHeadDim) + lane);
      vr[u] = __ldg(reinterpret_cast<const uint2*>(c.v_cache + row * kHeadDim) + lane);
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      float d = q0 * bf16_lo(kr[u].x);
      d = fmaf(q1, bf16_hi(kr[u].x), d);
      d = fmaf(q2, bf16_lo(kr[u].y), d);
      d = fmaf(q3, bf16_hi(kr[u].y), d);
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) d += __shfl_xor_sync(kFull, d, off);
      if (t0 + u >= n) continue;
      const float mn = fmaxf(m, d);
      const float a = fast_exp2(m - mn);  // 0 while m is -inf
      const float p = fast_exp2(d - mn);
      l = fmaf(l, a, p);
      o.x = fmaf(o.x, a, p * bf16_lo(vr[u].x));
      o.y = fmaf(o.y, a, p * bf16_hi(vr[u].x));
      o.z = fmaf(o.z, a, p * bf16_lo(vr[u].y));
      o.w = fmaf(o.w, a, p * bf16_hi(vr[u].y));
      m = mn;
    }
  }
}

// One warp per (sequence, query head): merge its prefix record (if the
// sequence shares anything) with its own part -- attended here, or a record
// of the tensor-core pass -- into the bf16 output.
__global__ void __launch_bounds__(128) cascade_merge_kernel(const CascadeParams c) {
  // Launched as a programmatic dependent of the prefix kernel when it attends
  // the own positions itself: those need only this call's inputs, so they
  // run before the wait, overlapping the prefix kernel's tail.
  const bool own_here = c.own_cap >= 0 && !c.own_in_prefix;
  if (!own_here) grid_dependency_wait();  // the own parts come in records of the previous kernels
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int64_t idx = static_cast<int64_t>(blockIdx.x) * 4 + warp;
  if (idx >= static_cast<int64_t>(c.B) * c.Hq) return;
  const int i = static_cast<int>(idx / c.Hq);
  const int h = static_cast<int>(idx % c.Hq);
  const int kvh = h / c.G;
  const int gi = h % c.G;
  const int g = group_of(c.group_start, c.num_groups, i);
  const int kg = i - c.group_start[g];
  const int sb_in = c.shared_blocks[g];
  const int sb = sb_in < 0 ? 0 : (sb_in > c.max_blocks ? c.max_blocks : sb_in);
  if (c.checked && lane == 0 && (sb != sb_in || c.ctx[i] < sb * c.bs))
    record_error(c.err, kErrContext);  // the group's shared blocks are not all this member's
  // The own part: attended here, or the tensor-core pass's record.
  const float* rs = c.rec_s + idx * kRecStride;
  float ms, ls;
  float4 os;
  if (c.own_in_prefix) {  // in the prefix records
    ms = -INFINITY;
    ls = 0.f;
    os = make_float4(0.f, 0.f, 0.f, 0.f);
  } else if (c.own_cap >= 0) {
    int n = c.ctx[i] - sb * c.bs;
    if (n > c.own_cap) {
      if (c.checked && (threadIdx.x & 31) == 0) record_error(c.err, kErrContext);
      n = c.own_cap;  // the bound was wrong: the later positions are left out
    }
    own_attention(c, i, h, sb, n > 0 ? n : 0, os, ms, ls);
    const float inv_own = ls > 0.f ? 1.f / ls : 0.f;
    os = make_float4(os.x * inv_own, os.y * inv_own, os.z * inv_own, os.w * inv_own);
  } else {
    ms = __ldcg(rs + 128);
    ls = __ldcg(rs + 129);
    os = ls > 0.f ? __ldcg(reinterpret_cast<const float4*>(rs) + lane)
                  : make_float4(0.f, 0.f, 0.f, 0.f);
  }
  if (own_here) grid_dependency_wait();  // the prefix records are complete
  grid_dependency_trigger();
  // Fold in the prefix records, two per chunk of the shared positions (even
  // and odd key tiles; the second only if the chunk has more than one tile,
  // always when the own tiles follow the last chunk: a group then has at
  // least one chunk and the prefix kernel writes every half).
  // A member beyond the group size bound has none: the caller broke the
  // contract, nothing is read.  Lane k loads record k's (m, l), all at once;
  // every lane loads its four o values of four records at a time; then
  //   M' = max(M, m_k),  acc' = acc 2^(M - M') + sum_k l_k 2^(m_k - M') o_k,
  //   W' = W 2^(M - M') + sum_k l_k 2^(m_k - M').
  constexpr int kMaxRec = 16;  // 2 records per chunk, at most 8 chunks
  const bool member = kg >= 0 && kg * c.G < c.prefix_rows;
  const int shared = sb * c.bs;
  const int nch = (shared + c.prefix_chunk_keys - 1) / c.prefix_chunk_keys;
  const int chunks = member ? min(c.own_in_prefix ? max(nch, 1) : nch,
                                  min(c.prefix_chunks, kMaxRec / 2))
                            : 0;
  auto used = [&](int kh) {
    return kh < 2 * chunks &&
           (c.own_in_prefix || (kh & 1) == 0 ||
            min(c.prefix_chunk_keys, shared - (kh >> 1) * c.prefix_chunk_keys) > 128);
  };
  auto rec = [&](int kh) {
    return c.rec_p + ((((static_cast<int64_t>(g) * c.prefix_chunks + (kh >> 1)) * 2 + (kh & 1)) *
                           c.Hkv + kvh) * c.prefix_rows + kg * c.G + gi) * kRecStride;
  };
  float mk = -INFINITY, lk = 0.f;
  if (lane < kMaxRec && used(lane)) {
    mk = __ldcg(rec(lane) + 128);
    lk = __ldcg(rec(lane) + 129);
  }
  float M = ls > 0.f ? ms : -INFINITY;
  float mx = lk > 0.f ? mk : -INFINITY;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  const float Mn = fmaxf(M, mx);
  const float wk = lk > 0.f ? lk * fast_exp2(mk - Mn) : 0.f;  // lane k: record k's weight
  const float a = ls > 0.f ? ls * fast_exp2(M - Mn) : 0.f;     // the own part's weight
  float W = a;
  float4 acc = make_float4(os.x * a, os.y * a, os.z * a, os.w * a);
  for (int k0 = 0; k0 < 2 * chunks; k0 += 4) {  // o of four records at a time
    float4 op[4];
#pragma unroll
    for (int u = 0; u < 4; ++u)
      op[u] = used(k0 + u) ? __ldcg(reinterpret_cast<const float4*>(rec(k0 + u)) + lane)
                           : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const float w = __shfl_sync(0xffffffffu, wk, k0 + u);
      W += w;
      acc = make_float4(fmaf(w, op[u].x, acc.x), fmaf(w, op[u].y, acc.y), fmaf(w, op[u].z, acc.z),
                        fmaf(w, op[u].w, acc.w));
    }
  }
  const float inv = W > 0.f ? 1.f / W : 0.f;
  const float x = acc.x * inv, y = acc.y * inv, z = acc.z * inv, w = acc.w * inv;
  const uint32_t lo16 = f32_to_bf16_bits(x) | (uint32_t(f32_to_bf16_bits(y)) << 16);
  const uint32_t hi16 = f32_to_bf16_bits(z) | (uint32_t(f32_to_bf16_bits(w)) << 16);
  *reinterpret_cast<uint2*>(c.out + idx * kHeadDim + lane * 4) = make_uint2(lo16, hi16);
}

cudaError_t launch_cascade_prep(const CascadeParams& c, cudaStream_t stream) {
  return launch_pdl(cascade_prep_kernel, dim3(static_cast<unsigned>(c.B)), dim3(256), 0, stream,
                    c);
}

cudaError_t launch_cascade_merge(const CascadeParams& c, cudaStream_t stream) {
  const int64_t warps = static_cast<int64_t>(c.B) * c.Hq;
  return launch_pdl_if(c.own_cap >= 0 || pdl_enabled(), cascade_merge_kernel,
                       dim3(static_cast<unsigned>((warps + 3) / 4)), dim3(128), 0, stream, c);
}

}  // namespace pkv
