// prefill.cu -- causal prefill attention over a paged KV cache on the
// fifth-generation tensor cores (tcgen05: operands in shared or tensor
// memory, fp32 accumulators in tensor memory).
//
// Sequence i's chunk of Lq new tokens (rows cu_q[i] .. cu_q[i+1]-1 of q, whose
// K and V rows are already in the cache) holds the last Lq of its ctx
// positions; new token j, at position ctx - Lq + j, attends positions
// 0 .. ctx - Lq + j ("Running Out of Cache": a block table maps positions to
// blocks; a chunk of one token is the decode step).
//
// Work: one CTA per (256 query rows, KV head, sequence).  The rows are the
// chunk's (token, query head) pairs of the KV head's group, token major (row
// r: token r / G, head r % G), so every K/V tile serves the whole group.  The
// CTA's rows form two tiles of 128 (the M of one tcgen05.mma), each with its
// own softmax warpgroup; one warp streams K/V, one warp issues the MMAs:
//
//   warps 0-3  softmax of row tile 0      warps 4-7  softmax of row tile 1
//   warp 8     K/V tiles of 128 keys by TMA into a 2-stage ring: one box per
//              run of a block's rows (gcd(bs, 128) rows), landing as 8-row x
//              128-byte swizzled atoms ordered (row group, column half)
//   warp 9     tensor-memory owner and MMA issuer (one thread)
//
// Tensor memory (512 columns, lane = query row of the tile): S_t = Q_t K^T in
// columns 128t .. 128t+127, O_t in columns 256 + 128t ..  For key tile j the
// MMA thread issues PV_0(j) S_0(j+1) | PV_1(j) S_1(j+1), so the tensor cores
// run one row tile's products while the other tile's softmax runs.  The
// softmax thread of row r reads its row of S, masks keys past its position
// and writes P = 2^(S * scale * log2 e - m) as packed bf16 pairs over the
// first 64 columns of S in place; PV_t(j) takes P straight from tensor memory
// (A operand) and V from shared memory (MN-major B operand).  The running
// maximum m is updated lazily: O and l are rescaled only when a row's
// maximum grows by more than 8 (a factor 2^8), so P stays below 256 and most
// tiles skip the rescale.  The MMAs of one thread complete in issue order, so
// the barrier that reports S_t(j+1) also reports PV_t(j): from then on the
// softmax warps own O_t until they hand P_t(j+1) over.
#include <cudaTypedefs.h>

#include <mutex>

#include "pkv_device.cuh"
#include "prefill.cuh"
#include "umma.cuh"

namespace pkv {

using namespace umma;

namespace {

constexpr int kStages = 2;
constexpr int kOffK = 2 * kOpBytes;                   // after Q_0, Q_1
constexpr int kStageBytes = 2 * kOpBytes;             // K then V
constexpr int kTilesBytes = kOffK + kStages * kStageBytes;  // 192 KiB
constexpr int kSmemBytes = kTilesBytes + 256 + 1024;
constexpr int kThreads = 320;

}  // namespace

__global__ void __launch_bounds__(kThreads, 1)
    prefill_kernel(const __grid_constant__ CUtensorMap tmk,
                   const __grid_constant__ CUtensorMap tmv, const PrefillParams p) {
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem = smem_raw + ((1024 - (smem_addr(smem_raw) & 1023)) & 1023);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kTilesBytes);
  uint64_t* kfull = bars;        // [2] K of a stage landed
  uint64_t* vfull = bars + 2;    // [2] V of a stage landed
  uint64_t* vempty = bars + 4;   // [2] both P V products reading a stage's V completed
  uint64_t* sfull = bars + 6;    // [2] S_t of the current key tile (and PV_t before it) done
  uint64_t* pfull = bars + 8;    // [2] P_t written (one arrival per warp)
  uint64_t* ofull = bars + 10;   // [2] the last PV_t completed
  uint64_t* drain = bars + 13;   // wind-down after an abort
  uint64_t* kempty = bars + 14;  // [2] both S products reading a stage's K completed
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 16);
  volatile int* abort = reinterpret_cast<volatile int*>(bars + 17);

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const int i = blockIdx.z;
  const int kvh = blockIdx.y;
  const int rt = gridDim.x - 1 - blockIdx.x;  // latest (heaviest) rows first
  const int G = p.G;

  grid_dependency_wait();
  grid_dependency_trigger();

  const int q0 = p.cu_q[i];
  const int Lq = p.cu_q[i + 1] - q0;
  const int ctx = p.ctx_lens[i];
  if (p.checked) {
    const int64_t cap = static_cast<int64_t>(p.max_blocks) * p.bs;
    if (Lq < 0 || Lq > p.max_q || ctx < Lq || ctx > cap) {
      if (tid == 0 && blockIdx.x == 0 && kvh == 0) record_error(p.err, kErrContext);
      return;
    }
  }
  const int rows = Lq * G;
  const int row0 = rt * 2 * kRowTile;
  if (row0 >= rows) return;  // this CTA's rows lie past the chunk (uniform)
  const int base = ctx - Lq;  // position of the chunk's first token
  const int last_row = min(row0 + 2 * kRowTile, rows) - 1;
  const int kend = base + last_row / G + 1;  // keys this CTA needs
  if (kend <= 0) return;  // only when ctx < Lq (caught in checked mode)
  const int ntiles = (kend + kKeys - 1) / kKeys;
  const bool two = rows > row0 + kRowTile;  // row tile 1 holds rows (else it idles)

  // Producer state (warp 8): lanes 0-7 copy K of run r of a tile, lanes
  // 16-23 V of the same run; every row tile of the sequence and KV head
  // reads the same K/V tiles, so they are kept in L2 for the CTAs after.
  const uint64_t policy = l2_policy_evict_last();
  const int run = p.run_rows;    // rows per box (16 .. 128, divides 128 and bs)
  const int runs = kKeys / run;  // boxes per tile and tensor (<= 8)
  const int prun = lane & 15;
  // block-table entry of run prun of tile j (-1: past the context or rejected)
  auto entry = [&](int j) -> int32_t {
    const int kpos = j * kKeys + prun * run;
    int32_t e = -1;
    if (j < ntiles && prun < runs && kpos < ctx) {
      e = p.block_tables[static_cast<int64_t>(i) * p.max_blocks + kpos / p.bs];
      if (p.checked && (e < 0 || e >= p.num_blocks)) {
        record_error(p.err, kErrBlockId);
        e = -1;  // skip the copy: stale rows, undefined output, no fault
      }
    }
    return e;
  };
  int32_t e = -1;        // entries of the next tile to issue
  int issued = 0;        // tiles whose K and V were both issued
  bool kv_half = false;  // tile `issued` has its K issued, not its V
  // Issue tiles [j0, j1); false when a wait gave up.
  auto produce = [&](int j0, int j1) -> bool {
    for (int j = j0; j < j1; ++j) {
      const int s = j & 1;
      const uint32_t loaded = __popc(__ballot_sync(kFull, lane < 16 && e >= 0));
      const int off = (j * kKeys + prun * run) % p.bs;
      const int32_t grp =
          e >= 0 ? static_cast<int32_t>(cache_row(e, kvh, p.Hkv, p.bs, off) >> 3) : 0;
      unsigned char* dst = smem + kOffK + s * kStageBytes + prun * run * kRowBytes;
      // K first: its stage frees once both S products of tile j - 2 are done
      if (j >= kStages &&
          !__all_sync(kFull, wait_or_abort(&kempty[s], ((j >> 1) - 1) & 1, abort, p.err)))
        return false;
      if (lane == 0) mbar_arrive_expect_tx(&kfull[s], loaded * run * kRowBytes);
      __syncwarp();
      if (lane < 16 && e >= 0) tma_load_4d(dst, &tmk, grp, &kfull[s], policy);
      // then V, whose stage frees after both P V products of tile j - 2
      if (j >= kStages &&
          !__all_sync(kFull, wait_or_abort(&vempty[s], ((j >> 1) - 1) & 1, abort, p.err))) {
        kv_half = true;  // K of tile `issued` is in flight
        return false;
      }
      if (lane == 0) mbar_arrive_expect_tx(&vfull[s], loaded * run * kRowBytes);
      __syncwarp();
      if (lane >= 16 && e >= 0) tma_load_4d(dst + kOpBytes, &tmv, grp, &vfull[s], policy);
      issued = j + 1;
      e = entry(j + 1);  // the next tile's entries load while this one lands
    }
    return true;
  };

  // Softmax row of this thread (warps 0-7).
  const int t = (warp >> 2) & 1;                // row tile
  const int lr = tid & (kRowTile - 1);          // row in the tile = tensor-memory lane
  const int r = row0 + t * kRowTile + lr;       // row of the chunk
  const bool valid = r < rows;
  const int rr = valid ? r : rows - 1;          // padding rows mirror the last row
  const int tok = rr / G;
  const int head = kvh * G + rr % G;
  const int pos = base + tok;
  const int64_t qrow = (static_cast<int64_t>(q0) + tok) * p.Hq + head;

  // Prologue: every role starts its global reads before the CTA-wide barrier.
  if (warp == 8) {
    if (lane == 0) {
      for (int b = 0; b < 12; ++b) mbar_init(&bars[b], (b == 8 || b == 9) ? 4 : 1);
      mbar_init(drain, 1);
      mbar_init(&kempty[0], 1);
      mbar_init(&kempty[1], 1);
      *abort = 0;
      fence_barrier_init();
      prefetch_tensormap(&tmk);
      prefetch_tensormap(&tmv);
    }
    __syncwarp();
    e = entry(0);
    produce(0, min(kStages, ntiles));  // no waits: the stages are fresh
  } else if (warp == 9) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_addr(tmem_slot)),
                 "r"(kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  } else {
    const uint4* src = reinterpret_cast<const uint4*>(p.q + qrow * kHeadDim);
    unsigned char* dst = smem + t * kOpBytes;
#pragma unroll
    for (int c = 0; c < 16; ++c) {
      const uint4 v = valid ? ld_global_nc_v4(src + c) : make_uint4(0u, 0u, 0u, 0u);
      *reinterpret_cast<uint4*>(dst + q_chunk_offset(lr, c)) = v;
    }
    fence_proxy_async_smem();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t smem_base = smem_addr(smem);

  if (warp < 8 && t == 1 && !two) {
    // row tile 1 holds no rows: its softmax warpgroup has nothing to do
  } else if (warp < 8) {
    // ================= softmax warpgroups =================
    const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t s_tm = tmem + lane_base + t * 128;
    const uint32_t o_tm = tmem + lane_base + 256 + t * 128;
    const float sc = p.qscale;
    float m_used = -INFINITY;  // the maximum P is taken against (scaled logits)
    float l = 0.f;
    bool ok = true;
    for (int j = 0; j < ntiles; ++j) {
      ok = __all_sync(kFull, wait_or_abort(&sfull[t], j & 1, abort, p.err));
      if (!ok) break;
      tc_fence_after();
      const int k0 = j * kKeys;
      const bool diag = k0 + kKeys - 1 > pos;  // some key of the tile lies past the row
      // general: a masked tile in this warp, or a negative scale (the maximum
      // of the scaled logits is then not the scaled maximum)
      const bool general = __any_sync(kFull, diag) || !(sc >= 0.f);
      // pass 1: the row maximum of the scaled, masked logits
      float tmax;
      if (!general) {
        float mx[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) mx[u] = -INFINITY;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          uint32_t a[32], b[32];
          tmem_ld32(a, s_tm + 64 * h);
          tmem_ld32(b, s_tm + 64 * h + 32);
          tmem_wait_ld(a);
          tmem_ready(b);
#pragma unroll
          for (int c = 0; c < 16; ++c) {
            mx[c & 3] = fmax3(mx[c & 3], __uint_as_float(a[2 * c]), __uint_as_float(a[2 * c + 1]));
            mx[(c + 2) & 3] =
                fmax3(mx[(c + 2) & 3], __uint_as_float(b[2 * c]), __uint_as_float(b[2 * c + 1]));
          }
        }
        tmax = fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])) * sc;
      } else {
        float mx[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) mx[u] = -INFINITY;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          uint32_t a[32], b[32];
          tmem_ld32(a, s_tm + 64 * h);
          tmem_ld32(b, s_tm + 64 * h + 32);
          tmem_wait_ld(a);
          tmem_ready(b);
#pragma unroll
          for (int c = 0; c < 64; ++c) {
            const float x = __uint_as_float(c < 32 ? a[c] : b[c - 32]) * sc;
            mx[c & 7] = fmaxf(mx[c & 7], !diag || k0 + 64 * h + c <= pos ? x : -INFINITY);
          }
        }
        tmax = fmaxf(fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])),
                     fmaxf(fmaxf(mx[4], mx[5]), fmaxf(mx[6], mx[7])));
      }
      const float m_new = fmaxf(m_used, tmax);
      if (j == 0) {
        m_used = m_new;  // finite: position 0 is visible to every row
      } else {
        const bool grow = m_new > m_used + kRescaleLog2;
        if (__any_sync(kFull, grow)) {
          const float alpha = grow ? fast_exp2(m_used - m_new) : 1.f;
          if (grow) {
            l *= alpha;
            m_used = m_new;
          }
#pragma unroll
          for (int c0 = 0; c0 < kHeadDim; c0 += 32) {
            uint32_t w[32];
            tmem_ld32(w, o_tm + c0);
            tmem_wait_ld(w);
#pragma unroll
            for (int c = 0; c < 32; ++c) w[c] = __float_as_uint(__uint_as_float(w[c]) * alpha);
            tmem_st32(o_tm + c0, w);
          }
        }
      }
      // pass 2: P = 2^(s * scale - m) as bf16 pairs over the columns already read
      const float neg_m = -m_used;
      if (!general) {
        const uint64_t sc2 = f2_pack(__float_as_uint(sc), __float_as_uint(sc));
        const uint64_t nm2 = f2_pack(__float_as_uint(neg_m), __float_as_uint(neg_m));
        uint64_t ls2[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) ls2[u] = 0ull;  // (+0, +0)
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          uint32_t a[32], b[32];
          tmem_ld32(a, s_tm + 64 * h);
          tmem_ld32(b, s_tm + 64 * h + 32);
          tmem_wait_ld(a);
          tmem_ready(b);
          uint32_t pk[32];
#pragma unroll
          for (int c = 0; c < 32; ++c) {
            const uint32_t u0 = c < 16 ? a[2 * c] : b[2 * c - 32];
            const uint32_t u1 = c < 16 ? a[2 * c + 1] : b[2 * c - 31];
            float x0, x1;
            f2_unpack(f2_fma(f2_pack(u0, u1), sc2, nm2), x0, x1);
            const float e0 = fast_exp2(x0), e1 = fast_exp2(x1);
            const uint64_t e2 = f2_pack(__float_as_uint(e0), __float_as_uint(e1));
            ls2[c & 3] = f2_add(ls2[c & 3], e2);
            pk[c] = pack_bf16x2(e0, e1);
          }
          tmem_st32(s_tm + 32 * h, pk);
        }
        float l0, l1, l2, l3;
        f2_unpack(f2_add(ls2[0], ls2[1]), l0, l1);
        f2_unpack(f2_add(ls2[2], ls2[3]), l2, l3);
        l += (l0 + l2) + (l1 + l3);
      } else {
        float ls[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) ls[u] = 0.f;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          uint32_t a[32], b[32];
          tmem_ld32(a, s_tm + 64 * h);
          tmem_ld32(b, s_tm + 64 * h + 32);
          tmem_wait_ld(a);
          tmem_ready(b);
          // keys of this half the row sees: bit c of (lo, hi) for key 64h + c
          const int seen = diag ? min(max(pos - k0 - 64 * h + 1, 0), 64) : 64;
          const uint32_t lo = seen >= 32 ? 0xffffffffu : (1u << seen) - 1u;
          const uint32_t hi =
              seen >= 64 ? 0xffffffffu : (seen <= 32 ? 0u : (1u << (seen - 32)) - 1u);
          uint32_t pk[32];
#pragma unroll
          for (int c = 0; c < 32; ++c) {
            const uint32_t u0 = c < 16 ? a[2 * c] : b[2 * c - 32];
            const uint32_t u1 = c < 16 ? a[2 * c + 1] : b[2 * c - 31];
            float e0 = fast_exp2(fmaf(__uint_as_float(u0), sc, neg_m));
            float e1 = fast_exp2(fmaf(__uint_as_float(u1), sc, neg_m));
            const uint32_t bits = c < 16 ? lo : hi;
            e0 = (bits >> ((2 * c) & 31)) & 1u ? e0 : 0.f;
            e1 = (bits >> ((2 * c + 1) & 31)) & 1u ? e1 : 0.f;
            ls[c & 7] += e0 + e1;
            pk[c] = pack_bf16x2(e0, e1);
          }
          tmem_st32(s_tm + 32 * h, pk);
        }
        l += ((ls[0] + ls[1]) + (ls[2] + ls[3])) + ((ls[4] + ls[5]) + (ls[6] + ls[7]));
      }
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&pfull[t]);
    }
    if (ok) ok = __all_sync(kFull, wait_or_abort(&ofull[t], 0, abort, p.err));
    if (ok) {
      tc_fence_after();
      const float inv = l > 0.f ? 1.f / l : 0.f;
      uint4* dst = reinterpret_cast<uint4*>(p.out + qrow * kHeadDim);
#pragma unroll
      for (int c0 = 0; c0 < kHeadDim; c0 += 32) {
        uint32_t w[32];
        tmem_ld32(w, o_tm + c0);
        tmem_wait_ld(w);
        if (valid) {
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            uint4 o;
            o.x = pack_bf16x2(__uint_as_float(w[8 * q + 0]) * inv, __uint_as_float(w[8 * q + 1]) * inv);
            o.y = pack_bf16x2(__uint_as_float(w[8 * q + 2]) * inv, __uint_as_float(w[8 * q + 3]) * inv);
            o.z = pack_bf16x2(__uint_as_float(w[8 * q + 4]) * inv, __uint_as_float(w[8 * q + 5]) * inv);
            o.w = pack_bf16x2(__uint_as_float(w[8 * q + 6]) * inv, __uint_as_float(w[8 * q + 7]) * inv);
            dst[c0 / 8 + q] = o;
          }
        }
      }
    }
  } else if (warp == 8) {
    // ================= K/V producer: the remaining tiles =================
    produce(kStages, ntiles);
    if (*abort && lane == 0) {
      // let the copies in flight land before the CTA's shared memory is released
      for (int j = max(0, issued - kStages); j < issued; ++j) {
        mbar_wait_bounded(&kfull[j & 1], (j >> 1) & 1);
        mbar_wait_bounded(&vfull[j & 1], (j >> 1) & 1);
      }
      if (kv_half) mbar_wait_bounded(&kfull[issued & 1], (issued >> 1) & 1);
    }
  } else if (warp == 9) {
    // ================= MMA issuer (warp 9, lane 0 issues) =================
    auto issue_s = [&](int t, int j) {  // S_t = Q_t K_j^T
      const uint32_t q_addr = smem_base + t * kOpBytes;
      const uint32_t k_addr = smem_base + kOffK + (j & 1) * kStageBytes;
#pragma unroll
      for (int kk = 0; kk < 8; ++kk) {
        const uint32_t koff = (kk & 3) * 32;
        umma_ss(tmem + t * 128, smem_desc(q_addr + (kk >> 2) * kHalfBytes + koff, 16, 1024),
                smem_desc(k_addr + (kk >> 2) * 1024 + koff, 16, 2048), kIdescS, kk > 0);
      }
    };
    auto issue_pv = [&](int t, int j) {  // O_t (+)= P_t V_j
      const uint32_t v_addr = smem_base + kOffK + (j & 1) * kStageBytes + kOpBytes;
#pragma unroll
      for (int kk = 0; kk < 8; ++kk)
        umma_ts(tmem + 256 + t * 128, tmem + t * 128 + kk * 8,
                smem_desc(v_addr + kk * 4096, 1024, 2048), kIdescPV, (j > 0 || kk > 0));
    };
    // Q is in shared memory: written and fenced before the CTA-wide barrier
    bool ok = __all_sync(kFull, wait_or_abort(&kfull[0], 0, abort, p.err));
    if (ok) {
      tc_fence_after();
      if (lane == 0) {
        issue_s(0, 0);
        umma_commit(&sfull[0]);
        if (two) {
          issue_s(1, 0);
          umma_commit(&sfull[1]);
        }
        if (kStages < ntiles) umma_commit(&kempty[0]);
      }
      __syncwarp();
    }
    for (int j = 0; ok && j < ntiles; ++j) {
      const int s = j & 1;
      ok = __all_sync(kFull, wait_or_abort(&vfull[s], (j >> 1) & 1, abort, p.err));
      if (!ok) break;
      const int k0 = j * kKeys;
      if (k0 + kKeys > ctx) {  // zero V rows at or past the context (0 x stale bytes)
        unsigned char* vt = smem + kOffK + s * kStageBytes + kOpBytes;
        const int first = ctx - k0;
        for (int idx = lane; idx < (kKeys - first) * 16; idx += 32)
          *reinterpret_cast<uint4*>(vt + kv_chunk_offset(first + (idx >> 4), idx & 15)) =
              make_uint4(0u, 0u, 0u, 0u);
        fence_proxy_async_smem();
        __syncwarp();
      }
      const bool more = j + 1 < ntiles;
      ok = __all_sync(kFull, wait_or_abort(&pfull[0], j & 1, abort, p.err));
      if (ok && more)
        ok = __all_sync(kFull, wait_or_abort(&kfull[s ^ 1], ((j + 1) >> 1) & 1, abort, p.err));
      if (!ok) break;
      tc_fence_after();
      if (lane == 0) {
        issue_pv(0, j);
        if (!two && j + kStages < ntiles) umma_commit(&vempty[s]);
        if (more) {
          issue_s(0, j + 1);
          umma_commit(&sfull[0]);
          if (!two && j + 1 + kStages < ntiles) umma_commit(&kempty[s ^ 1]);
        } else {
          umma_commit(&ofull[0]);
        }
      }
      __syncwarp();
      if (!two) continue;  // a single row tile
      ok = __all_sync(kFull, wait_or_abort(&pfull[1], j & 1, abort, p.err));
      if (!ok) break;
      tc_fence_after();
      if (lane == 0) {
        issue_pv(1, j);
        if (j + kStages < ntiles) umma_commit(&vempty[s]);  // the producer reuses the stage
        if (more) {
          issue_s(1, j + 1);
          umma_commit(&sfull[1]);
          if (j + 1 + kStages < ntiles) umma_commit(&kempty[s ^ 1]);
        } else {
          umma_commit(&ofull[1]);
        }
      }
      __syncwarp();
    }
    if (!ok && lane == 0) {
      // let the MMAs in flight finish before tensor memory is released
      umma_commit(drain);
      mbar_wait_bounded(drain, 0);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 9) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                 "r"(kTmemCols)
                 : "memory");
  }
}

namespace {

PFN_cuTensorMapEncodeTiled_v12000 prefill_map_encoder() {
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

bool encode_prefill_runs(CUtensorMap* map, const void* base, int64_t rows, int run_rows) {
  auto enc = prefill_map_encoder();
  if (enc == nullptr || rows % 8 != 0 || run_rows % 8 != 0 || run_rows > 128) return false;
  // dims (innermost first): 64 columns, 8 rows of a group, 2 column halves, groups
  const cuuint64_t dims[4] = {64u, 8u, 2u, static_cast<cuuint64_t>(rows / 8)};
  const cuuint64_t strides[3] = {static_cast<cuuint64_t>(kRowBytes), 128u,
                                 static_cast<cuuint64_t>(8 * kRowBytes)};
  const cuuint32_t box[4] = {64u, 8u, 2u, static_cast<cuuint32_t>(run_rows / 8)};
  const cuuint32_t estr[4] = {1u, 1u, 1u, 1u};
  const CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims,
                         strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                         CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

cudaError_t launch_prefill(const CUtensorMap& tk, const CUtensorMap& tv, const PrefillParams& p,
                           cudaStream_t stream) {
  static bool attr_done = false;  // one device per process in practice; repeated calls are harmless
  if (!attr_done) {
    const cudaError_t e = cudaFuncSetAttribute(
        prefill_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    if (e != cudaSuccess) return e;
    attr_done = true;
  }
  const int row_tiles = (p.max_q * p.G + 2 * kRowTile - 1) / (2 * kRowTile);
  return launch_pdl(prefill_kernel, dim3(row_tiles, p.Hkv, p.num_seqs), dim3(kThreads),
                    kSmemBytes, stream, tk, tv, p);
}

}  // namespace pkv
