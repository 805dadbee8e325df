// prefix.cu -- shared-prefix attention for decode on the fifth-generation
// tensor cores (tcgen05): sequences sampled from one prompt share its blocks
// ("Running Out of Cache", "Fragmentation is lost users"), and a group's
// shared positions are attended here once for all its members.  Softmax over
// a context splits into per-part partial results (o, m, l); the merge kernel
// (cascade.cu) folds this kernel's records with each member's own positions.
//
// Work: one CTA per (128 rows, KV head, group, chunk of the shared
// positions), chunks with the most key tiles first.  The rows are the
// group's (member, query head) pairs of the KV head; every row attends every
// shared position (no causal mask).  A group has few rows (28 for 4 branches
// at G = 7), so both row tiles of the CTA hold the same rows (one Q tile in
// shared memory, row tile 1's copy further down when the rows fit twice) and
// take alternate key tiles: tile j goes to row tile j % 2, whose S, softmax
// and P V run while the other row tile's run -- each writes its own record
// (half j % 2).  K/V come by TMA (the 4-D boxes of prefill.cu) through a
// 3-stage ring: with each tile used by one row tile, a third stage keeps the
// next loads ahead of the chain S -> softmax -> P V.  K and V have a producer
// warp each.  Tensor memory as in prefill.cu: S_t in columns 128t .., O_t in
// 256 + 128t ..; P over S in place; lazy rescale.
//
// Own positions (with a host bound on them): a group's last chunk takes
// extra key tiles holding every member's own positions, own_slots key slots
// per member, and a row sees only its member's slots (a per-row window in
// the softmax mask; V rows of empty slots are zeroed).  The records then
// hold the whole attention, split in parts.  With one chunk per group the
// CTA also merges its two halves and writes the bf16 output: the call is
// this one launch.
#include "pkv_device.cuh"
#include "prefix.cuh"
#include "umma.cuh"

namespace pkv {

using namespace umma;

namespace {

constexpr int kStages = 3;
constexpr int kOffK = kOpBytes;                       // after the one Q tile
constexpr int kStageBytes = 2 * kOpBytes;             // K then V
constexpr int kTilesBytes = kOffK + kStages * kStageBytes;  // 224 KiB
constexpr int kOwnLenOff = kTilesBytes + 256;                // [members of the row block] own lengths
constexpr int kOwnLenBytes = 576;                           // up to 144 members
constexpr int kSmemBytes = kOwnLenOff + kOwnLenBytes + 1024;
// The fused ending's exchange of the two halves' rows, [2][kRowTile][kPrefixRecStride]
// fp32, in the K/V stages (idle by then).
static_assert(2 * kRowTile * kPrefixRecStride * 4 <= kStages * kStageBytes, "exchange area");

// Bits [a, b) of a 32-bit word, 0 <= a, b <= 32.
__device__ __forceinline__ uint32_t bit_range(int a, int b) {
  if (b <= a) return 0u;
  const uint32_t below_b = b >= 32 ? 0xffffffffu : (1u << b) - 1u;
  const uint32_t below_a = a >= 32 ? 0xffffffffu : (1u << a) - 1u;
  return below_b & ~below_a;
}
constexpr int kThreads = 352;  // 8 softmax warps, K producer, MMA issuer, V producer
static_assert(kSmemBytes <= 232448, "shared memory per CTA");

}  // namespace

__global__ void __launch_bounds__(kThreads, 1)
    prefix_kernel(const __grid_constant__ CUtensorMap tmk,
                  const __grid_constant__ CUtensorMap tmv, const PrefixParams p) {
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem = smem_raw + ((1024 - (smem_addr(smem_raw) & 1023)) & 1023);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kTilesBytes);
  uint64_t* kfull = bars;        // [3] K of a stage landed
  uint64_t* vfull = bars + 3;    // [3] V of a stage landed
  uint64_t* kempty = bars + 6;   // [3] the S product reading a stage's K completed
  uint64_t* vempty = bars + 9;   // [3] the P V product reading a stage's V completed
  uint64_t* sfull = bars + 12;   // [2] S_t of its current tile (and PV_t before it) done
  uint64_t* pfull = bars + 14;   // [2] P_t written (one arrival per warp)
  uint64_t* ofull = bars + 16;   // [2] the last PV_t completed
  uint64_t* drain = bars + 18;   // wind-down after an abort
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 19);
  volatile int* abort = reinterpret_cast<volatile int*>(bars + 20);

  int* pick = reinterpret_cast<int*>(bars + 22);  // [2] the chosen key-tile count, chunk
  int* own_len = reinterpret_cast<int*>(smem + kOwnLenOff);  // own positions of the members here

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const int kvh = blockIdx.y;
  const int G = p.G;

  grid_dependency_wait();
  grid_dependency_trigger();

  // ---- longest chunks first.  CTAs start in index order as SMs free up, so
  // CTA z takes the chunk of rank z in the order (key tiles descending, chunk
  // index ascending): the long chunks start first and the short ones fill
  // the tail.  A counting sort over key-tile counts, its scratch in the K/V
  // stages (nothing is loaded there yet).
  int item = blockIdx.z;
  {
    const int N = p.num_groups * p.chunks;
    const int nb = p.chunk_keys / kKeys + 1;  // key-tile counts 0 .. chunk_keys / 128
    int* shared_pos = reinterpret_cast<int*>(smem + kOffK);  // [num_groups]
    int* hist = shared_pos + p.num_groups;                   // [nb]
    int* start = hist + nb;                                  // [nb] rank of a count's first chunk
    if (p.num_groups + 2 * nb <= kStages * kStageBytes / 4) {
      for (int i = tid; i < p.num_groups; i += kThreads)
        shared_pos[i] = min(max(p.shared_blocks[i], 0), p.max_blocks) * static_cast<int>(p.bs);
      for (int i = tid; i < nb; i += kThreads) hist[i] = 0;
      if (tid == 0) {  // identity, should no count match (it always does: z < N)
        pick[0] = -1;
        pick[1] = blockIdx.z;
      }
      __syncthreads();
      auto tiles_of = [&](int i) -> int {
        const int kb = (i % p.chunks) * p.chunk_keys;
        const int len = min(shared_pos[i / p.chunks] - kb, p.chunk_keys);
        return len > 0 ? (len + kKeys - 1) / kKeys : 0;
      };
      for (int i = tid; i < N; i += kThreads) atomicAdd(&hist[tiles_of(i)], 1);
      __syncthreads();
      if (warp == 0) {  // start[b] = chunks with more key tiles than b
        int carry = 0;
        for (int top = nb - 1; top >= 0; top -= 32) {
          const int b = top - lane;
          const int v = b >= 0 ? hist[b] : 0;
          int incl = v;
#pragma unroll
          for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(kFull, incl, o);
            if (lane >= o) incl += y;
          }
          if (b >= 0) start[b] = carry + incl - v;
          carry += __shfl_sync(kFull, incl, 31);
        }
      }
      __syncthreads();
      const int z = blockIdx.z;
      for (int b = tid; b < nb; b += kThreads)
        if (start[b] <= z && z < start[b] + hist[b]) pick[0] = b;
      __syncthreads();
      const int b = pick[0];
      if (warp == 0 && b >= 0 && b < nb) {  // the (z - start[b])-th chunk, in index order, with b key tiles
        int want = z - start[b];
        for (int base = 0; base < N; base += 32) {
          const int i = base + lane;
          const unsigned m = __ballot_sync(kFull, i < N && tiles_of(i) == b);
          const int c = __popc(m);
          if (want < c) {
            unsigned x = m;
            for (int k = 0; k < want; ++k) x &= x - 1;
            if (lane == 0) pick[1] = base + __ffs(x) - 1;
            break;
          }
          want -= c;
        }
      }
      fence_proxy_async_smem();  // the stages are TMA destinations from here on
      __syncthreads();
      item = min(max(pick[1], 0), N - 1);
    }
  }
  const int g = item / p.chunks;
  const int kc = item % p.chunks;

  const int seq = p.group_start[g];  // the group's first member: its block table
  const int rows = (p.group_start[g + 1] - seq) * G;
  const int row0 = blockIdx.x * kRowTile;
  if (row0 >= rows) return;  // past the group's rows (uniform)
  const int sb_in = p.shared_blocks[g];
  const int sb = min(max(sb_in, 0), p.max_blocks);
  const int ctx = sb * static_cast<int>(p.bs);  // the shared positions
  const int kbase = kc * p.chunk_keys;
  // the group's chunks (at least one when own tiles follow: the last takes them)
  const int nch = (ctx + p.chunk_keys - 1) / p.chunk_keys;
  const int nch_all = p.own_slots > 0 ? max(nch, 1) : nch;
  if (kc >= nch_all) return;  // a chunk past them (uniform)
  const int kend = min(ctx, kbase + p.chunk_keys);
  const int nts = kend > kbase ? (kend - kbase + kKeys - 1) / kKeys : 0;  // shared key tiles
  const int rows_here = min(rows - row0, kRowTile);
  const int m_first = row0 / G;  // the row block's members: m_first .. + members_here - 1
  const int members_here = (row0 + rows_here - 1) / G - m_first + 1;
  const int nto = p.own_slots > 0 && kc == nch_all - 1
                      ? (members_here * p.own_slots + kKeys - 1) / kKeys
                      : 0;  // own key tiles
  const int ntiles = nts + nto;
  const bool two = ntiles > 1;  // row tile 1 has odd tiles to take
  const bool fused = p.out != nullptr;

  // Producers: warp 8 copies K, warp 10 copies V, each on its own stage
  // schedule -- K of tile j waits only for the S product of tile j - 3, not
  // for its P V, so the K loads run a tile further ahead of the S chain.
  // Lane r < runs copies run r of a tile.
  const uint64_t policy = l2_policy_evict_first();  // read once
  const int run = p.run_rows;    // rows per box (16 .. 128, divides 128 and bs)
  const int runs = kKeys / run;  // boxes per tile and tensor (<= 8)
  // Tile j < nts: shared positions kbase + 128 j ..; else own slots
  // 128 (j - nts) .. (member k's own position o at slot k * own_slots + o).
  // A run of rows never crosses a block: own_slots and every run start are
  // multiples of run, which divides bs.
  auto entry = [&](int j) -> int32_t {
    int32_t e = -1;
    if (j < ntiles && lane < runs) {
      int64_t at = -1;  // index into the block tables
      if (j < nts) {
        const int kpos = kbase + j * kKeys + lane * run;
        if (kpos < ctx) at = static_cast<int64_t>(seq) * p.max_blocks + kpos / p.bs;
      } else {
        const int s0 = (j - nts) * kKeys + lane * run;
        const int k = s0 / p.own_slots, o = s0 - k * p.own_slots;
        if (k < members_here && o < own_len[k])
          at = static_cast<int64_t>(seq + m_first + k) * p.max_blocks + sb + o / p.bs;
      }
      if (at >= 0) {
        e = p.block_tables[at];
        if (p.checked && (e < 0 || e >= p.num_blocks)) {
          record_error(p.err, kErrBlockId);
          e = -1;  // skip the copy: stale rows, undefined output, no fault
        }
      }
    }
    return e;
  };
  auto run_offset = [&](int j) -> int {  // in-block offset of this lane's run of tile j
    if (j < nts) return (kbase + j * kKeys + lane * run) % static_cast<int>(p.bs);
    const int s0 = (j - nts) * kKeys + lane * run;
    return (s0 % p.own_slots) % static_cast<int>(p.bs);
  };
  const bool is_v = warp == 10;
  const CUtensorMap* tm = is_v ? &tmv : &tmk;
  uint64_t* full = is_v ? vfull : kfull;
  uint64_t* empty = is_v ? vempty : kempty;
  int32_t e = -1;   // entries of the next tile to issue
  int issued = 0;   // tiles this producer issued
  auto produce = [&](int j0, int j1) -> bool {
    for (int j = j0; j < j1; ++j) {
      const int s = j % kStages;
      const uint32_t u = static_cast<uint32_t>(j / kStages);  // use of the stage
      const uint32_t loaded = __popc(__ballot_sync(kFull, e >= 0));
      const int off = run_offset(j);
      const int32_t grp =
          e >= 0 ? static_cast<int32_t>(cache_row(e, kvh, p.Hkv, p.bs, off) >> 3) : 0;
      unsigned char* dst =
          smem + kOffK + s * kStageBytes + (is_v ? kOpBytes : 0) + lane * run * kRowBytes;
      if (j >= kStages &&
          !__all_sync(kFull, wait_or_abort(&empty[s], (u - 1) & 1, abort, p.err)))
        return false;
      if (lane == 0) mbar_arrive_expect_tx(&full[s], loaded * run * kRowBytes);
      __syncwarp();
      if (e >= 0) tma_load_4d(dst, tm, grp, &full[s], policy);
      issued = j + 1;
      e = entry(j + 1);  // the next tile's entries load while this one lands
    }
    return true;
  };
  // after an abort: let this producer's copies in flight land before the
  // CTA's shared memory is released
  auto drain_copies = [&]() {
    if (*abort && lane == 0)
      for (int j = max(0, issued - kStages); j < issued; ++j)
        mbar_wait_bounded(&full[j % kStages], static_cast<uint32_t>(j / kStages) & 1);
  };

  // Rows: row r -> (member r / G, head r % G).  Both row tiles hold the same
  // rows; a TMEM lane quadrant can only be read by the warps of one SM
  // sub-partition, so when the rows fit twice (at most 64), row tile 1 reads
  // them from a copy `shift` rows further down the Q tile: its softmax then
  // runs in other quadrants, on other sub-partitions, than row tile 0's.
  // Softmax warps whose quadrant holds none of their row tile's rows idle.
  const int t = (warp >> 2) & 1;
  const int lr = tid & (kRowTile - 1);  // Q row / TMEM lane
  const int nq = (rows_here + 31) / 32;                  // quadrants of a row tile at work
  const int shift = two && nq <= 2 ? 32 * nq : 0;
  const int qr = shift > 0 && lr >= shift && lr < 2 * shift ? lr - shift : lr;  // row of Q lane lr
  const int rr = qr < rows_here ? row0 + qr : rows - 1;  // padding rows mirror the last row
  const int64_t qrow = (static_cast<int64_t>(seq) + rr / G) * p.Hq + kvh * G + rr % G;
  // row tile t's row at lane lr, and whether row tile t owns that lane
  auto row_of = [&]() { return t == 1 ? lr - shift : lr; };
  auto owns = [&]() {
    const int rt = row_of();
    return rt >= 0 && rt < rows_here && (t == 1 || shift == 0 || lr < shift);
  };

  if (warp == 8) {
    if (lane == 0) {
      for (int b = 0; b < 18; ++b) mbar_init(&bars[b], (b == 14 || b == 15) ? nq : 1);
      mbar_init(drain, 1);
      *abort = 0;
      fence_barrier_init();
      prefetch_tensormap(&tmk);
      prefetch_tensormap(&tmv);
    }
    if (nto > 0) {
      // own positions of the row block's members (read before their tiles'
      // entries need them), clamped to the bound and to the table
      const int cap = min(min(p.own_cap, p.own_slots),
                          (p.max_blocks - sb) * static_cast<int>(p.bs));
      for (int k = lane; k < members_here; k += 32) {
        const int n = p.ctx[seq + m_first + k] - ctx;
        if (p.checked && (n < 0 || n > cap || sb != sb_in)) record_error(p.err, kErrContext);
        own_len[k] = min(max(n, 0), cap);
      }
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
  } else if (warp < 4) {
    // the Q tile; the MMA warp reads it after the barrier
    const uint4* src = reinterpret_cast<const uint4*>(p.q + qrow * kHeadDim);
#pragma unroll
    for (int c = 0; c < 16; ++c) {
      const uint4 v = qr < rows_here ? ld_global_nc_v4(src + c) : make_uint4(0u, 0u, 0u, 0u);
      *reinterpret_cast<uint4*>(smem + q_chunk_offset(lr, c)) = v;
    }
    fence_proxy_async_smem();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t smem_base = smem_addr(smem);

  // a softmax lane's (l, m) and whether its O is complete, for the fused ending
  float fin_l = 0.f, fin_m = -INFINITY;
  bool fin_ok = false;
  auto record_of = [&](int half) {  // this lane's record: (member, head) row, half of the chunk
    return p.rec_out + ((((static_cast<int64_t>(g) * p.chunks + kc) * 2 + half) * p.Hkv + kvh) *
                            p.rows + row0 + row_of()) *
                           kPrefixRecStride;
  };

  if (warp < 8 && ((t == 1 && !two) || !__any_sync(kFull, owns()))) {
    // one key tile (row tile 1 has nothing to do), or no row of this row tile
    // in this warp's quadrant.  With own tiles the merge reads both halves of
    // every chunk: half 1 of a one-tile chunk is an empty record.
    if (t == 1 && !two && p.own_slots > 0 && !fused && owns()) {
      float* rec = record_of(1);
#pragma unroll
      for (int q = 0; q < kHeadDim / 4; ++q)
        reinterpret_cast<float4*>(rec)[q] = make_float4(0.f, 0.f, 0.f, 0.f);
      rec[128] = -INFINITY;
      rec[129] = 0.f;
    }
  } else if (warp < 8) {
    // ================= softmax: row tile t takes key tiles t, t + 2, ... =================
    const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t s_tm = tmem + lane_base + t * 128;
    const uint32_t o_tm = tmem + lane_base + 256 + t * 128;
    const float sc = p.qscale;
    // this lane's record: (member, head) row of row tile t, half t of the chunk
    const bool own = owns();
    // the keys this lane's row sees: shared positions [0, ctx), then its
    // member's own slots [own_lo, own_hi) of the own tiles
    const int own_k = (row0 + min(max(row_of(), 0), rows_here - 1)) / G - m_first;  // member
    float m_used = -INFINITY;  // the maximum P is taken against (scaled logits)
    float l = 0.f;
    bool ok = true;
    for (int j = t, n = 0; j < ntiles; j += 2, ++n) {
      ok = __all_sync(kFull, wait_or_abort(&sfull[t], n & 1, abort, p.err));
      if (!ok) break;
      tc_fence_after();
      // tile keys k0 .. k0 + 127 against the row's window [wlo, whi)
      const bool own_tile = j >= nts;
      const int k0 = own_tile ? (j - nts) * kKeys : kbase + j * kKeys;
      const int wlo = own_tile ? own_k * p.own_slots : 0;
      const int whi = own_tile ? wlo + own_len[own_k] : ctx;
      const bool diag = k0 < wlo || k0 + kKeys > whi;  // some key of the tile is not seen
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
        // (not unrolled: masked tiles are few, and a smaller kernel measured faster)
#pragma unroll 1
        for (int h = 0; h < 2; ++h) {
          uint32_t a[32], b[32];
          tmem_ld32(a, s_tm + 64 * h);
          tmem_ld32(b, s_tm + 64 * h + 32);
          tmem_wait_ld(a);
          tmem_ready(b);
#pragma unroll
          for (int c = 0; c < 64; ++c) {
            const float x = __uint_as_float(c < 32 ? a[c] : b[c - 32]) * sc;
            const int key = k0 + 64 * h + c;
            mx[c & 7] = fmaxf(mx[c & 7], !diag || (key >= wlo && key < whi) ? x : -INFINITY);
          }
        }
        tmax = fmaxf(fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])),
                     fmaxf(fmaxf(mx[4], mx[5]), fmaxf(mx[6], mx[7])));
      }
      const float m_new = fmaxf(m_used, tmax);
      if (n == 0) {
        // -inf for a row that sees none of the tile's keys (an own tile of
        // another member): its P is all zero by the mask, and the first
        // tile it sees scales the empty O and l by 2^-inf = 0
        m_used = m_new;
      } else {
        const bool grow = m_new > m_used + kRescaleLog2;
        if (__any_sync(kFull, grow)) {
          const float alpha = grow ? fast_exp2(m_used - m_new) : 1.f;
          if (grow) {
            l *= alpha;
            m_used = m_new;
          }
          // (not unrolled: the rescale is rare, and a smaller kernel measured faster)
#pragma unroll 1
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
        // (not unrolled: masked tiles are few, and a smaller kernel measured faster)
#pragma unroll 1
        for (int h = 0; h < 2; ++h) {
          uint32_t a[32], b[32];
          tmem_ld32(a, s_tm + 64 * h);
          tmem_ld32(b, s_tm + 64 * h + 32);
          tmem_wait_ld(a);
          tmem_ready(b);
          // keys of this half the row sees, [a, b): bit c of (lo, hi) for key 64h + c
          const int kh = k0 + 64 * h;
          const int ka = diag ? min(max(wlo - kh, 0), 64) : 0;
          const int kb = diag ? min(max(whi - kh, 0), 64) : 64;
          const uint32_t lo = bit_range(min(ka, 32), min(kb, 32));
          const uint32_t hi = bit_range(max(ka - 32, 0), max(kb - 32, 0));
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
    fin_l = l;
    fin_m = m_used;
    fin_ok = ok;
    if (ok && !fused) {
      // fp32 record of this (member, head) and half: o / l, m, l
      float* const rec = record_of(t);
      tc_fence_after();
      const float inv = l > 0.f ? 1.f / l : 0.f;
#pragma unroll
      for (int c0 = 0; c0 < kHeadDim; c0 += 32) {
        uint32_t w[32];
        tmem_ld32(w, o_tm + c0);
        tmem_wait_ld(w);
        if (own) {
#pragma unroll
          for (int q = 0; q < 8; ++q)
            reinterpret_cast<float4*>(rec + c0)[q] =
                make_float4(__uint_as_float(w[4 * q]) * inv, __uint_as_float(w[4 * q + 1]) * inv,
                            __uint_as_float(w[4 * q + 2]) * inv,
                            __uint_as_float(w[4 * q + 3]) * inv);
        }
      }
      if (own) {
        rec[128] = m_used;
        rec[129] = l;
      }
    }
  } else if (warp == 8) {
    // ================= K producer: the remaining tiles =================
    produce(kStages, ntiles);
    drain_copies();
  } else if (warp == 10) {
    // ================= V producer: every tile (the barriers exist now) =================
    e = entry(0);
    produce(0, ntiles);
    drain_copies();
  } else if (warp == 9) {
    // ================= MMA issuer (lane 0 issues) =================
    // order S_0(0) S_1(1) | PV_0(0) S_0(2) | PV_1(1) S_1(3) | PV_0(2) S_0(4) | ...
    auto issue_s = [&](int rt, int j) {  // S_rt = Q K_j^T
      const uint32_t k_addr = smem_base + kOffK + (j % kStages) * kStageBytes;
#pragma unroll
      for (int kk = 0; kk < 8; ++kk) {
        const uint32_t koff = (kk & 3) * 32;
        umma_ss(tmem + rt * 128, smem_desc(smem_base + (kk >> 2) * kHalfBytes + koff, 16, 1024),
                smem_desc(k_addr + (kk >> 2) * 1024 + koff, 16, 2048), kIdescS, kk > 0);
      }
    };
    auto issue_pv = [&](int rt, int j, bool acc) {  // O_rt (+)= P_rt V_j
      const uint32_t v_addr = smem_base + kOffK + (j % kStages) * kStageBytes + kOpBytes;
#pragma unroll
      for (int kk = 0; kk < 8; ++kk)
        umma_ts(tmem + 256 + rt * 128, tmem + rt * 128 + kk * 8,
                smem_desc(v_addr + kk * 4096, 1024, 2048), kIdescPV, (acc || kk > 0));
    };
    bool ok = true;
    for (int j = 0; ok && j < min(2, ntiles); ++j) {  // the first S of each row tile
      ok = __all_sync(kFull, wait_or_abort(&kfull[j], 0, abort, p.err));
      if (!ok) break;
      tc_fence_after();
      if (lane == 0) {
        issue_s(j, j);
        umma_commit(&sfull[j]);
        if (j + kStages < ntiles) umma_commit(&kempty[j]);
      }
      __syncwarp();
    }
    for (int j = 0; ok && j < ntiles; ++j) {
      const int tj = j & 1;                                // row tile
      const int s = j % kStages;                           // stage
      const uint32_t u = static_cast<uint32_t>(j / kStages);
      const uint32_t c = static_cast<uint32_t>(j >> 1);    // the row tile's tile count
      ok = __all_sync(kFull, wait_or_abort(&vfull[s], u & 1, abort, p.err));
      if (!ok) break;
      // V rows that hold no key of the tile (stale bytes, maybe NaN) must
      // not meet a zero P: zero them
      unsigned char* vt = smem + kOffK + s * kStageBytes + kOpBytes;
      if (j < nts) {
        const int k0 = kbase + j * kKeys;
        if (k0 + kKeys > ctx) {  // rows at or past the shared positions
          const int first = ctx - k0;
          for (int idx = lane; idx < (kKeys - first) * 16; idx += 32)
            *reinterpret_cast<uint4*>(vt + kv_chunk_offset(first + (idx >> 4), idx & 15)) =
                make_uint4(0u, 0u, 0u, 0u);
          fence_proxy_async_smem();
          __syncwarp();
        }
      } else {  // own slots past their member's own positions, or past the members
        for (int r = lane; r < kKeys; r += 32) {
          const int slot = (j - nts) * kKeys + r;
          const int k = slot / p.own_slots, o = slot - k * p.own_slots;
          if (k >= members_here || o >= own_len[k]) {
#pragma unroll
            for (int c = 0; c < 16; ++c)
              *reinterpret_cast<uint4*>(vt + kv_chunk_offset(r, c)) = make_uint4(0u, 0u, 0u, 0u);
          }
        }
        fence_proxy_async_smem();
        __syncwarp();
      }
      const bool more = j + 2 < ntiles;  // this row tile has another tile
      ok = __all_sync(kFull, wait_or_abort(&pfull[tj], c & 1, abort, p.err));
      if (ok && more)
        ok = __all_sync(kFull, wait_or_abort(&kfull[(j + 2) % kStages],
                                             static_cast<uint32_t>((j + 2) / kStages) & 1, abort,
                                             p.err));
      if (!ok) break;
      tc_fence_after();
      if (lane == 0) {
        issue_pv(tj, j, c > 0);
        if (j + kStages < ntiles) umma_commit(&vempty[s]);  // the producer reuses the stage
        if (more) {
          issue_s(tj, j + 2);
          umma_commit(&sfull[tj]);
          if (j + 2 + kStages < ntiles) umma_commit(&kempty[(j + 2) % kStages]);
        } else {
          umma_commit(&ofull[tj]);
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
  // Fused ending (one chunk per group, own positions included): the two
  // halves of every row meet in shared memory (the K/V stages: every copy
  // has landed and every product has completed) and the row's output is
  //   M = max(m_0, m_1),  w_t = l_t 2^(m_t - M),  o = (w_0 o_0 + w_1 o_1) / (w_0 + w_1)
  // with o_t the half's normalised O.  An abort leaves the output unwritten.
  const bool finish = fused && *abort == 0;  // uniform: nothing sets abort past the barrier
  float* xo = reinterpret_cast<float*>(smem + kOffK);  // [2][kRowTile][kPrefixRecStride]
  if (finish) {
    if (fin_ok) {  // a softmax warp that ran (uniform over the warp)
      tc_fence_after();
      const uint32_t o_tm = tmem + (static_cast<uint32_t>((warp & 3) * 32) << 16) + 256 + t * 128;
      const float inv = fin_l > 0.f ? 1.f / fin_l : 0.f;
      float* dst = xo + (t * kRowTile + row_of()) * kPrefixRecStride;
      const bool own = owns();
#pragma unroll
      for (int c0 = 0; c0 < kHeadDim; c0 += 32) {
        uint32_t w[32];
        tmem_ld32(w, o_tm + c0);
        tmem_wait_ld(w);
        if (own) {
#pragma unroll
          for (int q = 0; q < 8; ++q)
            reinterpret_cast<float4*>(dst + c0)[q] =
                make_float4(__uint_as_float(w[4 * q]) * inv, __uint_as_float(w[4 * q + 1]) * inv,
                            __uint_as_float(w[4 * q + 2]) * inv,
                            __uint_as_float(w[4 * q + 3]) * inv);
        }
      }
      if (own) {
        dst[128] = fin_m;
        dst[129] = fin_l;
      }
    }
    tc_fence_before();
    __syncthreads();
  }
  if (warp == 9) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                 "r"(kTmemCols)
                 : "memory");
  }
  if (finish) {
    for (int r = warp; r < rows_here; r += kThreads / 32) {  // a warp per row, 4 dims a lane
      const float* h0 = xo + r * kPrefixRecStride;
      const float* h1 = xo + (kRowTile + r) * kPrefixRecStride;
      const float l0 = h0[129], l1 = two ? h1[129] : 0.f;
      const float m0 = l0 > 0.f ? h0[128] : -INFINITY, m1 = l1 > 0.f ? h1[128] : -INFINITY;
      const float M = fmaxf(m0, m1);
      const float w0 = l0 > 0.f ? l0 * fast_exp2(m0 - M) : 0.f;
      const float w1 = l1 > 0.f ? l1 * fast_exp2(m1 - M) : 0.f;
      const float W = w0 + w1;
      const float inv = W > 0.f ? 1.f / W : 0.f;
      float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
      if (w0 > 0.f) {
        const float4 a = reinterpret_cast<const float4*>(h0)[lane];
        o = make_float4(a.x * w0, a.y * w0, a.z * w0, a.w * w0);
      }
      if (w1 > 0.f) {
        const float4 b = reinterpret_cast<const float4*>(h1)[lane];
        o = make_float4(fmaf(b.x, w1, o.x), fmaf(b.y, w1, o.y), fmaf(b.z, w1, o.z),
                        fmaf(b.w, w1, o.w));
      }
      const int rr = row0 + r;
      const int64_t orow = (static_cast<int64_t>(seq) + rr / G) * p.Hq + kvh * G + rr % G;
      const uint32_t lo16 = f32_to_bf16_bits(o.x * inv) | (uint32_t(f32_to_bf16_bits(o.y * inv)) << 16);
      const uint32_t hi16 = f32_to_bf16_bits(o.z * inv) | (uint32_t(f32_to_bf16_bits(o.w * inv)) << 16);
      *reinterpret_cast<uint2*>(p.out + orow * kHeadDim + lane * 4) = make_uint2(lo16, hi16);
    }
  }
}

cudaError_t launch_prefix(const CUtensorMap& tk, const CUtensorMap& tv, const PrefixParams& p,
                          cudaStream_t stream) {
  static bool attr_done = false;  // one device per process in practice; repeated calls are harmless
  if (!attr_done) {
    const cudaError_t e = cudaFuncSetAttribute(
        prefix_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    if (e != cudaSuccess) return e;
    attr_done = true;
  }
  const int row_blocks = (p.rows + kRowTile - 1) / kRowTile;
  return launch_pdl(prefix_kernel, dim3(row_blocks, p.Hkv, p.num_groups * p.chunks),
                    dim3(kThreads), kSmemBytes, stream, tk, tv, p);
}

}  // namespace pkv
