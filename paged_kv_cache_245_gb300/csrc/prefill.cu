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
// Work items: (two row tiles, KV head, sequence).  The rows are the chunk's
// (token, query head) pairs of the KV head's group, token major (row r: token
// r / G, head r % G), so every K/V tile serves the whole group.  A row tile
// is the M = 128 of one tcgen05.mma and holds TR = (128 / G) G rows, whole
// tokens (128, or 126 / 125 when G does not divide 128; the rest is zero
// padding), so that its Q rows are TMA boxes of whole tokens; each row tile
// has its own softmax warpgroup.  The grid is persistent, one CTA per SM, and each CTA
// walks a fixed list of items: heaviest (latest rows) first, dealt to the
// CTAs in rounds whose direction alternates, which balances the CTAs about as
// well as a dynamic queue would (no shared counter, nothing to reset).  The
// roles run ahead of one another across item boundaries, so the next item's
// Q rows, table entries and first K/V tiles load during the current item:
//
//   warps 0-3  softmax and output of row tile 0   warps 4-7  of row tile 1
//   warp 8     the K/V tiles of 128 keys by TMA into a 2-stage ring: one box per run
//              of a block's rows (gcd(bs, 128) rows), landing as 8-row x
//              128-byte swizzled atoms ordered (row group, column half)
//   warp 9     tensor-memory owner and MMA issuer (one thread)
//   warp 10    the item list (descriptors into a 4-slot ring) and the Q rows,
//              by TMA into two rotating 32 KiB slots
//
// Tensor memory (512 columns, lane = query row of the tile): S_t = Q_t K^T in
// columns 128t .. 128t+127, O_t in columns 256 + 128t ..  For key tile j the
// MMA thread issues PV_0(j) S_0(j+1) | PV_1(j) S_1(j+1), where tile j+1 may
// be the next item's first tile, so the tensor cores run one row tile's
// products while the other tile's softmax runs.  The softmax thread of row r
// reads its row of S, masks keys past its position and writes
// P = 2^(S * scale * log2 e - m) as packed bf16 pairs over the first 64
// columns of S in place; PV_t(j) takes P straight from tensor memory (A
// operand) and V from shared memory (MN-major B operand).  The running
// maximum m is updated lazily: O and l are rescaled only when a row's
// maximum grows by more than 8 (a factor 2^8), so P stays below 256 and most
// tiles skip the rescale.  The MMAs of one thread complete in issue order, so
// the barrier that reports S_t(j+1) also reports PV_t(j): from then on the
// softmax warps own O_t until they hand P_t(j+1) over.  An item's first P V
// product overwrites O_t, and is issued only once the same warps have handed
// over that item's first P, after reading the previous item's O_t out.
#include <cudaTypedefs.h>

#include <atomic>
#include <climits>
#include <mutex>

#include "pkv_device.cuh"
#include "prefill.cuh"
#include "umma.cuh"

namespace pkv {

using namespace umma;

namespace {

constexpr int kStages = 2;
constexpr int kQSlots = 2;                            // Q tiles in rotation (a third measured slower)
constexpr int kOffK = kQSlots * kOpBytes;             // after the Q slots
constexpr int kStageBytes = 2 * kOpBytes;             // K then V
constexpr int kOffOut = kOffK + kStages * kStageBytes;  // output staging, 4 KiB per softmax warp
constexpr int kTilesBytes = kOffOut + 8 * 4096;       // 224 KiB
constexpr int kSmemBytes = kTilesBytes + 512 + 1024;  // + barriers and item ring, alignment
static_assert(kSmemBytes <= 232448, "shared memory per CTA exceeds 227 KiB");
constexpr int kThreads = 352;
constexpr int kRing = 4;                              // item descriptors in flight
constexpr int kRingUsers = 10;                        // readers: softmax warps, K/V and MMA warps

// One work item as the scheduling warp (10) publishes it; ntiles == 0 ends
// the list.
struct PItem {
  int32_t seq, kvh, row0, rows, base, ntiles, q0, ctx;
};

// A Q tile's slot in the rotation and the phase of that slot's barriers.
struct QCursor {
  int slot;
  uint32_t phase;
  __device__ QCursor next(int nslots) const {
    QCursor c = *this;
    if (++c.slot == nslots) {
      c.slot = 0;
      c.phase ^= 1u;
    }
    return c;
  }
};

// The mbarriers after the tiles.
struct PBars {
  uint64_t* kfull;      // [2] K of a stage landed
  uint64_t* vfull;      // [2] V of a stage landed
  uint64_t* kempty;     // [2] both S products reading a stage's K completed
  uint64_t* vempty;     // [2] both P V products reading a stage's V completed
  uint64_t* sfull;      // [2] S_t of the next key tile (and PV_t before it) done
  uint64_t* pfull;      // [2] P_t written (one arrival per warp)
  uint64_t* ofull;      // [2] an item's last PV_t completed
  uint64_t* qfull;      // [2] a Q slot written (every lane of warp 10 arrives)
  uint64_t* qempty;     // [2] the last S product reading a Q slot completed
  uint64_t* ifull;      // [4] an item descriptor published
  uint64_t* iempty;     // [4] every reader took its copy
  uint64_t* drain;      // the MMA warp's final wait
};

}  // namespace

__global__ void __launch_bounds__(kThreads, 1)
    prefill_kernel(const __grid_constant__ CUtensorMap tmk,
                   const __grid_constant__ CUtensorMap tmv,
                   const __grid_constant__ CUtensorMap tmq,
                   const __grid_constant__ CUtensorMap tmo, const PrefillParams p) {
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem = smem_raw + ((1024 - (smem_addr(smem_raw) & 1023)) & 1023);
  uint64_t* bar0 = reinterpret_cast<uint64_t*>(smem + kTilesBytes);
  PBars B;
  B.kfull = bar0;
  B.vfull = bar0 + 2;
  B.kempty = bar0 + 4;
  B.vempty = bar0 + 6;
  B.sfull = bar0 + 8;
  B.pfull = bar0 + 10;
  B.ofull = bar0 + 12;
  B.qfull = bar0 + 14;
  B.qempty = B.qfull + kQSlots;
  B.ifull = B.qempty + kQSlots;
  B.iempty = B.ifull + kRing;
  B.drain = B.iempty + kRing;
  constexpr int kNumBars = 15 + 2 * kQSlots + 2 * kRing;
  static_assert(kNumBars * 8 + 8 <= 256, "barriers, tensor-memory address and abort flag");
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bar0 + kNumBars);
  volatile int* abort = reinterpret_cast<volatile int*>(bar0 + kNumBars) + 1;
  PItem* ring = reinterpret_cast<PItem*>(smem + kTilesBytes + 256);  // [kRing]

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const int G = p.G;
  const int TR = p.tile_rows;  // rows of a row tile: whole tokens, (128 / G) G
  auto q_off = [](int slot) { return slot * kOpBytes; };

  grid_dependency_wait();
  grid_dependency_trigger();

  // Read descriptor n of the ring (every lane of the calling warp); false
  // when a wait gave up.  The warp's lane 0 then frees its claim on the slot.
  auto read_item = [&](int n, PItem& it) -> bool {
    const int slot = n & (kRing - 1);
    if (!__all_sync(kFull, wait_or_abort(&B.ifull[slot], (n / kRing) & 1, abort, p.err)))
      return false;
    it = ring[slot];
    __syncwarp();
    if (lane == 0) mbar_arrive(&B.iempty[slot]);
    return true;
  };

  // Setup: barriers (warp 8) and the tensor memory (warp 9).
  if (warp == 8) {
    if (lane == 0) {
      for (int s = 0; s < 2; ++s) {
        mbar_init(&B.kfull[s], 1);
        mbar_init(&B.vfull[s], 1);
        mbar_init(&B.kempty[s], 1);
        mbar_init(&B.vempty[s], 1);
        mbar_init(&B.sfull[s], 1);
        mbar_init(&B.pfull[s], 4);  // one arrival per softmax warp
        mbar_init(&B.ofull[s], 1);
      }
      for (int s = 0; s < kQSlots; ++s) {
        mbar_init(&B.qfull[s], 32);  // every lane of the Q warp
        mbar_init(&B.qempty[s], 1);
      }
      for (int s = 0; s < kRing; ++s) {
        mbar_init(&B.ifull[s], 1);
        mbar_init(&B.iempty[s], kRingUsers);
      }
      mbar_init(B.drain, 1);
      *abort = 0;
      fence_barrier_init();
      prefetch_tensormap(&tmk);
      prefetch_tensormap(&tmv);
      prefetch_tensormap(&tmq);
      if (p.out_tma) prefetch_tensormap(&tmo);
    }
  } else if (warp == 10 && TR < kRowTile) {
    // rows TR .. 127 of every Q slot are padding that no copy writes: zero
    for (int slot = 0; slot < kQSlots; ++slot)
      for (int x = lane; x < (kRowTile - TR) * 16; x += 32)
        *reinterpret_cast<uint4*>(smem + q_off(slot) + q_chunk_offset(TR + (x >> 4), x & 15)) =
            make_uint4(0u, 0u, 0u, 0u);
    fence_proxy_async_smem();
  } else if (warp == 9) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_addr(tmem_slot)),
                 "r"(kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t smem_base = smem_addr(smem);

  if (warp == 8) {
    // ================= K/V producer =================
    // Every row tile of a sequence and KV head reads the same K/V tiles: keep
    // them in L2 for the items after.
    const uint64_t policy = l2_policy_evict_last();
    const int run = p.run_rows;    // rows per box (16 .. 128, divides 128 and bs)
    const int runs = kKeys / run;  // boxes per tile and tensor (<= 8)
    const int prun = lane & 15;    // lanes 0-15 copy K of run prun, lanes 16-31 V
    // block-table entry of run prun of tile j of `it` (-1: past the context or rejected)
    auto entry = [&](const PItem& it, int j) -> int32_t {
      const int kpos = j * kKeys + prun * run;
      int32_t e = -1;
      if (prun < runs && kpos < it.ctx) {
        e = p.block_tables[static_cast<int64_t>(it.seq) * p.max_blocks + kpos / p.bs];
        if (p.checked && (e < 0 || e >= p.num_blocks)) {
          record_error(p.err, kErrBlockId);
          e = -1;  // skip the copy: stale rows, undefined output, no fault
        }
      }
      return e;
    };
    int g = 0;             // tiles (of all items) whose K and V were both issued
    bool kv_half = false;  // tile g has its K issued, not its V
    int nread = 0;
    PItem cur;
    bool ok = read_item(nread++, cur);
    int32_t e = ok && cur.ntiles > 0 ? entry(cur, 0) : -1;  // entries of the next tile to issue
    while (ok && cur.ntiles > 0) {
      PItem nx = cur;
      for (int j = 0; j < cur.ntiles; ++j) {
        const int s = g & 1;
        const uint32_t loaded = __popc(__ballot_sync(kFull, lane < 16 && e >= 0));
        const int off = (j * kKeys + prun * run) % p.bs;
        const int32_t grp =
            e >= 0 ? static_cast<int32_t>(cache_row(e, cur.kvh, p.Hkv, p.bs, off) >> 3) : 0;
        unsigned char* dst = smem + kOffK + s * kStageBytes + prun * run * kRowBytes;
        // K first: its stage frees once both S products of tile g - 2 are done
        if (g >= kStages && !__all_sync(kFull, wait_or_abort(&B.kempty[s], ((g >> 1) - 1) & 1,
                                                             abort, p.err))) {
          ok = false;
          break;
        }
        if (lane == 0) mbar_arrive_expect_tx(&B.kfull[s], loaded * run * kRowBytes);
        __syncwarp();
        if (lane < 16 && e >= 0) tma_load_4d(dst, &tmk, grp, &B.kfull[s], policy);
        // then V, whose stage frees after both P V products of tile g - 2
        if (g >= kStages && !__all_sync(kFull, wait_or_abort(&B.vempty[s], ((g >> 1) - 1) & 1,
                                                             abort, p.err))) {
          kv_half = true;
          ok = false;
          break;
        }
        if (lane == 0) mbar_arrive_expect_tx(&B.vfull[s], loaded * run * kRowBytes);
        __syncwarp();
        if (lane >= 16 && e >= 0) tma_load_4d(dst + kOpBytes, &tmv, grp, &B.vfull[s], policy);
        ++g;
        // the next tile's entries load while this one lands
        if (j + 1 < cur.ntiles) {
          e = entry(cur, j + 1);
        } else {
          ok = read_item(nread++, nx);
          e = ok && nx.ntiles > 0 ? entry(nx, 0) : -1;
        }
      }
      cur = nx;
    }
    if (*abort && lane == 0) {
      // let the copies in flight land before the CTA's shared memory is released
      for (int j = max(0, g - kStages); j < g; ++j) {
        mbar_wait_bounded(&B.kfull[j & 1], (j >> 1) & 1);
        mbar_wait_bounded(&B.vfull[j & 1], (j >> 1) & 1);
      }
      if (kv_half) mbar_wait_bounded(&B.kfull[g & 1], (g >> 1) & 1);
    }
  } else if (warp == 10) {
    // ================= item list and Q rows =================
    // Items in order of index: row tile rt (latest first), then sequence,
    // then KV head.  Round k deals items k P .. k P + P - 1 to the P CTAs,
    // forwards in even rounds and backwards in odd ones.  Q tile n (row tile
    // 0 of an item, then row tile 1 if it has rows) goes to slot n % 2 once
    // the last S product reading tile n - 2 completed.
    const int P = gridDim.x;
    const int R = (p.max_q * G + 2 * TR - 1) / (2 * TR);
    const int per = p.num_seqs * p.Hkv;
    const int total = R * per;
    const uint64_t qpolicy = l2_policy_evict_first();  // every Q row is read once
    int published = 0;
    uint32_t nq = 0;      // Q tiles loaded
    QCursor qc = {0, 0};  // slot of Q tile nq and its phase
    uint32_t last_phase = 0;  // bit s: phase of the last load into slot s
    bool ok = true;
    auto publish = [&](const PItem& it) -> bool {
      const int slot = published & (kRing - 1);
      if (published >= kRing &&
          !__all_sync(kFull, wait_or_abort(&B.iempty[slot], ((published / kRing) - 1) & 1,
                                           abort, p.err)))
        return false;
      if (lane == 0) {
        ring[slot] = it;
        mbar_arrive(&B.ifull[slot]);
      }
      __syncwarp();
      ++published;
      return true;
    };
    for (int k = 0; ok && k * P < total; ++k) {
      const int idx = k * P + ((k & 1) ? P - 1 - static_cast<int>(blockIdx.x) : blockIdx.x);
      if (idx >= total) continue;
      const int rt = R - 1 - idx / per;
      const int rem = idx - (idx / per) * per;
      PItem it;
      it.seq = rem / p.Hkv;
      it.kvh = rem - it.seq * p.Hkv;
      it.q0 = p.cu_q[it.seq];
      const int Lq = p.cu_q[it.seq + 1] - it.q0;
      it.ctx = p.ctx_lens[it.seq];
      if (p.checked) {
        const int64_t cap = static_cast<int64_t>(p.max_blocks) * p.bs;
        if (Lq < 0 || Lq > p.max_q || it.ctx < Lq || it.ctx > cap) {
          if (lane == 0 && rt == 0 && it.kvh == 0) record_error(p.err, kErrContext);
          continue;  // the sequence is left unwritten
        }
      }
      it.rows = Lq * G;
      it.row0 = rt * 2 * TR;
      if (it.row0 >= it.rows) continue;  // this item's rows lie past the chunk
      it.base = it.ctx - Lq;             // position of the chunk's first token
      const int last_row = min(it.row0 + 2 * TR, it.rows) - 1;
      const int kend = it.base + last_row / G + 1;  // keys the item needs
      if (kend <= 0) continue;  // only when ctx < Lq (caught in checked mode)
      it.ntiles = (kend + kKeys - 1) / kKeys;
      if (!publish(it)) {
        ok = false;
        break;
      }
      const int nt = it.rows > it.row0 + TR ? 2 : 1;
      for (int t = 0; t < nt; ++t, ++nq, qc = qc.next(kQSlots)) {
        const int qs = qc.slot;
        if (nq >= static_cast<uint32_t>(kQSlots) &&
            !__all_sync(kFull, wait_or_abort(&B.qempty[qs], qc.phase ^ 1u, abort, p.err))) {
          ok = false;
          break;
        }
        last_phase = (last_phase & ~(1u << qs)) | (qc.phase << qs);
        unsigned char* dst = smem + q_off(qs);
        // the tile is TR / G whole tokens, each column half one box of
        // (tokens, G heads, 64 columns); rows past the chunk bring the next
        // tokens' rows (or zeros past the tensor) and are never written out
        const int tok0 = it.q0 + (it.row0 + t * TR) / G;
        if (lane == 0) {
          // two column halves of TR rows x 128 bytes
          mbar_arrive_expect_tx(&B.qfull[qs], static_cast<uint32_t>(TR) * kRowBytes);
          tma_load_4d_at(dst, &tmq, 0, 0, it.kvh * G, tok0, &B.qfull[qs], qpolicy);
          tma_load_4d_at(dst + kHalfBytes, &tmq, 0, 1, it.kvh * G, tok0, &B.qfull[qs], qpolicy);
        } else {
          mbar_arrive(&B.qfull[qs]);
        }
      }
    }
    if (ok) {
      PItem end = {};  // ntiles 0: the end of this CTA's list
      publish(end);
    }
    if (*abort && lane == 0) {
      // let the Q copies in flight land before the shared memory is released
      for (int qs = 0; qs < kQSlots && static_cast<uint32_t>(qs) < nq; ++qs)
        mbar_wait_bounded(&B.qfull[qs], (last_phase >> qs) & 1u);
    }
  } else if (warp == 9) {
    // ================= MMA issuer: lane 0 alone =================
    // One thread issues every product, waits on single-lane barrier checks
    // and never votes or reconverges with the other lanes inside the loop.
    if (lane == 0) {
    auto issue_s = [&](int t, int qs, int stage) {  // S_t = Q K^T
      const uint32_t q_addr = smem_base + q_off(qs);
      const uint32_t k_addr = smem_base + kOffK + stage * kStageBytes;
#pragma unroll
      for (int kk = 0; kk < 8; ++kk) {
        const uint32_t koff = (kk & 3) * 32;
        umma_ss(tmem + t * 128, smem_desc(q_addr + (kk >> 2) * kHalfBytes + koff, 16, 1024),
                smem_desc(k_addr + (kk >> 2) * 1024 + koff, 16, 2048), kIdescS, kk > 0);
      }
    };
    auto issue_pv = [&](int t, int stage, bool acc) {  // O_t (+)= P_t V
      const uint32_t v_addr = smem_base + kOffK + stage * kStageBytes + kOpBytes;
#pragma unroll
      for (int kk = 0; kk < 8; ++kk)
        umma_ts(tmem + 256 + t * 128, tmem + t * 128 + kk * 8,
                smem_desc(v_addr + kk * 4096, 1024, 2048), kIdescPV, (acc || kk > 0));
    };
    auto waitb = [&](uint64_t* b, uint32_t parity) -> bool {
      return wait_or_abort(b, parity, abort, p.err);
    };
    auto read_item1 = [&](int n, PItem& it) -> bool {
      const int slot = n & (kRing - 1);
      if (!wait_or_abort(&B.ifull[slot], (n / kRing) & 1, abort, p.err)) return false;
      it = ring[slot];
      mbar_arrive(&B.iempty[slot]);
      return true;
    };
    auto has_two = [TR](const PItem& it) { return it.rows > it.row0 + TR; };
    // S products of an item's first tile, global tile g, its Q tiles at qa, qb
    auto first_s = [&](const PItem& it, QCursor qa, QCursor qb, int g) -> bool {
      if (!waitb(&B.kfull[g & 1], (g >> 1) & 1) || !waitb(&B.qfull[qa.slot], qa.phase))
        return false;
      tc_fence_after();
      {
        issue_s(0, qa.slot, g & 1);
        umma_commit(&B.sfull[0]);
        if (it.ntiles == 1) umma_commit(&B.qempty[qa.slot]);
      }
      if (has_two(it)) {
        if (!waitb(&B.qfull[qb.slot], qb.phase)) return false;
        tc_fence_after();
        {
          issue_s(1, qb.slot, g & 1);
          umma_commit(&B.sfull[1]);
          if (it.ntiles == 1) umma_commit(&B.qempty[qb.slot]);
        }
      }
      umma_commit(&B.kempty[g & 1]);  // both S products of tile g issued
      return true;
    };
    int nread = 0;
    PItem cur;
    bool ok = read_item1(nread++, cur);
    QCursor q0 = {0, 0};        // cur's Q tiles: row tile 0 at q0, row tile 1 at q1
    QCursor q1 = q0.next(kQSlots);
    int g = 0;                  // tile index over all items (ring stage g & 1)
    uint32_t np0 = 0, np1 = 0;  // P hand-overs taken per row tile
    if (ok && cur.ntiles > 0) ok = first_s(cur, q0, q1, g);
    // Tile g, (cur, j): within an item PV_0(j) S_0(j+1) | PV_1(j) S_1(j+1);
    // at an item's last tile both P V products go first, then the next
    // item's first S products, so the current item never waits on the next.
    int j = 0;
    while (ok && cur.ntiles > 0) {
      const int s = g & 1;
      const bool two = has_two(cur);
      const bool last = j == cur.ntiles - 1;
      const bool qlast = j + 1 == cur.ntiles - 1;  // S of tile j + 1 reads cur's Q last
      ok = waitb(&B.vfull[s], (g >> 1) & 1);
      if (!ok) break;
      const int k0 = j * kKeys;
      if (k0 + kKeys > cur.ctx) {  // zero V rows at or past the context (0 x stale bytes)
        unsigned char* vt = smem + kOffK + s * kStageBytes + kOpBytes;
        const int first = cur.ctx - k0;
        for (int idx = 0; idx < (kKeys - first) * 16; ++idx)
          *reinterpret_cast<uint4*>(vt + kv_chunk_offset(first + (idx >> 4), idx & 15)) =
              make_uint4(0u, 0u, 0u, 0u);
        fence_proxy_async_smem();
      }
      ok = waitb(&B.pfull[0], np0 & 1);
      ++np0;
      if (ok && !last) ok = waitb(&B.kfull[s ^ 1], ((g + 1) >> 1) & 1);
      if (!ok) break;
      tc_fence_after();
      {
        issue_pv(0, s, j > 0);
        if (last) umma_commit(&B.ofull[0]);
        if (!two) umma_commit(&B.vempty[s]);
        if (!last) {
          issue_s(0, q0.slot, s ^ 1);
          umma_commit(&B.sfull[0]);
          if (qlast) umma_commit(&B.qempty[q0.slot]);
          if (!two) umma_commit(&B.kempty[s ^ 1]);
        }
      }
      if (two) {
        ok = waitb(&B.pfull[1], np1 & 1);
        ++np1;
        if (!ok) break;
        tc_fence_after();
        {
          issue_pv(1, s, j > 0);
          if (last) umma_commit(&B.ofull[1]);
          umma_commit(&B.vempty[s]);  // the producer reuses the stage
          if (!last) {
            issue_s(1, q1.slot, s ^ 1);
            umma_commit(&B.sfull[1]);
            if (qlast) umma_commit(&B.qempty[q1.slot]);
            umma_commit(&B.kempty[s ^ 1]);
          }
        }
      }
      ++g;
      if (last) {
        PItem nx;
        ok = read_item1(nread++, nx);
        if (!ok) break;
        q0 = two ? q1.next(kQSlots) : q1;  // the next item's Q tiles follow cur's
        q1 = q0.next(kQSlots);
        cur = nx;
        j = 0;
        if (cur.ntiles > 0) ok = first_s(cur, q0, q1, g);
      } else {
        ++j;
      }
    }
      // every MMA issued has completed before the tensor memory is released
      umma_commit(B.drain);
      mbar_wait_bounded(B.drain, 0);
    }
    __syncwarp();
  } else {
    // ================= softmax warpgroups (warps 0-7) =================
    const int t = warp >> 2;                      // row tile
    const int lr = tid & (kRowTile - 1);          // row in the tile = tensor-memory lane
    const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t s_tm = tmem + lane_base + t * 128;
    const uint32_t o_tm = tmem + lane_base + 256 + t * 128;
    const float sc = p.qscale;
    uint32_t ns = 0, no = 0;  // S tiles and items this row tile took
    bool ok = true;
    for (int n = 0; ok; ++n) {
      PItem it;
      if (!read_item(n, it) || it.ntiles == 0) break;
      if (t == 1 && it.rows <= it.row0 + TR) continue;  // row tile 1 holds no rows
      const int r = it.row0 + t * TR + lr;  // row of the chunk
      const bool valid = lr < TR && r < it.rows;
      const int rr = valid ? r : it.rows - 1;     // padding rows mirror the last row
      const int tok = rr / G;
      const int head = it.kvh * G + rr % G;
      const int pos = it.base + tok;
      const int64_t qrow = (static_cast<int64_t>(it.q0) + tok) * p.Hq + head;
      float m_used = -INFINITY;  // the maximum P is taken against (scaled logits)
      float l = 0.f;
      for (int j = 0; j < it.ntiles; ++j) {
        ok = __all_sync(kFull, wait_or_abort(&B.sfull[t], ns & 1, abort, p.err));
        ++ns;
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
          // (not unrolled: the masked path runs once per item, and a smaller kernel
          // measured faster)
#pragma unroll 1
          for (int h = 0; h < 2; ++h) {
            // a half whose keys no row of the warp sees adds nothing to the maximum
            if (!__any_sync(kFull, !diag || k0 + 64 * h <= pos)) continue;
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
          // (not unrolled: the masked path runs once per item, and a smaller kernel
          // measured faster)
#pragma unroll 1
          for (int h = 0; h < 2; ++h) {
            if (!__any_sync(kFull, !diag || k0 + 64 * h <= pos)) {
              // no row of the warp sees a key of this half: its P is zero
              uint32_t pz[32];
#pragma unroll
              for (int c = 0; c < 32; ++c) pz[c] = 0u;
              tmem_st32(s_tm + 32 * h, pz);
              continue;
            }
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
        if (lane == 0) mbar_arrive(&B.pfull[t]);
      }
      if (!ok) break;
      ok = __all_sync(kFull, wait_or_abort(&B.ofull[t], no & 1, abort, p.err));
      ++no;
      if (!ok) break;
      // the item's output rows; the next item's first P V product overwrites
      // O_t only after these warps hand over its first P
      tc_fence_after();
      const float inv = l > 0.f ? 1.f / l : 0.f;
      const int wrow0 = it.row0 + t * TR + 32 * (warp & 3);  // this warp's first row
      if (p.out_tma && 32 * (warp & 3) + 32 <= TR && wrow0 + 32 <= it.rows) {
        // G divides 32: the warp's 32 rows are 32 / G whole tokens.  Each
        // column half goes through the warp's 4 KiB of staging (row = lane,
        // 128-byte swizzled) and one tensor store.
        unsigned char* stg = smem + kOffOut + warp * 4096;
        const int tokw = it.q0 + wrow0 / G;
        // the row's 128 columns in one tensor-memory round trip
        uint32_t wa[32], wb[32], wc[32], wd[32];
        tmem_ld32(wa, o_tm);
        tmem_ld32(wb, o_tm + 32);
        tmem_ld32(wc, o_tm + 64);
        tmem_ld32(wd, o_tm + 96);
        tmem_wait_ld(wa);
        tmem_ready(wb);
        tmem_ready(wc);
        tmem_ready(wd);
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const uint32_t* w = h == 0 ? wa : wc;
          const uint32_t* w2 = h == 0 ? wb : wd;
          if (lane == 0) bulk_wait_read();  // the warp's last store has read the staging
          __syncwarp();
#pragma unroll
          for (int c = 0; c < 8; ++c) {
            const uint32_t* x = c < 4 ? w + 8 * c : w2 + 8 * (c - 4);
            uint4 o;
            o.x = pack_bf16x2(__uint_as_float(x[0]) * inv, __uint_as_float(x[1]) * inv);
            o.y = pack_bf16x2(__uint_as_float(x[2]) * inv, __uint_as_float(x[3]) * inv);
            o.z = pack_bf16x2(__uint_as_float(x[4]) * inv, __uint_as_float(x[5]) * inv);
            o.w = pack_bf16x2(__uint_as_float(x[6]) * inv, __uint_as_float(x[7]) * inv);
            *reinterpret_cast<uint4*>(stg + lane * 128 + ((c ^ (lane & 7)) << 4)) = o;
          }
          fence_proxy_async_smem();  // the tensor store reads the staging through the async proxy
          __syncwarp();
          if (lane == 0) {
            tma_store_4d_at(&tmo, stg, 0, h, it.kvh * G, tokw);
            bulk_commit();
          }
        }
      } else {
        uint4* dst = reinterpret_cast<uint4*>(p.out + qrow * kHeadDim);
#pragma unroll 1
        for (int c0 = 0; c0 < kHeadDim; c0 += 32) {
          uint32_t w[32];
          tmem_ld32(w, o_tm + c0);
          tmem_wait_ld(w);
          if (valid) {
            uint4 o[4];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              o[q].x = pack_bf16x2(__uint_as_float(w[8 * q + 0]) * inv, __uint_as_float(w[8 * q + 1]) * inv);
              o[q].y = pack_bf16x2(__uint_as_float(w[8 * q + 2]) * inv, __uint_as_float(w[8 * q + 3]) * inv);
              o[q].z = pack_bf16x2(__uint_as_float(w[8 * q + 4]) * inv, __uint_as_float(w[8 * q + 5]) * inv);
              o[q].w = pack_bf16x2(__uint_as_float(w[8 * q + 6]) * inv, __uint_as_float(w[8 * q + 7]) * inv);
            }
            if (p.out_v8) {  // out 32-byte aligned: whole 32-byte sectors
              st_global_v8(dst + c0 / 8, o[0], o[1]);
              st_global_v8(dst + c0 / 8 + 2, o[2], o[3]);
            } else {
#pragma unroll
              for (int q = 0; q < 4; ++q) dst[c0 / 8 + q] = o[q];
            }
          }
        }
      }
      tc_fence_before();
    }
    if (lane == 0) bulk_wait_done();  // the warp's tensor stores completed
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

bool encode_prefill_rows(CUtensorMap* map, const void* base, int64_t num_tokens, int Hq, int G,
                         int box_rows) {
  auto enc = prefill_map_encoder();
  if (enc == nullptr || G <= 0 || box_rows % G != 0 || box_rows > 128 || box_rows / G > 256 ||
      Hq < G || num_tokens <= 0)
    return false;
  const cuuint64_t dims[4] = {64u, 2u, static_cast<cuuint64_t>(Hq),
                              static_cast<cuuint64_t>(num_tokens)};
  const cuuint64_t strides[3] = {128u, static_cast<cuuint64_t>(kRowBytes),
                                 static_cast<cuuint64_t>(Hq) * kRowBytes};
  const cuuint32_t box[4] = {64u, 1u, static_cast<cuuint32_t>(G),
                            static_cast<cuuint32_t>(box_rows / G)};
  const cuuint32_t estr[4] = {1u, 1u, 1u, 1u};
  const CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims,
                         strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                         CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

cudaError_t launch_prefill(const CUtensorMap& tk, const CUtensorMap& tv, const CUtensorMap& tq,
                           const CUtensorMap& to, const PrefillParams& p, cudaStream_t stream) {
  static std::atomic<bool> attr_done{false};  // repeated calls are harmless
  if (!attr_done.load()) {
    const cudaError_t e = cudaFuncSetAttribute(
        prefill_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    if (e != cudaSuccess) return e;
    attr_done.store(true);
  }
  // one CTA per SM (the shared memory admits no second), never more than items
  static std::atomic<int> sms[64];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  int n = dev < 64 ? sms[dev].load() : 0;
  if (n == 0) {
    e = cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    if (dev < 64) sms[dev].store(n);
  }
  if (p.tile_rows <= 0 || p.tile_rows > kRowTile || p.tile_rows % p.G != 0)
    return cudaErrorInvalidValue;
  const int64_t row_tiles =
      (static_cast<int64_t>(p.max_q) * p.G + 2 * p.tile_rows - 1) / (2 * p.tile_rows);
  const int64_t items = row_tiles * p.Hkv * p.num_seqs;
  if (items <= 0) return cudaSuccess;
  if (items > INT32_MAX) return cudaErrorInvalidValue;
  const int grid = static_cast<int>(items < n ? items : n);
  return launch_pdl(prefill_kernel, dim3(grid), dim3(kThreads), kSmemBytes, stream, tk, tv, tq,
                    to, p);
}

}  // namespace pkv
