// prefill.cu -- causal prefill attention over a paged KV cache (sm_103a).
//
// Sequence i's chunk of Lq new tokens (rows cu_q[i] .. cu_q[i+1]-1 of q, whose
// K and V rows are already in the cache) holds the last Lq of its ctx
// positions; new token j, at position ctx - Lq + j, attends positions
// 0 .. ctx - Lq + j ("Running Out of Cache": a block table maps positions to
// blocks; a chunk of one token is the decode step).
//
// Work: one CTA of 4 warps per (64 query rows, KV head, sequence).  The rows
// are the chunk's (token, query head) pairs of the KV head's group, token
// major (row r: token r / G, head r % G), so every K/V tile serves the whole
// group; warp w owns rows 16w .. 16w+15.  Keys come in tiles of 64 positions
// (four 16-position runs, each inside one block) through the TMA engine --
// 2-D tensor maps over the cache rows, 128-byte swizzled boxes of 16 rows x
// 64 columns -- into a 3-stage ring shared by the CTA.
//
// Math per warp and key tile, on tensor cores (mma.m16n8k16, bf16 in, fp32
// accumulate): S = Q K^T (16 x 64: 8 n-tiles x 8 k-steps; K from ldmatrix),
// causal mask, online softmax in base 2, then O += P V with P taken straight
// from the S accumulators as the A operand and V^T from ldmatrix.trans.  V
// rows at or past the context are zeroed in shared memory first, so stale
// bytes never reach P V.
#include "pkv_device.cuh"
#include "prefill.cuh"

namespace pkv {

namespace {

constexpr int kPfWarps = 4;
constexpr int kPfRows = 16 * kPfWarps;     // query rows per CTA
constexpr int kPfKeys = 64;                // keys per tile
constexpr int kPfStages = 3;
constexpr int kPfStageBytes = 2 * kPfKeys * kRowBytes;  // K then V: 32 KiB
constexpr int kPfBox = 2048;               // 16 rows x 128 B
constexpr int kPfSmem = kPfStages * kPfStageBytes + kPfStages * 8 + 1024;

}  // namespace

__global__ void __launch_bounds__(kPfWarps * 32, 2)
    prefill_kernel(const __grid_constant__ CUtensorMap tmk,
                   const __grid_constant__ CUtensorMap tmv, const PrefillParams p) {
  constexpr unsigned kFull = 0xffffffffu;
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem = smem_raw + ((1024 - (smem_addr(smem_raw) & 1023)) & 1023);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kPfStages * kPfStageBytes);
  __shared__ int32_t s_entry[kPfStages][kPfKeys / 16];

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const int g = lane >> 2;
  const int tq = lane & 3;
  const int i = blockIdx.z;
  const int kvh = blockIdx.y;
  const int rt = gridDim.x - 1 - blockIdx.x;  // latest (heaviest) rows first
  const int G = p.G;

  if (tid == 0) {
    for (int s = 0; s < kPfStages; ++s) mbar_init(&bars[s], 1);
    fence_barrier_init();
    prefetch_tensormap(&tmk);
    prefetch_tensormap(&tmv);
  }
  grid_dependency_wait();
  grid_dependency_trigger();

  const int q0 = p.cu_q[i];
  const int Lq = p.cu_q[i + 1] - q0;
  int ctx = p.ctx_lens[i];
  if (p.checked) {
    const int64_t cap = static_cast<int64_t>(p.max_blocks) * p.bs;
    if (Lq < 0 || Lq > p.max_q || ctx < Lq || ctx > cap) {
      if (tid == 0 && blockIdx.x == 0 && kvh == 0) record_error(p.err, kErrContext);
      return;
    }
  }
  const int rows = Lq * G;
  const int row0 = rt * kPfRows;
  if (row0 >= rows) return;  // this CTA's rows lie past the chunk (uniform)
  const int base = ctx - Lq;  // position of the chunk's first token
  // keys this CTA needs: up to the position of its last valid row
  const int last_row = min(row0 + kPfRows, rows) - 1;
  const int kend = base + last_row / G + 1;
  const int ntiles = (kend + kPfKeys - 1) / kPfKeys;

  const uint64_t policy = l2_policy_evict_first();
  __syncthreads();

  // ---- producer (thread 0): tile t into stage t % kPfStages
  auto issue = [&](int t) {
    const int stage = t % kPfStages;
    unsigned char* st = smem + stage * kPfStageBytes;
    if (lane < kPfKeys / 16) {  // warp 0: block-table entries of the 4 runs
      const int pos = t * kPfKeys + lane * 16;
      int32_t e = 0;
      if (pos < ctx) {
        e = p.block_tables[static_cast<int64_t>(i) * p.max_blocks + pos / p.bs];
        if (p.checked && (e < 0 || e >= p.num_blocks)) {
          record_error(p.err, kErrBlockId);
          e = -1;  // skip the copy: stale rows, undefined output, no fault
        }
      } else {
        e = -1;
      }
      s_entry[stage][lane] = e;
    }
    __syncwarp();
    if (lane == 0) {
      uint32_t bytes = 0;
      for (int r = 0; r < kPfKeys / 16; ++r)
        if (s_entry[stage][r] >= 0) bytes += 4 * kPfBox;
      mbar_arrive_expect_tx(&bars[stage], bytes);
      for (int r = 0; r < kPfKeys / 16; ++r) {
        const int32_t e = s_entry[stage][r];
        if (e < 0) continue;
        const int pos = t * kPfKeys + r * 16;
        const int32_t y = static_cast<int32_t>(cache_row(e, kvh, p.Hkv, p.bs, pos % p.bs));
        unsigned char* kd = st + r * 2 * kPfBox;
        unsigned char* vd = st + kPfKeys * kRowBytes + r * 2 * kPfBox;
        tma_load_2d(kd, &tmk, 0, y, &bars[stage], policy);
        tma_load_2d(kd + kPfBox, &tmk, 64, y, &bars[stage], policy);
        tma_load_2d(vd, &tmv, 0, y, &bars[stage], policy);
        tma_load_2d(vd + kPfBox, &tmv, 64, y, &bars[stage], policy);
      }
    }
  };
  int issued = 0;  // tiles issued so far (tracked by warp 0)
  if (warp == 0)
    for (; issued < kPfStages && issued < ntiles; ++issued) issue(issued);

  // ---- this warp's 16 query rows: A fragments of Q for the 8 k-steps
  const int ra = row0 + warp * 16 + g;  // rows g and g + 8 of the warp
  const int rb = ra + 8;
  const bool va = ra < rows, vb = rb < rows;
  const int pa = va ? base + ra / G : -1;  // query positions (-1: padding row)
  const int pb = vb ? base + rb / G : -1;
  uint32_t qa[8][4];
  {
    const uint32_t* qra = reinterpret_cast<const uint32_t*>(
        p.q + (static_cast<int64_t>(q0 + (va ? ra / G : 0)) * p.Hq + kvh * G + (va ? ra % G : 0)) *
                  kHeadDim);
    const uint32_t* qrb = reinterpret_cast<const uint32_t*>(
        p.q + (static_cast<int64_t>(q0 + (vb ? rb / G : 0)) * p.Hq + kvh * G + (vb ? rb % G : 0)) *
                  kHeadDim);
#pragma unroll
    for (int ks = 0; ks < 8; ++ks) {
      qa[ks][0] = va ? __ldg(qra + ks * 8 + tq) : 0u;
      qa[ks][1] = vb ? __ldg(qrb + ks * 8 + tq) : 0u;
      qa[ks][2] = va ? __ldg(qra + ks * 8 + 4 + tq) : 0u;
      qa[ks][3] = vb ? __ldg(qrb + ks * 8 + 4 + tq) : 0u;
    }
  }

  // per-lane ldmatrix offsets in a 128-byte-swizzled 16 x 128 B box
  // K (B operand, non-transposed): matrices (keys 0-7 | 8-15) x (dims lo | hi)
  const int krow = (lane >> 4) * 8 + (lane & 7);
  const int kchunk = (lane >> 3) & 1;
  // V (B operand via .trans): matrices (keys 0-7 | 8-15) x (dims d | d + 8)
  const int vrow = ((lane >> 3) & 1) * 8 + (lane & 7);
  const int vchunk = lane >> 4;

  float o[16][4];
#pragma unroll
  for (int n = 0; n < 16; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;
  float ma = -INFINITY, mb = -INFINITY, la = 0.f, lb = 0.f;
  bool dead = false;
  int consumed = 0;

  for (int t = 0; t < ntiles; ++t) {
    consumed = t;
    const int stage = t % kPfStages;
    if (!__all_sync(kFull, mbar_wait_bounded(&bars[stage], static_cast<uint32_t>(t / kPfStages) & 1u))) {
      dead = true;
      if (lane == 0) record_error(p.err, kErrTimeout);
    }
    dead = __syncthreads_or(dead);
    if (dead) break;
    unsigned char* st = smem + stage * kPfStageBytes;
    const int k0 = t * kPfKeys;
    if (k0 + kPfKeys > ctx) {  // zero V rows at or past the context
      unsigned char* vt = st + kPfKeys * kRowBytes;
      for (int idx = tid; idx < kPfKeys * 16; idx += kPfWarps * 32) {
        const int r = idx >> 4;
        if (k0 + r < ctx) continue;
        const int ch = idx & 15;
        *reinterpret_cast<uint4*>(vt + (r >> 4) * 2 * kPfBox + (ch >> 3) * kPfBox + (r & 15) * 128 +
                                  (ch & 7) * 16) = make_uint4(0u, 0u, 0u, 0u);
      }
      __syncthreads();
    }
    const uint32_t kbase = smem_addr(st);
    const uint32_t vbase = kbase + kPfKeys * kRowBytes;

    // ---- S = Q K^T: 16 rows x 64 keys
    float s[8][4];
#pragma unroll
    for (int n = 0; n < 8; ++n) s[n][0] = s[n][1] = s[n][2] = s[n][3] = 0.f;
#pragma unroll
    for (int r = 0; r < 4; ++r) {      // 16-key run r: n-tiles 2r, 2r + 1
#pragma unroll
      for (int ks = 0; ks < 8; ++ks) {
        uint32_t b[4];
        const int c = (ks & 3) * 2 + kchunk;
        ldmatrix_x4(b, kbase + (r * 2 + (ks >> 2)) * kPfBox + krow * 128 + ((c ^ (krow & 7)) << 4));
        mma_bf16_16816(s[2 * r], qa[ks], b[0], b[1]);
        mma_bf16_16816(s[2 * r + 1], qa[ks], b[2], b[3]);
      }
    }
    // ---- causal mask and online softmax (rows g and g + 8)
    float mxa = -INFINITY, mxb = -INFINITY;
#pragma unroll
    for (int n = 0; n < 8; ++n) {
      const int key = k0 + 8 * n + 2 * tq;
      s[n][0] = key <= pa ? s[n][0] * p.qscale : -INFINITY;
      s[n][1] = key + 1 <= pa ? s[n][1] * p.qscale : -INFINITY;
      s[n][2] = key <= pb ? s[n][2] * p.qscale : -INFINITY;
      s[n][3] = key + 1 <= pb ? s[n][3] * p.qscale : -INFINITY;
      mxa = fmaxf(mxa, fmaxf(s[n][0], s[n][1]));
      mxb = fmaxf(mxb, fmaxf(s[n][2], s[n][3]));
    }
#pragma unroll
    for (int off = 1; off < 4; off <<= 1) {
      mxa = fmaxf(mxa, __shfl_xor_sync(kFull, mxa, off));
      mxb = fmaxf(mxb, __shfl_xor_sync(kFull, mxb, off));
    }
    const float na = fmaxf(ma, mxa), nb = fmaxf(mb, mxb);
    const float fa = na == -INFINITY ? 1.f : fast_exp2(ma - na);
    const float fb = nb == -INFINITY ? 1.f : fast_exp2(mb - nb);
    la *= fa;
    lb *= fb;
#pragma unroll
    for (int n = 0; n < 16; ++n) {
      o[n][0] *= fa;
      o[n][1] *= fa;
      o[n][2] *= fb;
      o[n][3] *= fb;
    }
    ma = na;
    mb = nb;
    uint32_t pa_[8], pb_[8];  // P packed to bf16: row g / row g + 8, per n-tile
#pragma unroll
    for (int n = 0; n < 8; ++n) {
      const float e0 = na == -INFINITY ? 0.f : fast_exp2(s[n][0] - na);
      const float e1 = na == -INFINITY ? 0.f : fast_exp2(s[n][1] - na);
      const float e2 = nb == -INFINITY ? 0.f : fast_exp2(s[n][2] - nb);
      const float e3 = nb == -INFINITY ? 0.f : fast_exp2(s[n][3] - nb);
      la += e0 + e1;
      lb += e2 + e3;
      pa_[n] = pack_bf16x2(e0, e1);
      pb_[n] = pack_bf16x2(e2, e3);
    }
    // ---- O += P V: k-step r covers keys 16r .. 16r + 15 (n-tiles 2r, 2r + 1)
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      const uint32_t a[4] = {pa_[2 * r], pb_[2 * r], pa_[2 * r + 1], pb_[2 * r + 1]};
#pragma unroll
      for (int dp = 0; dp < 8; ++dp) {  // dims 16dp .. 16dp + 15: n-tiles 2dp, 2dp + 1
        uint32_t b[4];
        const int c = (dp & 3) * 2 + vchunk;
        ldmatrix_x4_trans(b, vbase + (r * 2 + (dp >> 2)) * kPfBox + vrow * 128 + ((c ^ (vrow & 7)) << 4));
        mma_bf16_16816(o[2 * dp], a, b[0], b[1]);
        mma_bf16_16816(o[2 * dp + 1], a, b[2], b[3]);
      }
    }
    __syncthreads();  // every warp is done with this stage
    if (warp == 0 && t + kPfStages < ntiles) {
      fence_proxy_async_smem();
      issue(t + kPfStages);
      ++issued;
    }
  }

  if (dead) {
    // give the copies still in flight a bounded chance to land before exit
    if (tid == 0)
      for (int k = consumed; k < issued; ++k)
        mbar_wait_bounded(&bars[k % kPfStages], static_cast<uint32_t>(k / kPfStages) & 1u);
    return;
  }
  // ---- normalise and store rows g and g + 8
#pragma unroll
  for (int off = 1; off < 4; off <<= 1) {
    la += __shfl_xor_sync(kFull, la, off);
    lb += __shfl_xor_sync(kFull, lb, off);
  }
  const float ia = la > 0.f ? 1.f / la : 0.f;
  const float ib = lb > 0.f ? 1.f / lb : 0.f;
  uint16_t* oa = p.out + (static_cast<int64_t>(q0 + (va ? ra / G : 0)) * p.Hq + kvh * G + (va ? ra % G : 0)) * kHeadDim;
  uint16_t* ob = p.out + (static_cast<int64_t>(q0 + (vb ? rb / G : 0)) * p.Hq + kvh * G + (vb ? rb % G : 0)) * kHeadDim;
#pragma unroll
  for (int n = 0; n < 16; ++n) {
    const int d = 8 * n + 2 * tq;
    if (va) *reinterpret_cast<uint32_t*>(oa + d) = pack_bf16x2(o[n][0] * ia, o[n][1] * ia);
    if (vb) *reinterpret_cast<uint32_t*>(ob + d) = pack_bf16x2(o[n][2] * ib, o[n][3] * ib);
  }
}

cudaError_t launch_prefill(const CUtensorMap& tk, const CUtensorMap& tv, const PrefillParams& p,
                           cudaStream_t stream) {
  static bool attr_done = false;  // one device per process in practice; repeated calls are harmless
  if (!attr_done) {
    const cudaError_t e =
        cudaFuncSetAttribute(prefill_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kPfSmem);
    if (e != cudaSuccess) return e;
    attr_done = true;
  }
  const int row_tiles = (p.max_q * p.G + kPfRows - 1) / kPfRows;
  return launch_pdl(prefill_kernel, dim3(row_tiles, p.Hkv, p.num_seqs), dim3(kPfWarps * 32),
                    kPfSmem, stream, tk, tv, p);
}

}  // namespace pkv
