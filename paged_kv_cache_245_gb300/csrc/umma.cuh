// umma.cuh -- device helpers shared by the tcgen05 attention kernels
// (prefill.cu, prefix.cu): fifth-generation tensor-core MMAs with operands in
// shared or tensor memory, tensor-memory loads and stores, packed fp32 pairs,
// bounded mbarrier waits, and the shared-memory layouts of the Q / K / V
// tiles (8-row x 128-byte atoms, 128-byte swizzled).
#pragma once

#include <cuda.h>
#include <stdint.h>

#include "pkv_device.cuh"

namespace pkv {
namespace umma {

constexpr int kRowTile = 128;              // query rows per tile (MMA M)
constexpr int kKeys = 128;                 // keys per K/V tile
constexpr int kOpBytes = 128 * kRowBytes;  // 32 KiB: a Q, K or V tile
constexpr int kHalfBytes = kOpBytes / 2;   // one 64-column half
constexpr uint32_t kTmemCols = 512;
constexpr unsigned kFull = 0xffffffffu;
constexpr float kRescaleLog2 = 8.f;

// Instruction descriptor of tcgen05.mma.kind::f16: fp32 accumulator (bits
// 4-5), bf16 A and B (7-9, 10-12), N / 8 (17-22), M / 16 (24-28); A K-major;
// B K-major for S = Q K^T, MN-major (bit 16) for O = P V, whose V rows hold
// the N (head) dimension contiguously.
constexpr uint32_t kIdescS = (1u << 4) | (1u << 7) | (1u << 10) | ((128u >> 3) << 17) |
                             ((128u >> 4) << 24);
constexpr uint32_t kIdescPV = kIdescS | (1u << 16);

// Shared-memory matrix descriptor with 128-byte swizzling: start address,
// leading and stride byte offsets (all / 16), the fixed 0b001 at bits 46-48
// and the swizzle mode at 61-63.  Operand tiles hold 8-row x 128-byte atoms.
// Q (written by the softmax threads): column half h at h * 16 KiB, 8-row
// groups 1024 bytes apart.  K and V (TMA): atom (row group g, half h) at
// g * 2048 + h * 1024.  K-major operands (Q, K): stride = the 8-row group
// step, leading offset unused, the k-step's half and 32-byte column offset
// in the start address.  The MN-major V: leading offset = the step between
// the two 64-column halves (1024), stride = 2048 bytes per 8 keys.
__device__ __forceinline__ uint64_t smem_desc(uint32_t addr, uint32_t lbo, uint32_t sbo) {
  return static_cast<uint64_t>((addr & 0x3FFFFu) >> 4) |
         (static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16) |
         (static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32) | (1ull << 46) | (2ull << 61);
}

__device__ __forceinline__ void umma_ss(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc,
                                        uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a), "l"(b), "r"(idesc), "r"(accumulate)
      : "memory");
}

__device__ __forceinline__ void umma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b,
                                        uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Arrive on `bar` once every MMA this thread issued so far has completed.
__device__ __forceinline__ void umma_commit(uint64_t* bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
          smem_addr(bar))
      : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

__device__ __forceinline__ uint64_t l2_policy_evict_last() {
  uint64_t policy;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(policy));
  return policy;
}

#define PKV_R32(F, r)                                                                          \
  F(r[0]), F(r[1]), F(r[2]), F(r[3]), F(r[4]), F(r[5]), F(r[6]), F(r[7]), F(r[8]), F(r[9]),    \
      F(r[10]), F(r[11]), F(r[12]), F(r[13]), F(r[14]), F(r[15]), F(r[16]), F(r[17]),          \
      F(r[18]), F(r[19]), F(r[20]), F(r[21]), F(r[22]), F(r[23]), F(r[24]), F(r[25]),          \
      F(r[26]), F(r[27]), F(r[28]), F(r[29]), F(r[30]), F(r[31])
#define PKV_OUT(x) "=r"(x)
#define PKV_IN(x) "r"(x)
#define PKV_INOUT(x) "+r"(x)
#define PKV_LIST32                                                                             \
  "%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24," \
  "%25,%26,%27,%28,%29,%30,%31"

// 32 consecutive 32-bit columns of this warp's 32 lanes (lane = thread).  The
// registers are valid only after tmem_wait_ld / tmem_ready on them.
__device__ __forceinline__ void tmem_ld32(uint32_t (&r)[32], uint32_t taddr) {
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x32.b32 {" PKV_LIST32 "}, [%32];"
               : PKV_R32(PKV_OUT, r)
               : "r"(taddr));
}

// Wait for this thread's tensor-memory loads; the registers named here (and
// through tmem_ready, any others loaded before the wait) are then valid.
__device__ __forceinline__ void tmem_wait_ld(uint32_t (&r)[32]) {
  asm volatile("tcgen05.wait::ld.sync.aligned;" : PKV_R32(PKV_INOUT, r) : : "memory");
}
__device__ __forceinline__ void tmem_ready(uint32_t (&r)[32]) {
  asm volatile("" : PKV_R32(PKV_INOUT, r) : : "memory");
}

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,"
               "%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,"
               "%31,%32};" ::"r"(taddr),
               PKV_R32(PKV_IN, r)
               : "memory");
}

__device__ __forceinline__ void tmem_wait_st() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// Packed pairs of fp32 (one register pair, lo in the low word) for the
// two-wide fp32 instructions of sm_100 and later.
__device__ __forceinline__ uint64_t f2_pack(uint32_t lo, uint32_t hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "r"(lo), "r"(hi));
  return r;
}
__device__ __forceinline__ void f2_unpack(uint64_t v, float& lo, float& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ uint64_t f2_fma(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t r;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
  return r;
}
__device__ __forceinline__ uint64_t f2_add(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("add.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}

// Wait for phase `parity` of `bar`; give up when another role has given up
// (*abort) or after kWaitLimitNs (then set *abort and record the timeout).
__device__ __forceinline__ bool wait_or_abort(uint64_t* bar, uint32_t parity,
                                              volatile int* abort, int* err) {
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = global_timer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (*abort) return false;
    if (global_timer_ns() - t0 > kWaitLimitNs) {
      *abort = 1;
      record_error(err, kErrTimeout);
      return false;
    }
  }
  return true;
}

// Byte offset of 16-byte chunk c (0..15) of row r in the Q tile: two
// 64-column halves of 128 rows x 128 bytes, 128-byte swizzled.
__device__ __forceinline__ int q_chunk_offset(int r, int c) {
  return (c >> 3) * kHalfBytes + r * 128 + (((c & 7) ^ (r & 7)) << 4);
}

// The same for a K or V tile as the 4-D boxes land: atom (r / 8, c / 8).
__device__ __forceinline__ int kv_chunk_offset(int r, int c) {
  return (r >> 3) * 2048 + (c >> 3) * 1024 + (r & 7) * 128 + (((c & 7) ^ (r & 7)) << 4);
}

__device__ __forceinline__ void tma_load_4d(void* dst_smem, const void* tmap, int32_t group,
                                            uint64_t* bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%2, %3, %4, %5}], [%6], %7;" ::"r"(smem_addr(dst_smem)),
      "l"(tmap), "r"(0), "r"(0), "r"(0), "r"(group), "r"(smem_addr(bar)), "l"(policy)
      : "memory");
}
// The same at coordinates (c0, c1, c2, c3), innermost first.
__device__ __forceinline__ void tma_load_4d_at(void* dst_smem, const void* tmap, int32_t c0,
                                               int32_t c1, int32_t c2, int32_t c3, uint64_t* bar,
                                               uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%2, %3, %4, %5}], [%6], %7;" ::"r"(smem_addr(dst_smem)),
      "l"(tmap), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(smem_addr(bar)), "l"(policy)
      : "memory");
}

// Tensor store from shared memory (box at coordinates c0..c3, innermost
// first) in this thread's bulk group; commit closes the group, and
// wait_read / wait_done wait until every committed group of this thread has
// read its shared memory / completed.
__device__ __forceinline__ void tma_store_4d_at(const void* tmap, const void* src_smem, int32_t c0,
                                                int32_t c1, int32_t c2, int32_t c3) {
  asm volatile(
      "cp.async.bulk.tensor.4d.global.shared::cta.bulk_group [%0, {%2, %3, %4, %5}], [%1];" ::"l"(
          tmap),
      "r"(smem_addr(src_smem)), "r"(c0), "r"(c1), "r"(c2), "r"(c3)
      : "memory");
}
// A 32-byte store (a whole sector) of a then b; the address 32-byte aligned.
__device__ __forceinline__ void st_global_v8(void* dst, const uint4& a, const uint4& b) {
  asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(dst), "r"(a.x),
               "r"(a.y), "r"(a.z), "r"(a.w), "r"(b.x), "r"(b.y), "r"(b.z), "r"(b.w)
               : "memory");
}

__device__ __forceinline__ void bulk_commit() {
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
__device__ __forceinline__ void bulk_wait_read() {
  asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}
__device__ __forceinline__ void bulk_wait_done() {
  asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}


}  // namespace umma
}  // namespace pkv
