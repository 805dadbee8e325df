// decode_launch.cuh -- host-side launch of the decode kernels for one layout,
// dispatching on the GQA group size G = Hq / Hkv (1..8).
#pragma once

#include "decode_attention.cuh"

namespace pkv {

constexpr int kDecodeStages = 3;  // per-warp ring depth (3 x 8 KiB per warp)

// Dynamic shared memory of the main kernel for group size g.
int decode_smem_bytes(int g);

// Sets the kernel's dynamic shared-memory limit once per device.
template <typename Kernel>
cudaError_t ensure_smem_limit(Kernel kernel, int bytes, unsigned long long* done_mask) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const unsigned long long bit = 1ull << (dev & 63);
  if (__atomic_load_n(done_mask, __ATOMIC_ACQUIRE) & bit) return cudaSuccess;
  e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess) __atomic_fetch_or(done_mask, bit, __ATOMIC_ACQ_REL);
  return e;
}

template <int G, bool kContig>
cudaError_t launch_decode_group(const DecodeParams& p, cudaStream_t stream) {
  using L = DecodeSmemLayout<G, kDecodeStages>;
  static unsigned long long done_mask = 0;
  auto kernel = decode_attention_kernel<G, kContig, kDecodeStages>;
  cudaError_t e = ensure_smem_limit(kernel, L::kTotal, &done_mask);
  if (e != cudaSuccess) return e;
  const dim3 grid(p.nsplit, p.Hkv, p.num_seqs);
  e = launch_pdl(kernel, grid, dim3(kDecodeThreads), L::kTotal, stream, p);
  if (e != cudaSuccess || p.nsplit == 1) return e;
  const int64_t rows = static_cast<int64_t>(p.num_seqs) * p.Hq;
  return launch_pdl(decode_combine_kernel<kContig>, dim3(static_cast<unsigned>((rows + 3) / 4)),
                    dim3(128), 0, stream, p);
}

template <bool kContig>
cudaError_t launch_decode(const DecodeParams& p, int group, cudaStream_t stream) {
  switch (group) {
    case 1: return launch_decode_group<1, kContig>(p, stream);
    case 2: return launch_decode_group<2, kContig>(p, stream);
    case 3: return launch_decode_group<3, kContig>(p, stream);
    case 4: return launch_decode_group<4, kContig>(p, stream);
    case 5: return launch_decode_group<5, kContig>(p, stream);
    case 6: return launch_decode_group<6, kContig>(p, stream);
    case 7: return launch_decode_group<7, kContig>(p, stream);
    case 8: return launch_decode_group<8, kContig>(p, stream);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_decode_paged(const DecodeParams& p, int group, cudaStream_t stream);
cudaError_t launch_decode_contig(const DecodeParams& p, int group, cudaStream_t stream);

}  // namespace pkv
