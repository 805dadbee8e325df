// decode_paged.cu -- instantiations of the decode kernels for the paged
// (block-table) layout.
#include "decode_launch.cuh"

namespace pkv {

cudaError_t launch_decode_paged(const DecodeParams& p, int group, cudaStream_t stream) {
  return launch_decode<false>(p, group, stream);
}

}  // namespace pkv
