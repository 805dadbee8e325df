// decode_contig.cu -- instantiations of the decode kernels for the contiguous
// (request row at reqId x S) layout.
#include "decode_launch.cuh"

namespace pkv {

cudaError_t launch_decode_contig(const DecodeParams& p, int group, cudaStream_t stream) {
  return launch_decode<true>(p, group, stream);
}

int decode_smem_bytes(int g) {
  switch (g) {
    case 1: return DecodeSmemLayout<1, kDecodeStages>::kTotal;
    case 2: return DecodeSmemLayout<2, kDecodeStages>::kTotal;
    case 3: return DecodeSmemLayout<3, kDecodeStages>::kTotal;
    case 4: return DecodeSmemLayout<4, kDecodeStages>::kTotal;
    case 5: return DecodeSmemLayout<5, kDecodeStages>::kTotal;
    case 6: return DecodeSmemLayout<6, kDecodeStages>::kTotal;
    case 7: return DecodeSmemLayout<7, kDecodeStages>::kTotal;
    case 8: return DecodeSmemLayout<8, kDecodeStages>::kTotal;
    default: return 0;
  }
}

}  // namespace pkv
