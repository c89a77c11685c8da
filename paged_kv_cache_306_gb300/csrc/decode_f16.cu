// decode_f16.cu -- decode kernels instantiated for f16 caches.
#include "decode_kernels.cuh"

namespace pa {

int decode_ctas_per_sm_f16(int head_size, int block_size, DecodeKind kind) {
  return decode_ctas_per_sm_dispatch<__half, __half>(head_size, block_size, kind);
}

cudaError_t launch_decode_f16(int head_size, int block_size, const DecodeParams& p, DecodeKind kind, int grid,
                              cudaStream_t s, int* n) {
  return launch_decode_dispatch<__half, __half>(head_size, block_size, p, kind, grid, s, n);
}

}  // namespace pa
