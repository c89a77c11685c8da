// decode_bf16.cu -- decode kernels instantiated for bf16 caches.
#include "decode_kernels.cuh"

namespace pa {

int decode_ctas_per_sm_bf16(int head_size, int block_size, DecodeKind kind) {
  return decode_ctas_per_sm_dispatch<__nv_bfloat16, __nv_bfloat16>(head_size, block_size, kind);
}

cudaError_t launch_decode_bf16(int head_size, int block_size, const DecodeParams& p, DecodeKind kind, int grid,
                              cudaStream_t s, int* n) {
  return launch_decode_dispatch<__nv_bfloat16, __nv_bfloat16>(head_size, block_size, p, kind, grid, s, n);
}

}  // namespace pa
