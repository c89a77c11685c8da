// decode_fp8.cu -- decode kernels instantiated for FP8 E4M3 caches read by fp16 or bf16 queries.
#include "decode_kernels.cuh"

namespace pa {

int decode_ctas_per_sm_fp8(bool q_is_bf16, int head_size, int block_size, DecodeKind kind) {
  return q_is_bf16 ? decode_ctas_per_sm_dispatch<__nv_bfloat16, __nv_fp8_e4m3>(head_size, block_size, kind)
                   : decode_ctas_per_sm_dispatch<__half, __nv_fp8_e4m3>(head_size, block_size, kind);
}

cudaError_t launch_decode_fp8(bool q_is_bf16, int head_size, int block_size, const DecodeParams& p, DecodeKind kind,
                              int grid, cudaStream_t s, int* n) {
  return q_is_bf16 ? launch_decode_dispatch<__nv_bfloat16, __nv_fp8_e4m3>(head_size, block_size, p, kind, grid, s, n)
                   : launch_decode_dispatch<__half, __nv_fp8_e4m3>(head_size, block_size, p, kind, grid, s, n);
}

}  // namespace pa
