// pa_launch.h -- host-side interface between the C ABI (api.cu) and the
// per-dtype kernel translation units.  Internal to libpa.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace pa {

// Everything a decode launch needs; passed to the kernels by value.
struct DecodeParams {
  void* out;                 // [S, H, D] in the cache dtype
  const void* q;             // [S, H, D]
  const void* k_cache;       // [NB, Hkv, D/x, BS, x]
  const void* v_cache;       // [NB, Hkv, D, BS]
  const int32_t* block_tables;  // [S, max_blocks_per_seq]
  const int32_t* seq_lens;      // [S]
  float* part_ml;            // [S, H, num_parts, 2]: (max in log2 units, sum) per partition
  float* part_o;             // [S, H, num_parts, D]: normalised partial outputs
  unsigned* err;             // device error word
  long long num_blocks;
  int max_blocks_per_seq;
  int num_seqs;
  int num_heads;
  int num_kv_heads;
  int group;                 // num_heads / num_kv_heads
  int max_seq_len;
  int block_size;
  int part_blocks;           // blocks per partition (>= every sequence's block count when unsplit)
  int num_parts;             // partitions of a max_seq_len sequence
  float scale_log2;          // scale * log2(e)
};

enum class DecodeKind { kSimt = 0, kMma = 1 };

// Kernel choice for a shape: tensor cores when a kv head serves >= 2 query
// heads of a 16-bit cache, CUDA cores otherwise.
inline DecodeKind decode_kind(int dtype, int group) {
  return (dtype != 0 && group >= 2) ? DecodeKind::kMma : DecodeKind::kSimt;
}

// Resident CTAs per SM of the main decode kernel for (dtype, D, BS, kind); 0 if unsupported.
int decode_ctas_per_sm(int dtype, int head_size, int block_size, DecodeKind kind);

// Enqueue the main decode kernel and, when some sequence spans more than one
// partition, the merge kernel.  *launches receives the number of kernels enqueued.
cudaError_t launch_decode(int dtype, int head_size, const DecodeParams& p, DecodeKind kind,
                          cudaStream_t stream, int* launches);

// Per-dtype entry points (decode_<dtype>.cu).
int decode_ctas_per_sm_f32(int head_size, int block_size, DecodeKind kind);
int decode_ctas_per_sm_f16(int head_size, int block_size, DecodeKind kind);
int decode_ctas_per_sm_bf16(int head_size, int block_size, DecodeKind kind);
cudaError_t launch_decode_f32(int head_size, const DecodeParams& p, DecodeKind kind, cudaStream_t s, int* n);
cudaError_t launch_decode_f16(int head_size, const DecodeParams& p, DecodeKind kind, cudaStream_t s, int* n);
cudaError_t launch_decode_bf16(int head_size, const DecodeParams& p, DecodeKind kind, cudaStream_t s, int* n);

// Write path (cache_ops.cu).
cudaError_t launch_reshape_and_cache(const void* key, const void* value, void* k_cache, void* v_cache,
                                     const int64_t* slot_mapping, int64_t num_tokens, int num_kv_heads,
                                     int head_size, int block_size, int64_t num_blocks, int elem_bytes,
                                     unsigned* err, cudaStream_t stream, int* launches);
cudaError_t launch_copy_blocks(void* k_cache, void* v_cache, const int64_t* src_dst, int64_t num_pairs,
                               int64_t block_bytes, int64_t num_blocks, unsigned* err, cudaStream_t stream,
                               int* launches);

}  // namespace pa
