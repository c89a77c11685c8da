// pa_launch.h -- host-side interface between the C ABI (api.cu) and the
// per-dtype kernel translation units.  Internal to libpa.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace pa {

// Sequences handled by one launch of the decode kernels (their per-sequence
// tables live in shared memory); larger batches are launched in chunks.
constexpr int kMaxSeqsPerLaunch = 1024;

// Shape of the decode CTA.  One CTA per SM; every warp is an independent worker
// with a ring of stages, one stage = the K tile and the V tile of one block.
// Measured on GB300: about 128 KiB of copies in flight per SM streams the pool
// fastest (more in flight queues up in the memory system, less leaves it idle).
// The math decides how many warps share those bytes.  The tensor-core kernel over
// one 8-head tile (mode 1) with stages of at most 4 KiB (FP8 tiles, or head size
// 64) runs 16 warps of two or more stages, four warps per scheduler to hide its
// latencies (its widening of FP8 codes makes it ALU-bound otherwise); with larger
// stages 16 warps would leave each warp a single stage, and 8 warps with two
// stages each measured faster.  The other kernels run 8 warps (4 for 32 KiB
// stages).
constexpr int kInFlightBytes = 128 * 1024;
__host__ __device__ constexpr int decode_warps(int stage_bytes, int mode) {
  return (mode == 1 && stage_bytes <= 4096) ? 16 : (stage_bytes <= 16384 ? 8 : 4);
}
__host__ __device__ constexpr int decode_stages(int stage_bytes, int mode) {
  return kInFlightBytes / (decode_warps(stage_bytes, mode) * stage_bytes) > 1
             ? kInFlightBytes / (decode_warps(stage_bytes, mode) * stage_bytes)
             : 1;
}

// Costs for balancing the decode warps' ranges (relative units): a block of a
// shared segment (two 8-column tiles of query rows; measured on GB300, ~1.28 times
// an 8-column block), an own block, and the fixed work of a segment (its query
// rows loaded with a global-memory round trip, its state reset, its last block's
// tail cleared and its result stored) -- about one and a half blocks.  Batches of
// many short sequences leave some warps with dozens of segments: counted in
// blocks alone, those warps finish last.
constexpr int kSharedCost = 5, kOwnCost = 4, kSegCost = 6;

// Everything a decode launch needs; passed to the kernels by value.
struct DecodeParams {
  void* out;                    // [S, H, D] in the cache dtype
  const void* q;                // [S, H, D]
  const void* k_cache;          // [NB, Hkv, D/x, BS, x]
  const void* v_cache;          // [NB, Hkv, D, BS]
  const int32_t* block_tables;  // [S, max_blocks_per_seq]
  const int32_t* seq_lens;      // [S]
  float* part_ml;               // [slots, rows, 2]: (max in log2 units, sum) of a piece
  float* part_o;                // [slots, rows, D]: normalised partial output of a piece
  int2* part_tag;               // [slots]: (segment, epoch) that wrote the slot
  int* seg_first;               // [S * units]: first piece's slot, or -1 when no merge is needed
  int* seg_last;                // [S * units]: last piece's slot
  unsigned* err;                // device error word
  long long num_blocks;
  int max_blocks_per_seq;
  int num_seqs;                 // <= kMaxSeqsPerLaunch
  int num_heads;
  int num_kv_heads;
  int group;                    // num_heads / num_kv_heads
  int units;                    // head units per sequence (a segment is one sequence x one unit)
  int rows;                     // query rows per unit stored in a partial slot
  int max_seq_len;
  int part_blocks;              // blocks per caller partition; a huge value when none
  int num_slots;                // partial-result slots in the workspace
  unsigned epoch;               // distinguishes this launch's partial slots from stale ones
  float scale_log2;             // scale * k_scale * log2(e)
  float out_scale;              // v_scale: a quantised cache's V reads back as code * v_scale
  // The fused step (pa_decode_step): the new token of each sequence s (rows s of
  // new_key and new_value, [S, Hkv, D] in the cache dtype) goes into position
  // seq_lens[s] - 1 as part of decode; fused == 0 for plain decode.
  const void* new_key;            // the query dtype for an FP8 pool (quantised with the scales below)
  const void* new_value;
  float write_k_scale, write_v_scale;  // FP8 pool: stored code = E4M3(x / scale)
  int fused;
  // > 0 only in the timeout-path test: every warp's first pipeline wait runs out
  // after this many nanoseconds (see pa_set_test_wait_limit)
  unsigned long long test_wait_ns;
  // Shared prefixes (pa_decode_shared): sequences with the same prefix_group[s]
  // (consecutive runs) hold the first prefix_blocks[s] blocks of a common prefix,
  // so any two of them agree on their first min(prefix_blocks) block-table entries.
  // A run is cut into clusters of up to `members` sequences; a cluster's prefix
  // blocks are read once for all its members (one segment whose tensor-core
  // columns are the members' query heads, read through the table of the member
  // that holds the most of them) and merged with each member's own blocks.
  // shared == 0: unused.
  const int32_t* prefix_group;
  const int32_t* prefix_blocks;
  int* seq_info;                // [2 S]: the cluster layout (s_info, then s_lead), written by CTA 0 for the merge
  int shared;
  int members;
};

// Packed per-sequence cluster layout (shared prefixes).  info: bits 0..21 the
// sequence's shared blocks sh (its own segment starts there), bits 22..26 its
// member index (0 = the cluster's leader), bits 27..31 the cluster size minus one
// (leaders only).  lead (leaders only): bits 0..21 the length B of the cluster's
// shared segment (the second largest prefix_blocks of its members: past it only one
// member holds the blocks), bits 22..26 the member whose table it is read through.
constexpr int kInfoOffBits = 22;
__host__ __device__ constexpr int info_off(int v) { return v & ((1 << kInfoOffBits) - 1); }
__host__ __device__ constexpr int info_member(int v) { return (v >> kInfoOffBits) & 31; }
__host__ __device__ constexpr int info_size(int v) { return ((v >> 27) & 31) + 1; }

// CUDA cores, or tensor cores with one (up to 8 query heads per kv head) or two
// 8-head tiles per head unit.
enum class DecodeKind { kSimt = 0, kMma8 = 1, kMma16 = 2 };

// Kernel choice for a shape: tensor cores when a kv head serves >= 2 query heads
// of a 16-bit cache, or any number of an FP8 cache; CUDA cores otherwise.  With
// one query head per kv head the tensor-core tile is 1/8 used, yet for FP8 it
// wins: its fp16 widening costs two instructions per four codes (measured on
// GB300, 16 x 2048-token MHA layer: 54.9 us against 88.1 us on CUDA cores), while
// a 16-bit cache streams as fast on CUDA cores (94.0 against 96.6 us).
inline DecodeKind decode_kind(int dtype, int group) {
  if (dtype == 0 || (group < 2 && dtype != 3)) return DecodeKind::kSimt;
  return group <= 8 ? DecodeKind::kMma8 : DecodeKind::kMma16;
}

// Head units per sequence and query rows per unit for a kernel kind: tensor-core
// units are one kv head's query heads, 16 at a time.
inline int decode_units(DecodeKind k, int num_heads, int num_kv_heads) {
  const int g = num_heads / num_kv_heads;
  return k != DecodeKind::kSimt ? num_kv_heads * ((g + 15) / 16) : num_heads;
}
inline int decode_rows(DecodeKind k, int num_heads, int num_kv_heads) {
  const int g = num_heads / num_kv_heads;
  return k != DecodeKind::kSimt ? (g < 16 ? g : 16) : 1;
}

// Warps per decode CTA for a cache dtype size, head size, block size and kind.
inline int decode_warps_for(int elem_bytes, int head_size, int block_size, DecodeKind kind) {
  return decode_warps(2 * head_size * block_size * elem_bytes, static_cast<int>(kind));
}

// Resident CTAs per SM of the main decode kernel for (dtype, D, BS, kind); 0 if unsupported.
int decode_ctas_per_sm(int dtype, int head_size, int block_size, DecodeKind kind);

// Enqueue the main decode kernel (grid CTAs) and the merge kernel for one chunk of sequences.
cudaError_t launch_decode(int dtype, int head_size, int block_size, const DecodeParams& p, DecodeKind kind,
                          int grid, cudaStream_t stream, int* launches);

// Per-dtype entry points (decode_<dtype>.cu).
int decode_ctas_per_sm_f32(int head_size, int block_size, DecodeKind kind);
int decode_ctas_per_sm_f16(int head_size, int block_size, DecodeKind kind);
int decode_ctas_per_sm_bf16(int head_size, int block_size, DecodeKind kind);
cudaError_t launch_decode_f32(int head_size, int block_size, const DecodeParams& p, DecodeKind kind, int grid,
                              cudaStream_t s, int* n);
cudaError_t launch_decode_f16(int head_size, int block_size, const DecodeParams& p, DecodeKind kind, int grid,
                              cudaStream_t s, int* n);
cudaError_t launch_decode_bf16(int head_size, int block_size, const DecodeParams& p, DecodeKind kind, int grid,
                               cudaStream_t s, int* n);
// FP8 E4M3 cache with fp16 (q_is_bf16 == false) or bf16 queries (decode_fp8.cu).
int decode_ctas_per_sm_fp8(bool q_is_bf16, int head_size, int block_size, DecodeKind kind);
cudaError_t launch_decode_fp8(bool q_is_bf16, int head_size, int block_size, const DecodeParams& p, DecodeKind kind,
                              int grid, cudaStream_t s, int* n);

// Chunked prefill (prefill.cu): causal attention of a chunk of new query tokens
// per sequence over the paged pool; 16-bit caches.
struct PrefillParams {
  void* out;                       // [num_query_tokens, H, D]
  const void* q;                   // [num_query_tokens, H, D]
  const void* k_cache;
  const void* v_cache;
  const int32_t* block_tables;     // [S, max_blocks_per_seq]
  const int32_t* seq_lens;         // [S]: tokens in the cache, the chunk's included
  const int32_t* query_start_loc;  // [S + 1]: the chunk of sequence s is rows qsl[s] .. qsl[s+1]-1
  unsigned* err;
  long long num_blocks;
  int max_blocks_per_seq;
  int num_seqs;                    // <= kMaxSeqsPerLaunch
  int num_query_tokens;
  int num_heads;
  int num_kv_heads;
  int group;
  int max_seq_len;
  float scale_log2;
  unsigned long long test_wait_ns;  // > 0 only in the timeout-path test (see pa_set_test_wait_limit)
};
cudaError_t launch_prefill(int dtype, int head_size, int block_size, const PrefillParams& p, cudaStream_t stream,
                           int* launches);

// Write path (cache_ops.cu).
cudaError_t launch_reshape_and_cache(const void* key, const void* value, void* k_cache, void* v_cache,
                                     const int64_t* slot_mapping, int64_t num_tokens, int num_kv_heads,
                                     int head_size, int block_size, int64_t num_blocks, int elem_bytes,
                                     unsigned* err, cudaStream_t stream, int* launches);
cudaError_t launch_reshape_and_cache_e4m3(const void* key, const void* value, void* k_cache, void* v_cache,
                                           const int64_t* slot_mapping, int64_t num_tokens, int num_kv_heads,
                                           int head_size, int block_size, int64_t num_blocks, int key_dtype,
                                           float k_scale, float v_scale, unsigned* err, cudaStream_t stream,
                                           int* launches);
cudaError_t launch_copy_blocks(void* k_cache, void* v_cache, const int64_t* src_dst, int64_t num_pairs,
                               int64_t block_bytes, int64_t num_blocks, unsigned* err, cudaStream_t stream,
                               int* launches);

}  // namespace pa
