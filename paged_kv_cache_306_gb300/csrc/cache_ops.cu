// cache_ops.cu -- the write side of the paged KV cache.
//
// reshape_and_cache ("Reading vLLM's PagedAttention kernel", §3.2): each new
// token carries a flat slot (physical block * block_size + offset); its K and V
// rows are copied into that slot of the pools.  In the K pool a token's row is
// head_size/x runs of 16 bytes (one per x-element group), so every 16-byte
// group of the key row lands as one 16-byte store; the V pool stores a token's
// row with a stride of block_size elements, so V is an element scatter.
//
// copy_blocks ("vLLM's PagedAttention: why the KV cache is paged", §4.2): before
// a shared block is written it is copied whole to a fresh block; a physical
// block of one pool is one contiguous run of bytes, copied with 16-byte vectors.
#include <stdint.h>

#include "pa_device.cuh"
#include "pa_launch.h"

namespace pa {

template <int E> struct Word;
template <> struct Word<1> { using type = uint8_t; };
template <> struct Word<2> { using type = uint16_t; };
template <> struct Word<4> { using type = uint32_t; };

// One warp per (token, kv head), kWriteWarps heads per CTA: grid = (tokens, head
// groups).  Each lane issues all of its loads before its stores, so a head's row
// costs one round trip to memory.
constexpr int kWriteWarps = 4;

template <int E>
__global__ void __launch_bounds__(kWriteWarps * 32)
    reshape_and_cache_kernel(const unsigned char* __restrict__ key, const unsigned char* __restrict__ value,
                             unsigned char* __restrict__ k_cache, unsigned char* __restrict__ v_cache,
                             const int64_t* __restrict__ slot_mapping, int num_kv_heads, int head_size,
                             int block_size, long long num_blocks, unsigned* err) {
  using W = typename Word<E>::type;
  constexpr int X = 16 / E;
  griddep_wait();
  griddep_launch_dependents();
  const long long t = blockIdx.x;
  const int lane = threadIdx.x & 31;
  const int h = blockIdx.y * kWriteWarps + (threadIdx.x >> 5);
  if (h >= num_kv_heads) return;
  const long long slot = slot_mapping[t];
  if (slot < 0) return;  // padding token
  if (slot >= num_blocks * block_size) {
    if (h == 0 && lane == 0) set_error(err, kErrSlot);
    return;
  }
  const long long blk = slot / block_size;
  const int off = static_cast<int>(slot - blk * block_size);
  const int groups = head_size / X;
  const long long row = (t * num_kv_heads + h) * head_size;  // first element of the token's row for head h

  // K: 16-byte group g -> k_cache[blk, h, g, off, :]
  const long long kbase = (blk * num_kv_heads + h) * groups * block_size + off;  // in 16-byte groups
  for (int g0 = lane; g0 < groups; g0 += 64) {
    uint4 v[2];
#pragma unroll
    for (int j = 0; j < 2; ++j)
      if (g0 + 32 * j < groups) v[j] = *reinterpret_cast<const uint4*>(key + (row + (long long)(g0 + 32 * j) * X) * E);
#pragma unroll
    for (int j = 0; j < 2; ++j)
      if (g0 + 32 * j < groups)
        *reinterpret_cast<uint4*>(k_cache + (kbase + (long long)(g0 + 32 * j) * block_size) * 16) = v[j];
  }
  // V: element d -> v_cache[blk, h, d, off]
  const long long vbase = (blk * num_kv_heads + h) * head_size * block_size + off;
  for (int d0 = lane; d0 < head_size; d0 += 128) {
    W v[4];
#pragma unroll
    for (int j = 0; j < 4; ++j)
      if (d0 + 32 * j < head_size) v[j] = reinterpret_cast<const W*>(value)[row + d0 + 32 * j];
#pragma unroll
    for (int j = 0; j < 4; ++j)
      if (d0 + 32 * j < head_size) reinterpret_cast<W*>(v_cache)[vbase + (long long)(d0 + 32 * j) * block_size] = v[j];
  }
}

// The same write, a tile of kTokTile consecutive tokens of one kv head per CTA (the
// form a prefill chunk takes: consecutive tokens fill consecutive slots of a
// block).  The tile's key and value rows are loaded coalesced into shared memory,
// then stored with consecutive lanes on consecutive tokens: for a fixed 16-byte
// group of K (or a fixed dim of V) the tokens of one block land side by side, so a
// warp's stores to a block tile merge into few memory requests (one token per warp
// left V as a scatter of separate 2-byte stores).  Any slots work; padding tokens
// (slot < 0) are skipped.  Used for writes of many tokens whose tile fits the default
// shared memory.
constexpr int kTokTile = 32, kTiledThreads = 128;
// below this many tiles the per-token kernel spreads the stores over more SMs (measured
// on GB300: a Qwen-shaped decode step's 64 tokens x 4 kv heads wrote 5 us slower tiled)
constexpr long long kTiledMinCtas = 256;
__host__ __device__ constexpr int tiled_pitch_k(int row_bytes) { return row_bytes + 16; }  // 16-byte reads, spread banks
__host__ __device__ constexpr int tiled_pitch_v(int row_bytes) { return row_bytes + 4; }   // element reads, spread banks

template <int E>
__global__ void __launch_bounds__(kTiledThreads)
    reshape_and_cache_tiled_kernel(const unsigned char* __restrict__ key, const unsigned char* __restrict__ value,
                                   unsigned char* __restrict__ k_cache, unsigned char* __restrict__ v_cache,
                                   const int64_t* __restrict__ slot_mapping, long long num_tokens, int num_kv_heads,
                                   int head_size, int block_size, long long num_blocks, unsigned* err) {
  using W = typename Word<E>::type;
  constexpr int X = 16 / E;
  extern __shared__ __align__(16) unsigned char sm[];
  __shared__ long long s_blk[kTokTile];
  __shared__ int s_off[kTokTile];
  griddep_wait();
  griddep_launch_dependents();
  const int tid = threadIdx.x, h = blockIdx.y;
  const long long t0 = (long long)blockIdx.x * kTokTile;
  const int ntok = static_cast<int>(min((long long)kTokTile, num_tokens - t0));
  const int row_bytes = head_size * E, pk = tiled_pitch_k(row_bytes), pv = tiled_pitch_v(row_bytes);
  unsigned char* sK = sm;
  unsigned char* sV = sm + kTokTile * pk;
  if (tid < kTokTile) {
    long long blk = -1;
    int off = 0;
    if (tid < ntok) {
      const long long slot = slot_mapping[t0 + tid];
      if (slot >= num_blocks * block_size) {
        if (h == 0) set_error(err, kErrSlot);
      } else if (slot >= 0) {
        blk = slot / block_size;
        off = static_cast<int>(slot - blk * block_size);
      }
    }
    s_blk[tid] = blk;
    s_off[tid] = off;
  }
  // the tile's rows for head h, 16 bytes at a time (row_bytes is a multiple of 16); up to
  // kBatch chunks of each array per thread are loaded before any is stored, so a tile
  // of 16-bit rows of 128 dims costs one round trip to memory
  constexpr int kBatch = 4;
  const int chunks = row_bytes / 16, n = ntok * chunks;
  for (int base = 0; base < n; base += kBatch * kTiledThreads) {
    uint4 kv[kBatch], vv[kBatch];
#pragma unroll
    for (int q = 0; q < kBatch; ++q) {
      const int i = base + q * kTiledThreads + tid;
      if (i < n) {
        const int j = i / chunks, c = i - j * chunks;
        const long long row = ((t0 + j) * num_kv_heads + h) * (long long)row_bytes + c * 16;
        kv[q] = *reinterpret_cast<const uint4*>(key + row);
        vv[q] = *reinterpret_cast<const uint4*>(value + row);
      }
    }
#pragma unroll
    for (int q = 0; q < kBatch; ++q) {
      const int i = base + q * kTiledThreads + tid;
      if (i < n) {
        const int j = i / chunks, c = i - j * chunks;
        *reinterpret_cast<uint4*>(sK + j * pk + c * 16) = kv[q];
        uint32_t* dv = reinterpret_cast<uint32_t*>(sV + j * pv + c * 16);
        dv[0] = vv[q].x;
        dv[1] = vv[q].y;
        dv[2] = vv[q].z;
        dv[3] = vv[q].w;
      }
    }
  }
  __syncthreads();
  // K: 16-byte group g of token j -> k_cache[blk_j, h, g, off_j, :]
  const int groups = head_size / X;
  for (int i = tid; i < groups * kTokTile; i += kTiledThreads) {
    const int g = i / kTokTile, j = i - g * kTokTile;
    const long long blk = s_blk[j];
    if (j < ntok && blk >= 0)
      *reinterpret_cast<uint4*>(k_cache + (((blk * num_kv_heads + h) * groups + g) * block_size + s_off[j]) * 16) =
          *reinterpret_cast<const uint4*>(sK + j * pk + g * 16);
  }
  // V: element d of token j -> v_cache[blk_j, h, d, off_j]
  for (int i = tid; i < head_size * kTokTile; i += kTiledThreads) {
    const int d = i / kTokTile, j = i - d * kTokTile;
    const long long blk = s_blk[j];
    if (j < ntok && blk >= 0)
      reinterpret_cast<W*>(v_cache)[((blk * num_kv_heads + h) * head_size + d) * block_size + s_off[j]] =
          *reinterpret_cast<const W*>(sV + j * pv + d * E);
  }
}

// Quantising write into an FP8 E4M3 cache (the kv_cache_dtype, k_scale and v_scale
// arguments of the write, "Reading vLLM's PagedAttention kernel" §3.2): element x
// of the key (value) row is stored as the E4M3 code of x / k_scale (x / v_scale),
// the division correctly rounded in fp32, the code rounded to nearest (ties to
// even) and clamped to +-448.  One warp per (token, kv head) as above; in the K
// pool a 16-element group of a head is 16 contiguous codes, one 16-byte store.
template <typename TS>
__global__ void __launch_bounds__(kWriteWarps * 32)
    reshape_and_cache_e4m3_kernel(const TS* __restrict__ key, const TS* __restrict__ value,
                                  unsigned char* __restrict__ k_cache, unsigned char* __restrict__ v_cache,
                                  const int64_t* __restrict__ slot_mapping, int num_kv_heads, int head_size,
                                  int block_size, long long num_blocks, float k_scale, float v_scale, unsigned* err) {
  constexpr int NV = sizeof(TS);  // 16-byte loads per 16-element group
  griddep_wait();
  griddep_launch_dependents();
  const long long t = blockIdx.x;
  const int lane = threadIdx.x & 31;
  const int h = blockIdx.y * kWriteWarps + (threadIdx.x >> 5);
  if (h >= num_kv_heads) return;
  const long long slot = slot_mapping[t];
  if (slot < 0) return;  // padding token
  if (slot >= num_blocks * block_size) {
    if (h == 0 && lane == 0) set_error(err, kErrSlot);
    return;
  }
  const long long blk = slot / block_size;
  const int off = static_cast<int>(slot - blk * block_size);
  const int groups = head_size / 16;
  const long long row = (t * num_kv_heads + h) * head_size;
  for (int g = lane; g < groups; g += 32) {
    uint4 raw[NV];
#pragma unroll
    for (int i = 0; i < NV; ++i) raw[i] = reinterpret_cast<const uint4*>(key + row + (long long)g * 16)[i];
    const TS* src = reinterpret_cast<const TS*>(raw);
    uint32_t w[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      uint32_t packed = 0;
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        const float a = __fdiv_rn(DType<TS>::to_f32(src[4 * i + 2 * j]), k_scale);
        const float b = __fdiv_rn(DType<TS>::to_f32(src[4 * i + 2 * j + 1]), k_scale);
        const uint32_t two = __nv_cvt_float2_to_fp8x2(make_float2(a, b), __NV_SATFINITE, __NV_E4M3);
        packed |= (two & 0xffffu) << (16 * j);
      }
      w[i] = packed;
    }
    *reinterpret_cast<uint4*>(k_cache + (((blk * num_kv_heads + h) * groups + g) * block_size + off) * 16) =
        make_uint4(w[0], w[1], w[2], w[3]);
  }
  const long long vbase = (blk * num_kv_heads + h) * head_size * block_size + off;
  for (int d0 = lane; d0 < head_size; d0 += 128) {
    TS v[4];
#pragma unroll
    for (int j = 0; j < 4; ++j)
      if (d0 + 32 * j < head_size) v[j] = value[row + d0 + 32 * j];
#pragma unroll
    for (int j = 0; j < 4; ++j)
      if (d0 + 32 * j < head_size) {
        const float x = __fdiv_rn(DType<TS>::to_f32(v[j]), v_scale);
        v_cache[vbase + (long long)(d0 + 32 * j) * block_size] =
            static_cast<unsigned char>(__nv_cvt_float_to_fp8(x, __NV_SATFINITE, __NV_E4M3));
      }
  }
}

// grid = (num_pairs, 2 [K, V], chunks)
__global__ void __launch_bounds__(256)
    copy_blocks_kernel(unsigned char* k_cache, unsigned char* v_cache, const int64_t* __restrict__ src_dst,
                       long long block_bytes, long long num_blocks, unsigned* err) {
  griddep_wait();
  griddep_launch_dependents();
  const long long i = blockIdx.x;
  const long long src = src_dst[2 * i], dst = src_dst[2 * i + 1];
  if (src < 0 || src >= num_blocks || dst < 0 || dst >= num_blocks) {
    if (threadIdx.x == 0 && blockIdx.y == 0 && blockIdx.z == 0) set_error(err, kErrCopyId);
    return;
  }
  unsigned char* base = blockIdx.y == 0 ? k_cache : v_cache;
  const uint4* s = reinterpret_cast<const uint4*>(base + src * block_bytes);
  uint4* d = reinterpret_cast<uint4*>(base + dst * block_bytes);
  const long long nvec = block_bytes / 16;
  for (long long v = (long long)blockIdx.z * blockDim.x + threadIdx.x; v < nvec; v += (long long)gridDim.z * blockDim.x)
    d[v] = s[v];
}

cudaError_t launch_reshape_and_cache(const void* key, const void* value, void* k_cache, void* v_cache,
                                     const int64_t* slot_mapping, int64_t num_tokens, int num_kv_heads,
                                     int head_size, int block_size, int64_t num_blocks, int elem_bytes,
                                     unsigned* err, cudaStream_t stream, int* launches) {
  *launches = 0;
  if (num_tokens == 0) return cudaSuccess;
  const auto* kp = static_cast<const unsigned char*>(key);
  const auto* vp = static_cast<const unsigned char*>(value);
  auto* kc = static_cast<unsigned char*>(k_cache);
  auto* vc = static_cast<unsigned char*>(v_cache);
  const int row_bytes = head_size * elem_bytes;
  const int tiled_smem = kTokTile * (tiled_pitch_k(row_bytes) + tiled_pitch_v(row_bytes));
  // the tiled form for writes of many tokens (a prefill chunk; its tiles fill the GPU
  // and its consecutive slots merge stores), within the default dynamic shared memory;
  // a decode step's one token per sequence spreads better one token per warp
  const long long tiles = (num_tokens + kTokTile - 1) / kTokTile * num_kv_heads;
  if (tiles >= kTiledMinCtas && tiled_smem <= 40 * 1024) {
    const dim3 grid(static_cast<unsigned>((num_tokens + kTokTile - 1) / kTokTile), static_cast<unsigned>(num_kv_heads));
    const dim3 block(kTiledThreads);
    const cudaError_t e =
        elem_bytes == 4   ? launch_pdl(reshape_and_cache_tiled_kernel<4>, grid, block, tiled_smem, stream, kp, vp, kc,
                                       vc, slot_mapping, (long long)num_tokens, num_kv_heads, head_size, block_size,
                                       (long long)num_blocks, err)
        : elem_bytes == 2 ? launch_pdl(reshape_and_cache_tiled_kernel<2>, grid, block, tiled_smem, stream, kp, vp, kc,
                                       vc, slot_mapping, (long long)num_tokens, num_kv_heads, head_size, block_size,
                                       (long long)num_blocks, err)
                          : launch_pdl(reshape_and_cache_tiled_kernel<1>, grid, block, tiled_smem, stream, kp, vp, kc,
                                       vc, slot_mapping, (long long)num_tokens, num_kv_heads, head_size, block_size,
                                       (long long)num_blocks, err);
    if (e == cudaSuccess) *launches = 1;
    return e;
  }
  const dim3 grid(static_cast<unsigned>(num_tokens), (num_kv_heads + kWriteWarps - 1) / kWriteWarps);
  const dim3 block(kWriteWarps * 32);
  const cudaError_t e =
      elem_bytes == 4   ? launch_pdl(reshape_and_cache_kernel<4>, grid, block, 0, stream, kp, vp, kc, vc,
                                     slot_mapping, num_kv_heads, head_size, block_size, (long long)num_blocks, err)
      : elem_bytes == 2 ? launch_pdl(reshape_and_cache_kernel<2>, grid, block, 0, stream, kp, vp, kc, vc,
                                     slot_mapping, num_kv_heads, head_size, block_size, (long long)num_blocks, err)
                        : launch_pdl(reshape_and_cache_kernel<1>, grid, block, 0, stream, kp, vp, kc, vc,
                                     slot_mapping, num_kv_heads, head_size, block_size, (long long)num_blocks, err);
  if (e == cudaSuccess) *launches = 1;
  return e;
}

cudaError_t launch_reshape_and_cache_e4m3(const void* key, const void* value, void* k_cache, void* v_cache,
                                           const int64_t* slot_mapping, int64_t num_tokens, int num_kv_heads,
                                           int head_size, int block_size, int64_t num_blocks, int key_dtype,
                                           float k_scale, float v_scale, unsigned* err, cudaStream_t stream,
                                           int* launches) {
  *launches = 0;
  if (num_tokens == 0) return cudaSuccess;
  auto* kc = static_cast<unsigned char*>(k_cache);
  auto* vc = static_cast<unsigned char*>(v_cache);
  const dim3 grid(static_cast<unsigned>(num_tokens), (num_kv_heads + kWriteWarps - 1) / kWriteWarps);
  const dim3 block(kWriteWarps * 32);
  const long long nb = num_blocks;
  cudaError_t e;
  if (key_dtype == 0)
    e = launch_pdl(reshape_and_cache_e4m3_kernel<float>, grid, block, 0, stream, static_cast<const float*>(key),
                   static_cast<const float*>(value), kc, vc, slot_mapping, num_kv_heads, head_size, block_size, nb,
                   k_scale, v_scale, err);
  else if (key_dtype == 1)
    e = launch_pdl(reshape_and_cache_e4m3_kernel<__half>, grid, block, 0, stream,
                   static_cast<const __half*>(key), static_cast<const __half*>(value), kc, vc, slot_mapping,
                   num_kv_heads, head_size, block_size, nb, k_scale, v_scale, err);
  else
    e = launch_pdl(reshape_and_cache_e4m3_kernel<__nv_bfloat16>, grid, block, 0, stream,
                   static_cast<const __nv_bfloat16*>(key), static_cast<const __nv_bfloat16*>(value), kc, vc,
                   slot_mapping, num_kv_heads, head_size, block_size, nb, k_scale, v_scale, err);
  if (e == cudaSuccess) *launches = 1;
  return e;
}

cudaError_t launch_copy_blocks(void* k_cache, void* v_cache, const int64_t* src_dst, int64_t num_pairs,
                               int64_t block_bytes, int64_t num_blocks, unsigned* err, cudaStream_t stream,
                               int* launches) {
  *launches = 0;
  if (num_pairs == 0) return cudaSuccess;
  const long long nvec = block_bytes / 16;
  long long chunks = (nvec + 256 * 4 - 1) / (256 * 4);
  if (chunks > 64) chunks = 64;
  dim3 grid(static_cast<unsigned>(num_pairs), 2, static_cast<unsigned>(chunks));
  const cudaError_t e = launch_pdl(copy_blocks_kernel, grid, dim3(256), 0, stream,
                                   static_cast<unsigned char*>(k_cache), static_cast<unsigned char*>(v_cache),
                                   src_dst, (long long)block_bytes, (long long)num_blocks, err);
  if (e == cudaSuccess) *launches = 1;
  return e;
}

}  // namespace pa
