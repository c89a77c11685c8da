// prefill.cu -- chunked-prefill attention over the paged pool, for sm_103a.
//
// What is computed: the step before decode ("vLLM's PagedAttention: why the KV
// cache is paged" §2.3: a prompt is processed and its K/V enter the cache, then
// tokens are generated one by one), read as causal attention of a chunk of new
// query tokens over the sequence's cache: for sequence s with L tokens cached
// (the chunk's own K/V already written) and a chunk of n tokens, query token i
// at position p = L - n + i attends to positions 0..p with
//     out = softmax(scale * q K^T) V
// over K, V gathered through the block table, as decode does for one token.
//
// The kernel is in prefill_ws.cuh (tcgen05 MMAs with accumulators in tensor
// memory, warp-specialised); this file holds its host-side launch: the two tensor
// maps its TMA copies read the pools through, and the dispatch over dtype, head
// size and block size.
#include <math.h>

#include <type_traits>

#include "pa_device.cuh"
#include "pa_launch.h"
#include "prefill_ws.cuh"

namespace pa {

// ---- host side ------------------------------------------------------------------------------

// cuTensorMapEncodeTiled, looked up once through the runtime (no link-time libcuda)
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
static EncodeTiledFn encoder() {
  static EncodeTiledFn fn = [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      f = nullptr;
    return reinterpret_cast<EncodeTiledFn>(f);
  }();
  return fn;
}

// The K pool [NB][Hkv][D/8][bs][8] seen as rows of 16 keys x 8 dims (128 16-bit
// elements, 256 bytes); a box is one row (tile::gather4 takes four of them).
template <int D, int BS>
cudaError_t encode_k_map(const PrefillParams& p, CUtensorMap* map) {
  const EncodeTiledFn enc = encoder();
  if (!enc) return cudaErrorNotSupported;
  const unsigned long long rows = (unsigned long long)p.num_blocks * p.num_kv_heads * (D / 8) * (BS / 16);
  if (rows > 0x7fffffffULL) return cudaErrorInvalidValue;  // rows are addressed with int32 coordinates
  const cuuint64_t dims[2] = {128, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {256};
  const cuuint32_t box[2] = {128, 1};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT16, 2, const_cast<void*>(p.k_cache), dims, strides, box,
                         estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                         CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

// The V pool [NB][Hkv][D][bs] seen as NB * Hkv * D rows of bs 16-bit elements; a box
// is one (block, kv head) tile, [D rows][bs keys], landing with the 32-byte (bs 16) or
// 64-byte (bs 32) swizzle: the K-major layout the P V MMA reads with the same swizzle.
template <int D, int BS>
cudaError_t encode_v_map(const PrefillParams& p, CUtensorMap* map) {
  const EncodeTiledFn enc = encoder();
  if (!enc) return cudaErrorNotSupported;
  const unsigned long long rows = (unsigned long long)p.num_blocks * p.num_kv_heads * D;
  if (rows > 0x7fffffffULL) return cudaErrorInvalidValue;  // box rows are addressed with int32 coordinates
  const cuuint64_t dims[2] = {(cuuint64_t)BS, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)BS * 2};
  const cuuint32_t box[2] = {(cuuint32_t)BS, (cuuint32_t)D};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT16, 2, const_cast<void*>(p.v_cache), dims, strides, box,
                         estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                         BS == 16 ? CU_TENSOR_MAP_SWIZZLE_32B : CU_TENSOR_MAP_SWIZZLE_64B,
                         CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

// The warp-specialised tcgen05 kernel (prefill_ws.cuh): clusters of two CTAs, each CTA a pair of 128-row query
// tiles, one CTA per SM.
template <typename T, int D, int BS>
cudaError_t launch_prefill_ws_t(const PrefillParams& p, cudaStream_t stream, int* launches) {
  using Sh = ws::Shape<T, D, BS>;
  *launches = 0;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  static unsigned done = 0;
  static int resident[32];  // clusters that fit on device d at once
  const bool cached = dev < 32 && (__atomic_load_n(&done, __ATOMIC_ACQUIRE) & (1u << dev));
  int clusters_resident = cached ? __atomic_load_n(&resident[dev], __ATOMIC_RELAXED) : 0;
  if (!cached) {
    e = cudaFuncSetAttribute(reinterpret_cast<const void*>(&ws::prefill_ws_kernel<T, D, BS>),
                             cudaFuncAttributeMaxDynamicSharedMemorySize, Sh::kSmem);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(reinterpret_cast<const void*>(&ws::prefill_ws_kernel<T, D, BS>),
                             cudaFuncAttributePreferredSharedMemoryCarveout, 100);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t q = {};
    q.gridDim = dim3(ws::kCluster);
    q.blockDim = dim3(ws::kThreads);
    q.dynamicSmemBytes = Sh::kSmem;
    cudaLaunchAttribute ca;
    ca.id = cudaLaunchAttributeClusterDimension;
    ca.val.clusterDim.x = ws::kCluster;
    ca.val.clusterDim.y = 1;
    ca.val.clusterDim.z = 1;
    q.attrs = &ca;
    q.numAttrs = 1;
    int n = 0;
    e = cudaOccupancyMaxActiveClusters(&n, reinterpret_cast<const void*>(&ws::prefill_ws_kernel<T, D, BS>), &q);
    if (e != cudaSuccess) return e;
    if (n < 1) return cudaErrorInvalidConfiguration;
    clusters_resident = n;
    if (dev < 32) {
      __atomic_store_n(&resident[dev], n, __ATOMIC_RELAXED);
      __atomic_fetch_or(&done, 1u << dev, __ATOMIC_RELEASE);
    }
  }
  CUtensorMap kmap, vmap;
  e = encode_k_map<D, BS>(p, &kmap);
  if (e != cudaSuccess) return e;
  e = encode_v_map<D, BS>(p, &vmap);
  if (e != cudaSuccess) return e;
  // sequence s has ceil(ceil(n_s G / 128) / 4) units of four tiles per kv head, at most
  // n_s G / 512 + 1 (rounded up); each cluster of two CTAs takes units until none is left
  const long long units = (long long)p.num_kv_heads * (((long long)p.num_query_tokens * p.group + ws::kUnitTiles * ws::kRows - 1) /
                                                           (ws::kUnitTiles * ws::kRows) +
                                                       p.num_seqs);
  long long clusters = units < clusters_resident ? units : clusters_resident;
  if (clusters > 32 * ws::kLoadsPerLane) clusters = 32 * ws::kLoadsPerLane;  // the scheduler's table of loads
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(clusters * ws::kCluster));
  cfg.blockDim = dim3(ws::kThreads);
  cfg.dynamicSmemBytes = Sh::kSmem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = ws::kCluster;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  e = cudaLaunchKernelEx(&cfg, ws::prefill_ws_kernel<T, D, BS>, p, kmap, vmap);
  if (e == cudaSuccess) *launches = 1;
  return e;
}

template <typename T, int D, int BS>
cudaError_t launch_prefill_t(const PrefillParams& p, cudaStream_t s, int* n) {
  return launch_prefill_ws_t<T, D, BS>(p, s, n);
}

template <typename T>
cudaError_t launch_prefill_dispatch(int head_size, int block_size, const PrefillParams& p, cudaStream_t s, int* n) {
  if (head_size == 64 && block_size == 16) return launch_prefill_t<T, 64, 16>(p, s, n);
  if (head_size == 64 && block_size == 32) return launch_prefill_t<T, 64, 32>(p, s, n);
  if (head_size == 128 && block_size == 16) return launch_prefill_t<T, 128, 16>(p, s, n);
  if (head_size == 128 && block_size == 32) return launch_prefill_t<T, 128, 32>(p, s, n);
  return cudaErrorInvalidValue;
}

cudaError_t launch_prefill(int dtype, int head_size, int block_size, const PrefillParams& p, cudaStream_t stream,
                           int* launches) {
  if (dtype == 1) return launch_prefill_dispatch<__half>(head_size, block_size, p, stream, launches);
  if (dtype == 2) return launch_prefill_dispatch<__nv_bfloat16>(head_size, block_size, p, stream, launches);
  return cudaErrorInvalidValue;
}

}  // namespace pa
