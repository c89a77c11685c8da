// decode_kernels.cuh -- paged-attention decode kernels for sm_103a.
//
// What is computed ("Reading vLLM's PagedAttention kernel", §2 flowchart, §3.3,
// §3.4): for one sequence s and the query heads that share kv head kvh, walk the
// sequence's block-table row in logical order; for each logical block look up
// the physical block, bring its K tile and V tile in, compute the scaled scores
// q.K^T, fold them into a running (max m, normaliser l, accumulator acc) online
// softmax, and finish with acc / l.  When the sequence is split into partitions
// ("PARTITION_SIZE" in §3.3) every partition is one CTA and writes
// (m, l, acc / l); the merge kernel combines them.
//
// How it maps to the GB300 SM:
//   * One CTA per (partition, head unit, sequence); NWARPS warps per CTA.  Warp w
//     takes the partition's logical blocks w, w + NWARPS, ...  Each warp owns a
//     STAGES-deep ring of shared-memory stages; a stage holds the K tile and the V
//     tile of one (physical block, kv head).  In this pool layout both tiles are
//     contiguous runs of head_size * block_size elements, so each is one 1-D bulk
//     copy issued by the TMA unit (cp.async.bulk) that signals an mbarrier with
//     its byte count.  The ring keeps STAGES blocks per warp in flight while the
//     warp computes on the oldest.
//   * Tensor-core kernel (16-bit caches, >= 2 query heads per kv head): the
//     query heads of one kv head are the 16 rows of an m16n8k16 tile, so one K/V
//     read serves all of them.  S = Q K^T takes K straight from the stage with
//     ldmatrix (a K-pool row of 8 dims x 16 B is exactly an 8x8 b16 fragment
//     row); P V takes V the same way (a V-pool row holds 8 consecutive tokens per
//     16 B).  P stays in registers between the two products.  P is split into a
//     rounded 16-bit high part and the rounded remainder, so P V keeps ~16
//     significant bits instead of 8 (bf16) or 11 (fp16).
//   * CUDA-core kernel (fp32 caches, or one query head per kv head): lanes split a
//     block's tokens and head dims; dot products and softmax statistics are
//     warp-shuffle reductions.
//   * The warps of a CTA merge their (m, l, acc) through shared memory at the end.
#pragma once

#include <math.h>

#include "pa_device.cuh"
#include "pa_launch.h"

namespace pa {

constexpr int kDecodeWarps = 4;
constexpr uint64_t kWaitLimitNs = 1000000000ull;  // 1 s, then PA_DEVERR_TIMEOUT

// Ring depth per warp from the bytes of one stage (K tile + V tile).
constexpr int decode_stages(int stage_bytes) {
  return stage_bytes <= 4096 ? 4 : stage_bytes <= 8192 ? 3 : stage_bytes <= 16384 ? 2 : 1;
}

template <typename T, int D, int BS>
struct DecodeShape {
  static constexpr int kElem = sizeof(T);
  static constexpr int kX = 16 / kElem;                   // elements per 16-byte K group
  static constexpr int kTile = D * BS * kElem;            // bytes of one K (or V) tile
  static constexpr int kStages = decode_stages(2 * kTile);
  static constexpr int kRingBytes = kDecodeWarps * kStages * 2 * kTile;
  static constexpr int kBarBytes = kDecodeWarps * kStages * 8;
};

// --- pieces shared by both kernels -------------------------------------------------------------

// Per-warp view of the work of one CTA: the partition's blocks assigned to this warp.
struct WarpWork {
  int blk0;      // first logical block of the partition
  int my_n;      // blocks this warp processes
  int warp;
  __device__ __forceinline__ int logical_block(int i) const { return blk0 + warp + i * kDecodeWarps; }
};

// Block-table lookups for a warp, 32 entries per global load.
struct TableCursor {
  const int32_t* row;
  long long num_blocks;
  unsigned* err;
  int loaded_group;
  int ids;
  __device__ __forceinline__ int phys(const WarpWork& w, int i, int lane) {
    const int grp = i >> 5;
    if (grp != loaded_group) {
      const int k = (grp << 5) + lane;
      ids = k < w.my_n ? __ldg(row + w.logical_block(k)) : 0;
      loaded_group = grp;
    }
    int b = __shfl_sync(0xffffffffu, ids, i & 31);
    if (b < 0 || b >= num_blocks) {  // out-of-pool entry: record it, read block 0 instead
      if (lane == 0) set_error(err, kErrBlockId);
      b = 0;
    }
    return b;
  }
};

// Issue the bulk copies of block i of this warp into its ring stage (lane 0 only).
template <int TILE, int STAGES>
__device__ __forceinline__ void issue_stage(unsigned char* ring, uint64_t* bars, const void* k_cache,
                                            const void* v_cache, long long tile_index, int i, int lane) {
  if (lane == 0) {
    const int st = i % STAGES;
    unsigned char* dst = ring + st * 2 * TILE;
    mbar_arrive_expect_tx(&bars[st], 2 * TILE);
    bulk_copy_g2s(dst, static_cast<const unsigned char*>(k_cache) + tile_index * TILE, TILE, &bars[st]);
    bulk_copy_g2s(dst + TILE, static_cast<const unsigned char*>(v_cache) + tile_index * TILE, TILE, &bars[st]);
  }
}

// Wait for block i's stage.  On timeout record the error and drain the copies
// still in flight (each with its own bounded wait) so none lands after exit.
template <int STAGES>
__device__ __forceinline__ bool wait_stage(uint64_t* bars, int i, int my_n, unsigned* err, int lane) {
  const int st = i % STAGES;
  const bool ok = __all_sync(0xffffffffu, mbar_wait_bounded(&bars[st], (i / STAGES) & 1, kWaitLimitNs));
  if (!ok) {
    if (lane == 0) set_error(err, kErrTimeout);
    for (int j = i + 1; j < my_n && j < i + STAGES; ++j)
      mbar_wait_bounded(&bars[j % STAGES], (j / STAGES) & 1, kWaitLimitNs / 8);
  }
  return ok;
}

// Zero the V columns of tokens >= rem in a stage (only the last, partial block):
// those slots may hold anything, and 0 * NaN would poison the sum.
template <typename T, int D, int BS>
__device__ __forceinline__ void zero_tail_v(unsigned char* vtile, int rem, int lane) {
  T* v = reinterpret_cast<T*>(vtile);
  for (int idx = lane; idx < D * BS; idx += 32)
    if ((idx % BS) >= rem) v[idx] = DType<T>::from_f32(0.f);
  __syncwarp();
}

// Combine the per-warp (m, l, acc) of `rows` query rows and write the output
// (single partition) or the partition's partial result.
//   wm, wl: [kDecodeWarps][rows_stride]; wo: [kDecodeWarps][rows_stride][D]
template <typename T, int D>
__device__ __forceinline__ void merge_and_store(const DecodeParams& p, const float* wm, const float* wl,
                                                const float* wo, int rows_stride, int nrows, int s, int h0,
                                                int part, bool single) {
  for (int idx = threadIdx.x; idx < nrows * D; idx += kDecodeWarps * 32) {
    const int r = idx / D, d = idx % D;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kDecodeWarps; ++w) M = fmaxf(M, wm[w * rows_stride + r]);
    float lsum = 0.f, o = 0.f;
#pragma unroll
    for (int w = 0; w < kDecodeWarps; ++w) {
      const float f = exp2f(wm[w * rows_stride + r] - M);
      lsum += wl[w * rows_stride + r] * f;
      o += wo[(w * rows_stride + r) * D + d] * f;
    }
    const long long sh = (long long)s * p.num_heads + h0 + r;
    if (single) {
      static_cast<T*>(p.out)[sh * D + d] = DType<T>::from_f32(o / lsum);
    } else {
      const long long slot = sh * p.num_parts + part;
      p.part_o[slot * D + d] = o / lsum;
      if (d == 0) {
        p.part_ml[slot * 2] = M;
        p.part_ml[slot * 2 + 1] = lsum;
      }
    }
  }
}

// A sequence whose length is outside [1, max_seq_len]: record it, zero its rows.
template <typename T, int D>
__device__ __forceinline__ void reject_sequence(const DecodeParams& p, int s, int h0, int nrows) {
  if (threadIdx.x == 0) set_error(p.err, kErrSeqLen);
  T* out = static_cast<T*>(p.out);
  for (int idx = threadIdx.x; idx < nrows * D; idx += blockDim.x)
    out[((long long)s * p.num_heads + h0 + idx / D) * D + idx % D] = DType<T>::from_f32(0.f);
}

// --- tensor-core kernel ------------------------------------------------------------------------
//
// grid = (num_parts, num_kv_heads * ceil(G / 16), num_seqs); 16 query heads per CTA.
template <typename T, int D, int BS>
__global__ void __launch_bounds__(kDecodeWarps * 32)
    decode_mma_kernel(const DecodeParams p) {
  using Sh = DecodeShape<T, D, BS>;
  constexpr int TILE = Sh::kTile, STAGES = Sh::kStages;
  constexpr int NT = BS / 8;   // token n-tiles of S
  constexpr int KS = D / 16;   // k-steps over head dims for S
  constexpr int DT = D / 8;    // head-dim n-tiles of O
  constexpr int KK = BS / 16;  // token k-steps for O
  static_assert(kDecodeWarps * (16 * D + 32) * 4 <= Sh::kRingBytes, "merge area must fit in the ring");
  extern __shared__ __align__(128) unsigned char smem[];

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, t4 = lane & 3;
  const int s = blockIdx.z, part = blockIdx.x;
  const int units = (p.group + 15) >> 4;
  const int kvh = blockIdx.y / units;
  const int h0 = kvh * p.group + (blockIdx.y % units) * 16;
  const int nh = min(16, kvh * p.group + p.group - h0);

  const int L = __ldg(p.seq_lens + s);
  if (L < 1 || L > p.max_seq_len) {
    if (part == 0) reject_sequence<T, D>(p, s, h0, nh);
    return;
  }
  const int nblk = (L + BS - 1) / BS;
  const int nparts = (nblk + p.part_blocks - 1) / p.part_blocks;
  if (part >= nparts) return;
  WarpWork work;
  work.blk0 = part * p.part_blocks;
  work.warp = warp;
  const int nb_part = min(nblk, work.blk0 + p.part_blocks) - work.blk0;
  work.my_n = nb_part > warp ? (nb_part - warp + kDecodeWarps - 1) / kDecodeWarps : 0;

  unsigned char* ring = smem + warp * STAGES * 2 * TILE;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + Sh::kRingBytes) + warp * STAGES;
  if (lane == 0) {
    for (int st = 0; st < STAGES; ++st) mbar_init(&bars[st], 1);
    fence_barrier_init();
  }
  __syncwarp();

  TableCursor tc{p.block_tables + (long long)s * p.max_blocks_per_seq, p.num_blocks, p.err, -1, 0};
  const long long head_tiles = p.num_kv_heads;
  for (int i = 0; i < STAGES && i < work.my_n; ++i) {
    const int phys = tc.phys(work, i, lane);
    issue_stage<TILE, STAGES>(ring, bars, p.k_cache, p.v_cache, phys * head_tiles + kvh, i, lane);
  }

  // Q fragments (A operand, rows = query heads h0 .. h0+15, zero past nh).
  uint32_t qf[KS][4];
  {
    const T* q = static_cast<const T*>(p.q);
    const T* q0 = q + ((long long)s * p.num_heads + h0 + g) * D;
    const T* q1 = q0 + 8 * D;
    const bool v0 = g < nh, v1 = g + 8 < nh;
#pragma unroll
    for (int ks = 0; ks < KS; ++ks) {
      const int d = ks * 16 + 2 * t4;
      qf[ks][0] = v0 ? __ldg(reinterpret_cast<const unsigned int*>(q0 + d)) : 0u;
      qf[ks][1] = v1 ? __ldg(reinterpret_cast<const unsigned int*>(q1 + d)) : 0u;
      qf[ks][2] = v0 ? __ldg(reinterpret_cast<const unsigned int*>(q0 + d + 8)) : 0u;
      qf[ks][3] = v1 ? __ldg(reinterpret_cast<const unsigned int*>(q1 + d + 8)) : 0u;
    }
  }

  float acc[DT][4];
#pragma unroll
  for (int i = 0; i < DT; ++i) acc[i][0] = acc[i][1] = acc[i][2] = acc[i][3] = 0.f;
  float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;

  // Per-lane ldmatrix offsets: matrix mi = lane / 8, row r = lane % 8.
  const int mi = lane >> 3, mr = lane & 7;
  const uint32_t k_lane_off = ((mi & 1) * BS + (mi >> 1) * 8 + mr) * 16;   // + (2*ks*BS + np*8) * 16
  const uint32_t v_lane_off = ((mi >> 1) * 8 + mr) * (BS * Sh::kElem) + (mi & 1) * 16;

  for (int i = 0; i < work.my_n; ++i) {
    if (!wait_stage<STAGES>(bars, i, work.my_n, p.err, lane)) break;
    unsigned char* stage = ring + (i % STAGES) * 2 * TILE;
    const int tok0 = work.logical_block(i) * BS;
    const int rem = L - tok0;  // valid tokens in this block (>= 1)
    if (rem < BS) zero_tail_v<T, D, BS>(stage + TILE, rem, lane);
    const uint32_t kb = smem_addr(stage), vb = kb + TILE;

    // S = Q K^T for the block's BS tokens.
    float sc[NT][4];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) sc[nt][0] = sc[nt][1] = sc[nt][2] = sc[nt][3] = 0.f;
#pragma unroll
    for (int ks = 0; ks < KS; ++ks) {
#pragma unroll
      for (int np = 0; np < NT; np += 2) {
        uint32_t b0, b1, b2, b3;
        ldsm_x4(kb + k_lane_off + (2 * ks * BS + np * 8) * 16, b0, b1, b2, b3);
        mma_16816<T>(sc[np], qf[ks], b0, b1);
        mma_16816<T>(sc[np + 1], qf[ks], b2, b3);
      }
    }

    // Online softmax update (log2 domain); tokens past the sequence get -inf.
    float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const int tok = nt * 8 + 2 * t4 + (c & 1);
        const float v = sc[nt][c] * p.scale_log2;
        sc[nt][c] = tok < rem ? v : -INFINITY;
      }
      mx0 = fmaxf(mx0, fmaxf(sc[nt][0], sc[nt][1]));
      mx1 = fmaxf(mx1, fmaxf(sc[nt][2], sc[nt][3]));
    }
    mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
    mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
    mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
    mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
    const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
    const float c0 = exp2f(m0 - mn0), c1 = exp2f(m1 - mn1);
    m0 = mn0;
    m1 = mn1;
    float ps0 = 0.f, ps1 = 0.f;
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      sc[nt][0] = exp2f(sc[nt][0] - mn0);
      sc[nt][1] = exp2f(sc[nt][1] - mn0);
      sc[nt][2] = exp2f(sc[nt][2] - mn1);
      sc[nt][3] = exp2f(sc[nt][3] - mn1);
      ps0 += sc[nt][0] + sc[nt][1];
      ps1 += sc[nt][2] + sc[nt][3];
    }
    l0 = l0 * c0 + ps0;
    l1 = l1 * c1 + ps1;
#pragma unroll
    for (int dt = 0; dt < DT; ++dt) {
      acc[dt][0] *= c0;
      acc[dt][1] *= c0;
      acc[dt][2] *= c1;
      acc[dt][3] *= c1;
    }

    // O += P V, with P = hi + lo in the cache's 16-bit type.
#pragma unroll
    for (int kk = 0; kk < KK; ++kk) {
      uint32_t ahi[4], alo[4];
#pragma unroll
      for (int r = 0; r < 4; ++r) {
        const float* src = sc[2 * kk + (r >> 1)] + (r & 1) * 2;
        ahi[r] = pack2<T>(src[0], src[1]);
        const float2 back = unpack2<T>(ahi[r]);
        alo[r] = pack2<T>(src[0] - back.x, src[1] - back.y);
      }
#pragma unroll
      for (int dp = 0; dp < DT; dp += 2) {
        uint32_t b0, b1, b2, b3;
        ldsm_x4(vb + v_lane_off + dp * 8 * (BS * Sh::kElem) + kk * 32, b0, b1, b2, b3);
        mma_16816<T>(acc[dp], ahi, b0, b1);
        mma_16816<T>(acc[dp + 1], ahi, b2, b3);
        mma_16816<T>(acc[dp], alo, b0, b1);
        mma_16816<T>(acc[dp + 1], alo, b2, b3);
      }
    }

    __syncwarp();
    if (i + STAGES < work.my_n) {
      fence_proxy_async_smem();
      const int phys = tc.phys(work, i + STAGES, lane);
      issue_stage<TILE, STAGES>(ring, bars, p.k_cache, p.v_cache, phys * head_tiles + kvh, i + STAGES, lane);
    }
  }

  // Row sums across the four lanes of a quad.
  l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
  l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
  l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
  l1 += __shfl_xor_sync(0xffffffffu, l1, 2);

  __syncthreads();  // every ring is drained: reuse it for the merge
  float* wo = reinterpret_cast<float*>(smem);                 // [warps][16][D]
  float* wm = wo + kDecodeWarps * 16 * D;                      // [warps][16]
  float* wl = wm + kDecodeWarps * 16;                          // [warps][16]
#pragma unroll
  for (int dt = 0; dt < DT; ++dt) {
    const int d = dt * 8 + 2 * t4;
    *reinterpret_cast<float2*>(wo + (warp * 16 + g) * D + d) = make_float2(acc[dt][0], acc[dt][1]);
    *reinterpret_cast<float2*>(wo + (warp * 16 + g + 8) * D + d) = make_float2(acc[dt][2], acc[dt][3]);
  }
  if (t4 == 0) {
    wm[warp * 16 + g] = m0;
    wm[warp * 16 + g + 8] = m1;
    wl[warp * 16 + g] = l0;
    wl[warp * 16 + g + 8] = l1;
  }
  __syncthreads();
  merge_and_store<T, D>(p, wm, wl, wo, 16, nh, s, h0, part, nparts == 1);
}

// --- CUDA-core kernel --------------------------------------------------------------------------
//
// grid = (num_parts, num_heads, num_seqs); one query head per CTA.
template <typename T, int D, int BS>
__global__ void __launch_bounds__(kDecodeWarps * 32)
    decode_simt_kernel(const DecodeParams p) {
  using Sh = DecodeShape<T, D, BS>;
  constexpr int TILE = Sh::kTile, STAGES = Sh::kStages, X = Sh::kX;
  constexpr int NGH = D / X / 2;         // 16-byte K groups per half-warp
  constexpr int TP = BS / 16;            // 16-token passes per block
  constexpr int CH = BS * Sh::kElem / 16;  // 16-byte chunks per V row
  constexpr int RPW = 32 / CH;           // V rows per warp pass
  constexpr int VP = D / RPW;            // V rows per lane
  static_assert(kDecodeWarps * (D + 2) * 4 <= Sh::kRingBytes, "merge area must fit in the ring");
  extern __shared__ __align__(128) unsigned char smem[];

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int half = lane >> 4, tl = lane & 15;
  const int s = blockIdx.z, part = blockIdx.x, h = blockIdx.y;
  const int kvh = h / p.group;

  const int L = __ldg(p.seq_lens + s);
  if (L < 1 || L > p.max_seq_len) {
    if (part == 0) reject_sequence<T, D>(p, s, h, 1);
    return;
  }
  const int nblk = (L + BS - 1) / BS;
  const int nparts = (nblk + p.part_blocks - 1) / p.part_blocks;
  if (part >= nparts) return;
  WarpWork work;
  work.blk0 = part * p.part_blocks;
  work.warp = warp;
  const int nb_part = min(nblk, work.blk0 + p.part_blocks) - work.blk0;
  work.my_n = nb_part > warp ? (nb_part - warp + kDecodeWarps - 1) / kDecodeWarps : 0;

  unsigned char* ring = smem + warp * STAGES * 2 * TILE;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + Sh::kRingBytes) + warp * STAGES;
  float* pw = reinterpret_cast<float*>(smem + Sh::kRingBytes + Sh::kBarBytes) + warp * BS;
  if (lane == 0) {
    for (int st = 0; st < STAGES; ++st) mbar_init(&bars[st], 1);
    fence_barrier_init();
  }
  __syncwarp();

  TableCursor tc{p.block_tables + (long long)s * p.max_blocks_per_seq, p.num_blocks, p.err, -1, 0};
  const long long head_tiles = p.num_kv_heads;
  for (int i = 0; i < STAGES && i < work.my_n; ++i) {
    const int phys = tc.phys(work, i, lane);
    issue_stage<TILE, STAGES>(ring, bars, p.k_cache, p.v_cache, phys * head_tiles + kvh, i, lane);
  }

  // This half-warp's half of the query row, in fp32.
  float qv[NGH * X];
  {
    const T* q = static_cast<const T*>(p.q) + ((long long)s * p.num_heads + h) * D + half * NGH * X;
#pragma unroll
    for (int k = 0; k < NGH * X; ++k) qv[k] = DType<T>::to_f32(q[k]);
  }

  float acc[VP];
#pragma unroll
  for (int k = 0; k < VP; ++k) acc[k] = 0.f;
  float m = -INFINITY, lpart = 0.f;
  const int vrow = lane / CH, vchunk = lane % CH;

  for (int i = 0; i < work.my_n; ++i) {
    if (!wait_stage<STAGES>(bars, i, work.my_n, p.err, lane)) break;
    unsigned char* stage = ring + (i % STAGES) * 2 * TILE;
    const int tok0 = work.logical_block(i) * BS;
    const int rem = L - tok0;
    if (rem < BS) zero_tail_v<T, D, BS>(stage + TILE, rem, lane);

    // Scores of this lane's token(s): each half-warp covers half of the head dims.
    float sc[TP];
#pragma unroll
    for (int tp = 0; tp < TP; ++tp) {
      const int tok = tp * 16 + tl;
      float dot = 0.f;
#pragma unroll
      for (int gi = 0; gi < NGH; ++gi) {
        const uint4 raw = *reinterpret_cast<const uint4*>(stage + ((half * NGH + gi) * BS + tok) * 16);
        const T* kv = reinterpret_cast<const T*>(&raw);
#pragma unroll
        for (int k = 0; k < X; ++k) dot = fmaf(qv[gi * X + k], DType<T>::to_f32(kv[k]), dot);
      }
      dot += __shfl_xor_sync(0xffffffffu, dot, 16);
      sc[tp] = tok < rem ? dot * p.scale_log2 : -INFINITY;
    }
    float mx = sc[0];
#pragma unroll
    for (int tp = 1; tp < TP; ++tp) mx = fmaxf(mx, sc[tp]);
#pragma unroll
    for (int o = 1; o < 16; o <<= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    const float mn = fmaxf(m, mx);
    const float corr = exp2f(m - mn);
    m = mn;
    float psum = 0.f;
#pragma unroll
    for (int tp = 0; tp < TP; ++tp) {
      sc[tp] = exp2f(sc[tp] - mn);
      psum += sc[tp];
      if (half == 0) pw[tp * 16 + tl] = sc[tp];
    }
    lpart = lpart * corr + (half == 0 ? psum : 0.f);
    __syncwarp();

    // acc[d] += sum_t p_t V[d, t] for this lane's rows and token chunk.
#pragma unroll
    for (int k = 0; k < VP; ++k) {
      const int d = k * RPW + vrow;
      const uint4 raw = *reinterpret_cast<const uint4*>(stage + TILE + d * BS * Sh::kElem + vchunk * 16);
      const T* vv = reinterpret_cast<const T*>(&raw);
      float a = acc[k] * corr;
#pragma unroll
      for (int e = 0; e < X; ++e) a = fmaf(pw[vchunk * X + e], DType<T>::to_f32(vv[e]), a);
      acc[k] = a;
    }

    __syncwarp();
    if (i + STAGES < work.my_n) {
      fence_proxy_async_smem();
      const int phys = tc.phys(work, i + STAGES, lane);
      issue_stage<TILE, STAGES>(ring, bars, p.k_cache, p.v_cache, phys * head_tiles + kvh, i + STAGES, lane);
    }
  }

  // Complete the row sums over the CH lanes of a V row, and l over the warp.
#pragma unroll
  for (int k = 0; k < VP; ++k)
#pragma unroll
    for (int o = 1; o < CH; o <<= 1) acc[k] += __shfl_xor_sync(0xffffffffu, acc[k], o);
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) lpart += __shfl_xor_sync(0xffffffffu, lpart, o);

  __syncthreads();
  float* wo = reinterpret_cast<float*>(smem);   // [warps][D]
  float* wm = wo + kDecodeWarps * D;             // [warps]
  float* wl = wm + kDecodeWarps;                 // [warps]
  if (vchunk == 0) {
#pragma unroll
    for (int k = 0; k < VP; ++k) wo[warp * D + k * RPW + vrow] = acc[k];
  }
  if (lane == 0) {
    wm[warp] = m;
    wl[warp] = lpart;
  }
  __syncthreads();
  merge_and_store<T, D>(p, wm, wl, wo, 1, 1, s, h, part, nparts == 1);
}

// --- merge of partitions -------------------------------------------------------------------------
//
// For every (sequence, head) split into n > 1 partitions with results (m_p, l_p, o_p),
// o_p = acc_p / l_p:  M = max_p m_p,  w_p = l_p * 2^(m_p - M),
// out = sum_p w_p o_p / sum_p w_p.  grid = (num_heads, num_seqs), D threads.
template <typename T, int D>
__global__ void __launch_bounds__(D) decode_merge_kernel(const DecodeParams p) {
  extern __shared__ float wsm[];  // [num_parts] weights, then [32] scratch
  float* red = wsm + p.num_parts;
  const int h = blockIdx.x, s = blockIdx.y, tid = threadIdx.x;
  const int L = __ldg(p.seq_lens + s);
  if (L < 1 || L > p.max_seq_len) return;
  const int nblk = (L + p.block_size - 1) / p.block_size;
  const int np = (nblk + p.part_blocks - 1) / p.part_blocks;
  if (np <= 1) return;
  const long long sh = (long long)s * p.num_heads + h;
  const float* ml = p.part_ml + sh * p.num_parts * 2;
  const float* po = p.part_o + sh * p.num_parts * D;
  const int lane = tid & 31, warp = tid >> 5;
  constexpr int NW = D / 32;

  float M = -INFINITY;
  for (int i = tid; i < np; i += D) M = fmaxf(M, ml[2 * i]);
#pragma unroll
  for (int o = 16; o; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
  if (lane == 0) red[warp] = M;
  __syncthreads();
  M = red[0];
#pragma unroll
  for (int w = 1; w < NW; ++w) M = fmaxf(M, red[w]);
  __syncthreads();

  float lsum = 0.f;
  for (int i = tid; i < np; i += D) {
    const float w = ml[2 * i + 1] * exp2f(ml[2 * i] - M);
    wsm[i] = w;
    lsum += w;
  }
#pragma unroll
  for (int o = 16; o; o >>= 1) lsum += __shfl_xor_sync(0xffffffffu, lsum, o);
  if (lane == 0) red[warp] = lsum;
  __syncthreads();
  lsum = 0.f;
#pragma unroll
  for (int w = 0; w < NW; ++w) lsum += red[w];

  float o = 0.f;
#pragma unroll 8
  for (int i = 0; i < np; ++i) o = fmaf(wsm[i], __ldg(po + (long long)i * D + tid), o);
  static_cast<T*>(p.out)[sh * D + tid] = DType<T>::from_f32(o / lsum);
}

// --- host-side launch helpers (instantiated per dtype) ------------------------------------------

template <typename T, int D, int BS>
constexpr int decode_smem_bytes(DecodeKind kind) {
  using Sh = DecodeShape<T, D, BS>;
  return Sh::kRingBytes + Sh::kBarBytes + (kind == DecodeKind::kSimt ? kDecodeWarps * BS * 4 : 0);
}

template <typename T, int D, int BS>
void* decode_kernel_ptr(DecodeKind kind) {
  if constexpr (sizeof(T) == 4) {
    return reinterpret_cast<void*>(&decode_simt_kernel<T, D, BS>);
  } else {
    return kind == DecodeKind::kMma ? reinterpret_cast<void*>(&decode_mma_kernel<T, D, BS>)
                                    : reinterpret_cast<void*>(&decode_simt_kernel<T, D, BS>);
  }
}

// Opt the kernel in to its dynamic shared memory, once per device.
inline cudaError_t ensure_smem_attr(void* fn, int bytes, unsigned* done_mask) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 32 && (__atomic_load_n(done_mask, __ATOMIC_ACQUIRE) >> dev) & 1u) return cudaSuccess;
  e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess && dev < 32) __atomic_fetch_or(done_mask, 1u << dev, __ATOMIC_RELEASE);
  return e;
}

template <typename T, int D, int BS>
int decode_ctas_per_sm_t(DecodeKind kind) {
  static unsigned done[2] = {0, 0};
  void* fn = decode_kernel_ptr<T, D, BS>(kind);
  const int bytes = decode_smem_bytes<T, D, BS>(kind);
  if (ensure_smem_attr(fn, bytes, &done[static_cast<int>(kind)]) != cudaSuccess) return 0;
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, fn, kDecodeWarps * 32, bytes) != cudaSuccess) return 0;
  return n;
}

template <typename T, int D, int BS>
cudaError_t launch_decode_t(const DecodeParams& p, DecodeKind kind, cudaStream_t stream, int* launches) {
  static unsigned done[2] = {0, 0};
  if (sizeof(T) == 4) kind = DecodeKind::kSimt;
  void* fn = decode_kernel_ptr<T, D, BS>(kind);
  const int bytes = decode_smem_bytes<T, D, BS>(kind);
  cudaError_t e = ensure_smem_attr(fn, bytes, &done[static_cast<int>(kind)]);
  if (e != cudaSuccess) return e;
  const int units = kind == DecodeKind::kMma ? p.num_kv_heads * ((p.group + 15) / 16) : p.num_heads;
  dim3 grid(p.num_parts, units, p.num_seqs);
  void* args[] = {const_cast<DecodeParams*>(&p)};
  e = cudaLaunchKernel(fn, grid, dim3(kDecodeWarps * 32), args, bytes, stream);
  if (e != cudaSuccess) return e;
  *launches = 1;
  if (p.num_parts > 1) {
    const int merge_bytes = (p.num_parts + 32) * 4;
    if (merge_bytes > 48 * 1024) {
      e = cudaFuncSetAttribute(reinterpret_cast<void*>(&decode_merge_kernel<T, D>),
                               cudaFuncAttributeMaxDynamicSharedMemorySize, merge_bytes);
      if (e != cudaSuccess) return e;
    }
    decode_merge_kernel<T, D><<<dim3(p.num_heads, p.num_seqs), D, merge_bytes, stream>>>(p);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    *launches = 2;
  }
  return cudaSuccess;
}

template <typename T>
int decode_ctas_per_sm_dispatch(int head_size, int block_size, DecodeKind kind) {
  if (head_size == 64 && block_size == 16) return decode_ctas_per_sm_t<T, 64, 16>(kind);
  if (head_size == 64 && block_size == 32) return decode_ctas_per_sm_t<T, 64, 32>(kind);
  if (head_size == 128 && block_size == 16) return decode_ctas_per_sm_t<T, 128, 16>(kind);
  if (head_size == 128 && block_size == 32) return decode_ctas_per_sm_t<T, 128, 32>(kind);
  return 0;
}

template <typename T>
cudaError_t launch_decode_dispatch(int head_size, const DecodeParams& p, DecodeKind kind, cudaStream_t s,
                                   int* n) {
  if (head_size == 64 && p.block_size == 16) return launch_decode_t<T, 64, 16>(p, kind, s, n);
  if (head_size == 64 && p.block_size == 32) return launch_decode_t<T, 64, 32>(p, kind, s, n);
  if (head_size == 128 && p.block_size == 16) return launch_decode_t<T, 128, 16>(p, kind, s, n);
  if (head_size == 128 && p.block_size == 32) return launch_decode_t<T, 128, 32>(p, kind, s, n);
  return cudaErrorInvalidValue;
}

}  // namespace pa
