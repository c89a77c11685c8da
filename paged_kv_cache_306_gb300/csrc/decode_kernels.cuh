// decode_kernels.cuh -- paged-attention decode kernels for sm_103a.
//
// What is computed ("Reading vLLM's PagedAttention kernel", §2 flowchart, §3.3,
// §3.4): for a sequence s and the query heads that share a kv head, walk the
// sequence's block-table row in logical order; for each logical block look up the
// physical block, bring its K tile and V tile in, compute the scaled scores q.K^T,
// fold them into a running (max m, normaliser l, accumulator acc) online softmax,
// and finish with acc / l.  A run of blocks processed on its own produces
// (m, l, acc / l); runs of one sequence are merged with
//     M = max m_p,  w_p = l_p 2^(m_p - M),  out = sum_p w_p o_p / sum_p w_p
// -- the split-and-merge the pages describe for PARTITION_SIZE (§3.3).
//
// How the work maps to the GB300:
//   * Persistent, load-balanced ("stream-K") schedule.  A segment is one
//     (sequence, head unit) pair and its blocks; all segments laid end to end form
//     T blocks of work.  The grid holds exactly the resident CTAs; each of their
//     warps is an independent worker that takes one contiguous range of T / W
//     blocks (W = warps in the grid), crossing segment boundaries.  Every warp thus
//     streams the same number of blocks from start to finish with its pipeline
//     full: no per-CTA ramp-up, no tail wave, no idle SMs on ragged batches.
//     A segment cut by a warp boundary leaves pieces whose (m, l, acc / l) go to
//     partial slots; a second kernel merges them.  A segment done wholly by one
//     warp is written straight to the output.  Caller partitions (PARTITION_SIZE)
//     that end inside a warp's piece are merged into the piece at once with the
//     same formula, through a running state in shared memory.
//   * Each warp owns a STAGES-deep ring of shared-memory stages.  A stage holds the
//     K tile and the V tile of one (physical block, kv head); in this pool layout
//     both are contiguous runs of head_size * block_size elements, so each is one
//     1-D bulk copy through the TMA unit (cp.async.bulk) that signals an mbarrier
//     with its byte count.  Block-table entries for the next 32 blocks are fetched
//     one group ahead, one lane per entry, so the table walk never stalls the ring.
//   * Tensor-core math (16-bit caches, >= 2 query heads per kv head): the query
//     heads of one kv head are the rows of m16n8k16 tiles, so one K/V read serves
//     all of them.  S = Q K^T takes K straight from the stage with ldmatrix (a
//     K-pool row of 8 dims is 16 B); P V takes V the same way (a V-pool row holds 8
//     consecutive tokens per 16 B).  P stays in registers, split into a rounded
//     16-bit high part and the rounded remainder so P V keeps ~16 significant bits.
//   * CUDA-core math (fp32 caches, or one query head per kv head): half-warps split
//     the head dims of the scores, lanes split V rows and token chunks for P V, and
//     the reductions are warp shuffles.
//   * Programmatic dependent launch (see pa_device.cuh): the decode kernel becomes
//     resident while the write-path kernel before it finishes, and the merge kernel
//     while the decode kernel finishes.
#pragma once

#include <math.h>

#include <type_traits>

#include "pa_device.cuh"
#include "pa_launch.h"

namespace pa {

constexpr uint64_t kWaitLimitNs = 1000000000ull;  // 1 s, then PA_DEVERR_TIMEOUT

template <typename T, int D, int BS>
struct DecodeShape {
  static constexpr int kElem = sizeof(T);
  static constexpr int kX = 16 / kElem;         // elements per 16-byte K group
  static constexpr int kTile = D * BS * kElem;  // bytes of one K (or V) tile
  static constexpr int kWarps = decode_warps(2 * kTile);
  static constexpr int kStages = decode_stages(2 * kTile);
  static constexpr int kRingBytes = kWarps * kStages * 2 * kTile;
  static constexpr int kBarBytes = kWarps * kStages * 8;
  // per-sequence tables: lengths, block prefix, warp sums
  static constexpr int kTableBytes = (kMaxSeqsPerLaunch + (kMaxSeqsPerLaunch + 1) + kWarps + 3) * 4;
};

// Wait for block i's stage.  On timeout record the error and drain the copies
// still in flight (each with its own bounded wait) so none lands after exit.
template <int STAGES>
__device__ __forceinline__ bool wait_stage(uint64_t* bars, int i, int n, unsigned* err, int lane) {
  const int st = i % STAGES;
  const bool ok = __all_sync(0xffffffffu, mbar_wait_bounded(&bars[st], (i / STAGES) & 1, kWaitLimitNs));
  if (!ok) {
    if (lane == 0) set_error(err, kErrTimeout);
    for (int j = i + 1; j < n && j < i + STAGES; ++j)
      mbar_wait_bounded(&bars[j % STAGES], (j / STAGES) & 1, kWaitLimitNs / 8);
  }
  return ok;
}

// Zero the V columns of tokens >= rem in a stage (only a sequence's last, partial
// block): those slots may hold anything, and 0 * NaN would poison the sum.
template <typename T, int D, int BS>
__device__ __forceinline__ void zero_tail_v(unsigned char* vtile, int rem, int lane) {
  T* v = reinterpret_cast<T*>(vtile);
  for (int idx = lane; idx < D * BS; idx += 32)
    if ((idx % BS) >= rem) v[idx] = DType<T>::from_f32(0.f);
  __syncwarp();
}

// --- per-warp math: tensor cores ---------------------------------------------------------------
//
// Up to 16 query rows (the heads of one head unit) against the tokens of a block.
//
// T is the query / output type and the type of the tensor-core operands; TC is
// the cache element type: T itself, or FP8 E4M3 (converted to T in registers).
// For an FP8 cache, ldmatrix over 16-byte rows hands each thread 4 consecutive
// codes, which must become the (k, k+1) and (k+8, k+9) operand pairs of the MMA:
// the head dims of Q are permuted to match within each 16-dim k-step, and the
// tokens of S's n-tiles are permuted so that P's fragments line up with V's.
template <typename T, typename TC, int D, int BS>
struct MmaMath {
  static constexpr int NT = BS / 8;   // token n-tiles of S
  static constexpr int KS = D / 16;   // k-steps over head dims for S
  static constexpr int DT = D / 8;    // head-dim n-tiles of O
  static constexpr int KK = BS / 16;  // token k-steps for O
  static constexpr int kElem = sizeof(TC);
  static constexpr bool kFp8 = sizeof(TC) == 1;

  // Token of column col (0..7) of S n-tile nt.
  __device__ __forceinline__ static int token(int nt, int col) {
    return kFp8 ? 16 * (nt >> 1) + 4 * (col >> 1) + (col & 1) + 2 * (nt & 1) : nt * 8 + col;
  }

  uint32_t qf[KS][4];
  float acc[DT][4];
  float m0, m1, l0, l1;
  uint32_t k_lane_off, v_lane_off;
  int g, t4;

  __device__ __forceinline__ void init(int lane, float*) {
    g = lane >> 2;
    t4 = lane & 3;
    const int mi = lane >> 3, mr = lane & 7;  // ldmatrix: matrix mi, row mr
    if (kFp8) {
      // K: matrix mi = (k-step mi & 1, n-tile mi >> 1), rows = that n-tile's tokens
      k_lane_off = ((mi & 1) * BS + token(mi >> 1, mr)) * 16;
      // V: matrix mi = head-dim n-tile mi, rows = 8 head dims of 16 tokens (16 bytes)
      v_lane_off = (mi * 8 + mr) * BS;
    } else {
      k_lane_off = ((mi & 1) * BS + (mi >> 1) * 8 + mr) * 16;
      v_lane_off = ((mi >> 1) * 8 + mr) * (BS * kElem) + (mi & 1) * 16;
    }
  }

  __device__ __forceinline__ void reset() {
#pragma unroll
    for (int i = 0; i < DT; ++i) acc[i][0] = acc[i][1] = acc[i][2] = acc[i][3] = 0.f;
    m0 = m1 = -INFINITY;
    l0 = l1 = 0.f;
  }

  // A-operand fragments of rows 0..nh-1 of q (row stride D), zero past nh.
  __device__ __forceinline__ void load_q(const T* q, int nh) {
    const T* q0 = q + g * D;
    const T* q1 = q0 + 8 * D;
    const bool v0 = g < nh, v1 = g + 8 < nh;
#pragma unroll
    for (int ks = 0; ks < KS; ++ks) {
      // operand k = 2t4, 2t4+1 and 2t4+8, 2t4+9 read head dims d, d+1 and d2, d2+1
      const int d = ks * 16 + (kFp8 ? 4 * t4 : 2 * t4);
      const int d2 = kFp8 ? d + 2 : d + 8;
      qf[ks][0] = v0 ? __ldg(reinterpret_cast<const unsigned int*>(q0 + d)) : 0u;
      qf[ks][1] = v1 ? __ldg(reinterpret_cast<const unsigned int*>(q1 + d)) : 0u;
      qf[ks][2] = v0 ? __ldg(reinterpret_cast<const unsigned int*>(q0 + d2)) : 0u;
      qf[ks][3] = v1 ? __ldg(reinterpret_cast<const unsigned int*>(q1 + d2)) : 0u;
    }
  }

  __device__ __forceinline__ void block(unsigned char* stage, int tile_bytes, int rem, float scale_log2) {
    const uint32_t kb = smem_addr(stage), vb = kb + tile_bytes;
    // S = Q K^T for the block's BS tokens.
    float sc[NT][4];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) sc[nt][0] = sc[nt][1] = sc[nt][2] = sc[nt][3] = 0.f;
    if constexpr (kFp8) {
#pragma unroll
      for (int kp = 0; kp < KS / 2; ++kp) {
#pragma unroll
        for (int np = 0; np < NT; np += 2) {
          uint32_t r[4];  // (k-step 2kp, n-tile np), (2kp+1, np), (2kp, np+1), (2kp+1, np+1)
          ldsm_x4(kb + k_lane_off + (2 * kp * BS + np * 8) * 16, r[0], r[1], r[2], r[3]);
#pragma unroll
          for (int i = 0; i < 4; ++i)
            mma_16816<T>(sc[np + (i >> 1)], qf[2 * kp + (i & 1)], e4m3x2_to<T>(r[i] & 0xffffu),
                         e4m3x2_to<T>(r[i] >> 16));
        }
      }
    } else {
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
    }
    // Online softmax update (log2 domain); tokens past the sequence get -inf.
    float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const int tok = token(nt, 2 * t4 + (c & 1));
        const float v = sc[nt][c] * scale_log2;
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
      if constexpr (kFp8) {
#pragma unroll
        for (int dp = 0; dp < DT; dp += 4) {
          uint32_t r[4];  // head-dim n-tiles dp .. dp+3, tokens 16kk .. 16kk+15
          ldsm_x4(vb + v_lane_off + dp * 8 * BS + kk * 16, r[0], r[1], r[2], r[3]);
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const uint32_t b0 = e4m3x2_to<T>(r[i] & 0xffffu), b1 = e4m3x2_to<T>(r[i] >> 16);
            mma_16816<T>(acc[dp + i], ahi, b0, b1);
            mma_16816<T>(acc[dp + i], alo, b0, b1);
          }
        }
      } else {
#pragma unroll
        for (int dp = 0; dp < DT; dp += 2) {
          uint32_t b0, b1, b2, b3;
          ldsm_x4(vb + v_lane_off + dp * 8 * (BS * kElem) + kk * 32, b0, b1, b2, b3);
          mma_16816<T>(acc[dp], ahi, b0, b1);
          mma_16816<T>(acc[dp + 1], ahi, b2, b3);
          mma_16816<T>(acc[dp], alo, b0, b1);
          mma_16816<T>(acc[dp + 1], alo, b2, b3);
        }
      }
    }
  }

  // Complete the row sums across the four lanes of a quad.
  __device__ __forceinline__ void finish() {
    l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
    l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
    l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
    l1 += __shfl_xor_sync(0xffffffffu, l1, 2);
  }

  // out rows 0..nh-1 (row stride D) = oscale * acc / l, rounded to T.
  __device__ __forceinline__ void store_out(T* out, int nh, float oscale) const {
    const float i0 = oscale / l0, i1 = oscale / l1;
    const bool v0 = g < nh, v1 = g + 8 < nh;
#pragma unroll
    for (int dt = 0; dt < DT; ++dt) {
      const int d = dt * 8 + 2 * t4;
      if (v0) *reinterpret_cast<uint32_t*>(out + g * D + d) = pack2<T>(acc[dt][0] * i0, acc[dt][1] * i0);
      if (v1) *reinterpret_cast<uint32_t*>(out + (g + 8) * D + d) = pack2<T>(acc[dt][2] * i1, acc[dt][3] * i1);
    }
  }

  // Partial result of rows 0..nh-1: o = oscale * acc / l (fp32, row stride D), (m, l).
  __device__ __forceinline__ void store_partial(float* po, float* pml, int nh, float oscale) const {
    const float i0 = oscale / l0, i1 = oscale / l1;
    const bool v0 = g < nh, v1 = g + 8 < nh;
#pragma unroll
    for (int dt = 0; dt < DT; ++dt) {
      const int d = dt * 8 + 2 * t4;
      if (v0) *reinterpret_cast<float2*>(po + g * D + d) = make_float2(acc[dt][0] * i0, acc[dt][1] * i0);
      if (v1) *reinterpret_cast<float2*>(po + (g + 8) * D + d) = make_float2(acc[dt][2] * i1, acc[dt][3] * i1);
    }
    if (t4 == 0) {
      if (v0) *reinterpret_cast<float2*>(pml + 2 * g) = make_float2(m0, l0);
      if (v1) *reinterpret_cast<float2*>(pml + 2 * (g + 8)) = make_float2(m1, l1);
    }
  }

  // Merge this partition's result (m, l, o = acc / l) into the warp's running
  // state (M, W, O) in shared memory: M' = max(M, m), O' = O 2^(M - M') + l 2^(m - M') o,
  // W' = W 2^(M - M') + l 2^(m - M').  so: [16][D], sml: [16][2].
  __device__ __forceinline__ void fold(float* so, float* sml, bool first) const {
    float M[2], Wt[2];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      M[h] = first ? -INFINITY : sml[2 * (g + 8 * h)];
      Wt[h] = first ? 0.f : sml[2 * (g + 8 * h) + 1];
    }
    __syncwarp();
    const float mp[2] = {m0, m1}, lp[2] = {l0, l1};
    float fo[2], fp[2];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const float mn = fmaxf(M[h], mp[h]);
      fo[h] = exp2f(M[h] - mn);
      fp[h] = exp2f(mp[h] - mn);  // l 2^(m - M') times o = acc / l
      if (t4 == 0) *reinterpret_cast<float2*>(sml + 2 * (g + 8 * h)) = make_float2(mn, Wt[h] * fo[h] + lp[h] * exp2f(mp[h] - mn));
    }
#pragma unroll
    for (int dt = 0; dt < DT; ++dt) {
      const int d = dt * 8 + 2 * t4;
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        float2* o = reinterpret_cast<float2*>(so + (g + 8 * h) * D + d);
        const float2 old = first ? make_float2(0.f, 0.f) : *o;
        *o = make_float2(old.x * fo[h] + fp[h] * acc[dt][2 * h], old.y * fo[h] + fp[h] * acc[dt][2 * h + 1]);
      }
    }
    __syncwarp();
  }

  // Take the running state as this piece's (m, l, acc): acc = O, l = W.
  __device__ __forceinline__ void load_state(const float* so, const float* sml) {
    m0 = sml[2 * g];
    l0 = sml[2 * g + 1];
    m1 = sml[2 * (g + 8)];
    l1 = sml[2 * (g + 8) + 1];
#pragma unroll
    for (int dt = 0; dt < DT; ++dt) {
      const int d = dt * 8 + 2 * t4;
      const float2 a = *reinterpret_cast<const float2*>(so + g * D + d);
      const float2 b = *reinterpret_cast<const float2*>(so + (g + 8) * D + d);
      acc[dt][0] = a.x;
      acc[dt][1] = a.y;
      acc[dt][2] = b.x;
      acc[dt][3] = b.y;
    }
    __syncwarp();
  }
};

// --- per-warp math: CUDA cores --------------------------------------------------------------------
//
// One query row against the tokens of a block.
template <typename T, typename TC, int D, int BS>
struct SimtMath {
  static constexpr int kElem = sizeof(TC);
  static constexpr int X = 16 / kElem;
  static constexpr int NGH = D / X / 2;        // 16-byte K groups per half-warp
  static constexpr int TP = BS / 16;           // 16-token passes per block
  static constexpr int CH = BS * kElem / 16;   // 16-byte chunks per V row
  static constexpr int RPW = 32 / CH;          // V rows per warp pass
  static constexpr int VP = D / RPW;           // V rows per lane

  float qv[NGH * X];
  float acc[VP];
  float m, lpart;
  float* pw;  // this warp's BS probabilities in shared memory
  int lane, half, tl, vrow, vchunk;

  __device__ __forceinline__ void init(int lane_, float* pw_) {
    lane = lane_;
    half = lane >> 4;
    tl = lane & 15;
    vrow = lane / CH;
    vchunk = lane % CH;
    pw = pw_;
  }

  __device__ __forceinline__ void reset() {
#pragma unroll
    for (int k = 0; k < VP; ++k) acc[k] = 0.f;
    m = -INFINITY;
    lpart = 0.f;
  }

  __device__ __forceinline__ void load_q(const T* q, int) {
    const T* qh = q + half * NGH * X;
#pragma unroll
    for (int k = 0; k < NGH * X; ++k) qv[k] = DType<T>::to_f32(qh[k]);
  }

  __device__ __forceinline__ void block(unsigned char* stage, int tile_bytes, int rem, float scale_log2) {
    // Scores of this lane's token(s); each half-warp covers half of the head dims.
    float sc[TP];
#pragma unroll
    for (int tp = 0; tp < TP; ++tp) {
      const int tok = tp * 16 + tl;
      float dot = 0.f;
#pragma unroll
      for (int gi = 0; gi < NGH; ++gi) {
        const uint4 raw = *reinterpret_cast<const uint4*>(stage + ((half * NGH + gi) * BS + tok) * 16);
        const TC* kv = reinterpret_cast<const TC*>(&raw);
#pragma unroll
        for (int k = 0; k < X; ++k) dot = fmaf(qv[gi * X + k], DType<TC>::to_f32(kv[k]), dot);
      }
      dot += __shfl_xor_sync(0xffffffffu, dot, 16);
      sc[tp] = tok < rem ? dot * scale_log2 : -INFINITY;
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
    const unsigned char* vt = stage + tile_bytes;
#pragma unroll
    for (int k = 0; k < VP; ++k) {
      const int d = k * RPW + vrow;
      const uint4 raw = *reinterpret_cast<const uint4*>(vt + d * BS * kElem + vchunk * 16);
      const TC* vv = reinterpret_cast<const TC*>(&raw);
      float a = acc[k] * corr;
#pragma unroll
      for (int e = 0; e < X; ++e) a = fmaf(pw[vchunk * X + e], DType<TC>::to_f32(vv[e]), a);
      acc[k] = a;
    }
    __syncwarp();
  }

  // Row sums over the CH lanes of a V row; l over the warp.
  __device__ __forceinline__ void finish() {
#pragma unroll
    for (int k = 0; k < VP; ++k)
#pragma unroll
      for (int o = 1; o < CH; o <<= 1) acc[k] += __shfl_xor_sync(0xffffffffu, acc[k], o);
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) lpart += __shfl_xor_sync(0xffffffffu, lpart, o);
  }

  __device__ __forceinline__ void store_out(T* out, int, float oscale) const {
    if (vchunk == 0) {
      const float il = oscale / lpart;
#pragma unroll
      for (int k = 0; k < VP; ++k) out[k * RPW + vrow] = DType<T>::from_f32(acc[k] * il);
    }
  }

  __device__ __forceinline__ void store_partial(float* po, float* pml, int, float oscale) const {
    if (vchunk == 0) {
      const float il = oscale / lpart;
#pragma unroll
      for (int k = 0; k < VP; ++k) po[k * RPW + vrow] = acc[k] * il;
    }
    if (lane == 0) *reinterpret_cast<float2*>(pml) = make_float2(m, lpart);
  }

  // As MmaMath::fold, for one row (after finish()): so: [D], sml: [2].
  __device__ __forceinline__ void fold(float* so, float* sml, bool first) const {
    const float M = first ? -INFINITY : sml[0], Wt = first ? 0.f : sml[1];
    __syncwarp();
    const float mn = fmaxf(M, m);
    const float fo = exp2f(M - mn), fp = exp2f(m - mn), e = lpart * fp;
    if (lane == 0) *reinterpret_cast<float2*>(sml) = make_float2(mn, Wt * fo + e);
    if (vchunk == 0) {
#pragma unroll
      for (int k = 0; k < VP; ++k) {
        float* o = so + k * RPW + vrow;
        *o = (first ? 0.f : *o) * fo + fp * acc[k];
      }
    }
    __syncwarp();
  }

  __device__ __forceinline__ void load_state(const float* so, const float* sml) {
    m = sml[0];
    lpart = sml[1];
#pragma unroll
    for (int k = 0; k < VP; ++k) acc[k] = so[k * RPW + vrow];
    __syncwarp();
  }
};

// --- the schedule ---------------------------------------------------------------------------------

// Head unit u of a sequence: its kv head, first query head and query-row count.
template <bool kMma>
__device__ __forceinline__ void unit_heads(const DecodeParams& p, int u, int& kvh, int& h0, int& nh) {
  if (kMma) {
    const int per = (p.group + 15) >> 4;
    kvh = u / per;
    h0 = kvh * p.group + (u - kvh * per) * 16;
    nh = min(16, kvh * p.group + p.group - h0);
  } else {
    kvh = u / p.group;
    h0 = u;
    nh = 1;
  }
}

// Segment and block of global work position g (g < T): the sequence s with
// units * pre[s] <= g < units * pre[s + 1] (empty sequences are skipped because
// their prefix equals the next one's), then the unit and the block within it.
__device__ __forceinline__ void locate(long long g, const int* pre, int S, int U, int& s, int& u, int& j) {
  int lo = 0, hi = S - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if ((long long)pre[mid] * U <= g) lo = mid;
    else hi = mid - 1;
  }
  s = lo;
  const int nb = pre[s + 1] - pre[s];
  const long long r = g - (long long)pre[s] * U;
  u = static_cast<int>(r / nb);
  j = static_cast<int>(r - (long long)u * nb);
}

// grid = resident CTAs (persistent); kDecodeWarps independent warps per CTA.
template <typename T, typename TC, int D, int BS, bool kMma>
__global__ void __launch_bounds__(DecodeShape<TC, D, BS>::kWarps * 32)
    decode_kernel(const DecodeParams p) {
  using Sh = DecodeShape<TC, D, BS>;
  constexpr int kDecodeWarps = Sh::kWarps;
  using Math = std::conditional_t<kMma, MmaMath<T, TC, D, BS>, SimtMath<T, TC, D, BS>>;
  constexpr int TILE = Sh::kTile, STAGES = Sh::kStages;
  extern __shared__ __align__(128) unsigned char smem[];

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  unsigned char* ring = smem + warp * STAGES * 2 * TILE;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + Sh::kRingBytes) + warp * STAGES;
  int* s_len = reinterpret_cast<int*>(smem + Sh::kRingBytes + Sh::kBarBytes);
  int* s_pre = s_len + kMaxSeqsPerLaunch;                 // [S + 1] block prefix per unit
  int* s_wsum = s_pre + kMaxSeqsPerLaunch + 1;             // [warps]
  float* pw = reinterpret_cast<float*>(smem + Sh::kRingBytes + Sh::kBarBytes + Sh::kTableBytes) + warp * BS;
  // running state of this warp's piece across caller partitions (see fold)
  constexpr int kRows = kMma ? 16 : 1;
  float* st_o = reinterpret_cast<float*>(smem + Sh::kRingBytes + Sh::kBarBytes + Sh::kTableBytes) +
                kDecodeWarps * BS + warp * kRows * (D + 2);
  float* st_ml = st_o + kRows * D;

  if (lane == 0) {
    for (int st = 0; st < STAGES; ++st) mbar_init(&bars[st], 1);
    fence_barrier_init();
  }
  __syncwarp();
  griddep_launch_dependents();
  griddep_wait();  // every input may come from the previous kernel in the stream

  // Per-sequence tables: length (0 when outside [1, max_seq_len]) and prefix sums
  // of blocks.  Each thread scans PER consecutive sequences.
  const int S = p.num_seqs, U = p.units, PB = p.part_blocks;
  {
    constexpr int PER = (kMaxSeqsPerLaunch + kDecodeWarps * 32 - 1) / (kDecodeWarps * 32);
    int nb[PER], sb = 0;
#pragma unroll
    for (int k = 0; k < PER; ++k) {
      const int i = tid * PER + k;
      int L = i < S ? __ldg(p.seq_lens + i) : 0;
      if (L < 1 || L > p.max_seq_len) L = 0;
      if (i < S) s_len[i] = L;
      nb[k] = (L + BS - 1) / BS;
      sb += nb[k];
    }
    int ib = sb;  // inclusive warp scan
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int xb = __shfl_up_sync(0xffffffffu, ib, o);
      if (lane >= o) ib += xb;
    }
    if (lane == 31) s_wsum[warp] = ib;
    __syncthreads();
    int ob = ib - sb;
    for (int w = 0; w < warp; ++w) ob += s_wsum[w];
#pragma unroll
    for (int k = 0; k < PER; ++k) {
      const int i = tid * PER + k;
      if (i <= S) s_pre[i] = ob;
      ob += nb[k];
    }
    if (tid == blockDim.x - 1) s_pre[S] = ob;  // the total (also covers S == kMaxSeqsPerLaunch)
    __syncthreads();
  }

  // Sequences outside the contract: record the error, zero their rows, mark their
  // segments as needing no merge.  One CTA does it.
  if (blockIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      if (s_len[s] != 0) continue;
      if (tid == 0) set_error(p.err, kErrSeqLen);
      T* out = static_cast<T*>(p.out) + (long long)s * p.num_heads * D;
      for (int i = tid; i < p.num_heads * D; i += blockDim.x) out[i] = DType<T>::from_f32(0.f);
      for (int u = tid; u < U; u += blockDim.x) p.seg_first[s * U + u] = -1;
    }
  }

  // This warp's range of the T blocks of work.
  const long long T_all = (long long)s_pre[S] * U;
  const int W = gridDim.x * kDecodeWarps;
  const int w = blockIdx.x * kDecodeWarps + warp;
  const long long qt = T_all / W, rt = T_all % W;
  const long long start = w * qt + (w * rt) / W;
  const long long end = (w + 1) * qt + ((w + 1) * rt) / W;
  const int len = static_cast<int>(end - start);
  if (len <= 0) return;

  // Table lookups: lane i resolves work position start + 32 * group + i.
  const int32_t* __restrict__ bt = p.block_tables;
  auto fetch = [&](int group, int& phys, int& kvh) {
    const long long gpos = start + 32LL * group + lane;
    phys = 0;
    kvh = 0;
    if (gpos < end) {
      int s, u, j, h0, nh;
      locate(gpos, s_pre, S, U, s, u, j);
      unit_heads<kMma>(p, u, kvh, h0, nh);
      phys = __ldg(bt + (long long)s * p.max_blocks_per_seq + j);
    }
  };
  int phys_cur, kvh_cur, phys_nxt, kvh_nxt, group_cur = 0;
  fetch(0, phys_cur, kvh_cur);
  fetch(1, phys_nxt, kvh_nxt);
  auto issue = [&](int k) {
    if ((k >> 5) != group_cur) {
      phys_cur = phys_nxt;
      kvh_cur = kvh_nxt;
      ++group_cur;
      fetch(group_cur + 1, phys_nxt, kvh_nxt);
    }
    int phys = __shfl_sync(0xffffffffu, phys_cur, k & 31);
    const int kvh = __shfl_sync(0xffffffffu, kvh_cur, k & 31);
    if (phys < 0 || phys >= p.num_blocks) {  // out-of-pool entry: record it, read block 0 instead
      if (lane == 0) set_error(p.err, kErrBlockId);
      phys = 0;
    }
    if (lane == 0) {
      const int st = k % STAGES;
      unsigned char* dst = ring + st * 2 * TILE;
      const long long tile = (long long)phys * p.num_kv_heads + kvh;
      mbar_arrive_expect_tx(&bars[st], 2 * TILE);
      bulk_copy_g2s(dst, static_cast<const unsigned char*>(p.k_cache) + tile * TILE, TILE, &bars[st]);
      bulk_copy_g2s(dst + TILE, static_cast<const unsigned char*>(p.v_cache) + tile * TILE, TILE, &bars[st]);
    }
  };
  for (int k = 0; k < STAGES && k < len; ++k) issue(k);

  // The compute cursor walks the same positions in order.
  Math math;
  math.init(lane, pw);
  int cs, cu, cj;
  locate(start, s_pre, S, U, cs, cu, cj);
  int L = 0, nblk = 0, kvh = 0, h0 = 0, nh = 0, seg = 0, j0 = cj;
  bool folded = false;  // earlier partitions of this piece are in the running state
  auto enter = [&]() {
    L = s_len[cs];
    nblk = s_pre[cs + 1] - s_pre[cs];
    unit_heads<kMma>(p, cu, kvh, h0, nh);
    seg = cs * U + cu;
    math.reset();
    math.load_q(static_cast<const T*>(p.q) + ((long long)cs * p.num_heads + h0) * D, nh);
  };
  enter();

  for (int k = 0; k < len; ++k) {
    if (!wait_stage<STAGES>(bars, k, len, p.err, lane)) break;
    unsigned char* stage = ring + (k % STAGES) * 2 * TILE;
    const int rem = L - cj * BS;  // valid tokens in this block (>= 1)
    if (rem < BS) zero_tail_v<TC, D, BS>(stage + TILE, rem, lane);
    math.block(stage, TILE, rem, p.scale_log2);
    ++cj;
    const bool seg_end = cj == nblk, last = k + 1 == len;
    if (seg_end || last) {  // the end of a piece
      math.finish();
      if (folded) {  // close the last caller partition and take the merged state
        math.fold(st_o, st_ml, false);
        math.load_state(st_o, st_ml);
        folded = false;
      }
      if (j0 == 0 && seg_end) {  // the whole segment: straight to the output
        math.store_out(static_cast<T*>(p.out) + ((long long)cs * p.num_heads + h0) * D, nh, p.out_scale);
        if (lane == 0) p.seg_first[seg] = -1;
      } else {
        // pieces start only at warp and segment boundaries, so this slot is unique
        const long long slot = (long long)w + seg;
        math.store_partial(p.part_o + slot * p.rows * D, p.part_ml + slot * p.rows * 2, nh, p.out_scale);
        if (lane == 0) {
          p.part_tag[slot] = make_int2(seg, static_cast<int>(p.epoch));
          if (j0 == 0) p.seg_first[seg] = static_cast<int>(slot);
          if (seg_end) p.seg_last[seg] = static_cast<int>(slot);
        }
      }
      if (!last) {
        if (++cu == U) {
          cu = 0;
          do {
            ++cs;
          } while (s_pre[cs + 1] == s_pre[cs]);
        }
        cj = 0;
        enter();
        j0 = 0;
      }
    } else if (cj % PB == 0) {  // a caller partition ends inside this piece: fold it
      math.finish();
      math.fold(st_o, st_ml, !folded);
      folded = true;
      math.reset();
    }
    __syncwarp();
    if (k + STAGES < len) {
      fence_proxy_async_smem();
      issue(k + STAGES);
    }
  }
}

// --- merge of pieces --------------------------------------------------------------------------------
//
// One CTA per segment (sequence, head unit).  Each query row of the segment gets
// g = 8 / rows warps (at least one); the warps of a row split its pieces 32 at a
// time: lanes take pieces for the maximum and the weights, then every lane owns
// D/32 head dims and sums the weighted partial outputs, with the loads of
// consecutive pieces in flight together.  The g warps of a row combine through
// shared memory.
constexpr int kMergeWarps = 8;

template <typename T, int D, bool kMma>
__global__ void __launch_bounds__(kMergeWarps * 32) decode_merge_kernel(const DecodeParams p) {
  constexpr int CPL = D / 32;  // head dims per lane
  __shared__ float s_m[kMergeWarps], s_l[kMergeWarps];
  __shared__ float s_o[kMergeWarps][D];
  griddep_wait();
  griddep_launch_dependents();
  const int seg = blockIdx.x;
  const int first = p.seg_first[seg], last = p.seg_last[seg];
  if (first < 0 || last < first || last >= p.num_slots) return;  // no merge (or an aborted launch)
  const int s = seg / p.units, u = seg - s * p.units;
  int kvh, h0, nh;
  unit_heads<kMma>(p, u, kvh, h0, nh);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int K = last - first + 1, ep = static_cast<int>(p.epoch);
  const int g = nh >= kMergeWarps ? 1 : kMergeWarps / nh;  // warps per row
  const int per_round = kMergeWarps / g;                     // rows per round
  const int j = warp % g, lead = warp - j;

  for (int r0 = 0; r0 < nh; r0 += per_round) {
    const int r = r0 + warp / g;
    const bool active = warp < per_round * g && r < nh;
    // the maximum over the row's valid pieces
    float M = -INFINITY;
    if (active) {
      for (int i = j * 32 + lane; i < K; i += g * 32) {
        const long long sl = first + i;
        const int2 tag = p.part_tag[sl];
        const float m = p.part_ml[(sl * p.rows + r) * 2];
        if (tag.x == seg && tag.y == ep) M = fmaxf(M, m);
      }
    }
#pragma unroll
    for (int o = 16; o; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
    if (g > 1) {
      if (lane == 0) s_m[warp] = M;
      __syncthreads();
      for (int jj = 0; jj < g; ++jj) M = fmaxf(M, s_m[lead + jj]);
    }
    // weights (lane i holds piece c0 + i) and the weighted sum of the partial outputs
    float lsum = 0.f, acc[CPL];
#pragma unroll
    for (int c = 0; c < CPL; ++c) acc[c] = 0.f;
    if (active) {
      for (int c0 = j * 32; c0 < K; c0 += g * 32) {
        float wgt = 0.f;
        if (c0 + lane < K) {
          const long long sl = first + c0 + lane;
          const int2 tag = p.part_tag[sl];
          const float2 ml = *reinterpret_cast<const float2*>(p.part_ml + (sl * p.rows + r) * 2);
          if (tag.x == seg && tag.y == ep) wgt = ml.y * exp2f(ml.x - M);
        }
        lsum += wgt;
        const int n = min(32, K - c0);
#pragma unroll 8
        for (int i = 0; i < n; ++i) {
          const float wi = __shfl_sync(0xffffffffu, wgt, i);
          if (wi != 0.f) {  // slots of other launches or segments have weight 0 and are never read
            const float* po = p.part_o + ((long long)(first + c0 + i) * p.rows + r) * D + lane * CPL;
            if constexpr (CPL == 4) {
              const float4 v = *reinterpret_cast<const float4*>(po);
              acc[0] = fmaf(wi, v.x, acc[0]);
              acc[1] = fmaf(wi, v.y, acc[1]);
              acc[2] = fmaf(wi, v.z, acc[2]);
              acc[3] = fmaf(wi, v.w, acc[3]);
            } else {
              const float2 v = *reinterpret_cast<const float2*>(po);
              acc[0] = fmaf(wi, v.x, acc[0]);
              acc[1] = fmaf(wi, v.y, acc[1]);
            }
          }
        }
      }
    }
#pragma unroll
    for (int o = 16; o; o >>= 1) lsum += __shfl_xor_sync(0xffffffffu, lsum, o);
    if (g > 1) {
      if (lane == 0) s_l[warp] = lsum;
#pragma unroll
      for (int c = 0; c < CPL; ++c) s_o[warp][lane * CPL + c] = acc[c];
      __syncthreads();
      if (j == 0) {
        for (int jj = 1; jj < g; ++jj) {
          lsum += s_l[lead + jj];
#pragma unroll
          for (int c = 0; c < CPL; ++c) acc[c] += s_o[lead + jj][lane * CPL + c];
        }
      }
    }
    if (active && j == 0) {
      const float il = 1.f / lsum;
      T* out = static_cast<T*>(p.out) + ((long long)s * p.num_heads + h0 + r) * D + lane * CPL;
#pragma unroll
      for (int c = 0; c < CPL; ++c) out[c] = DType<T>::from_f32(acc[c] * il);
    }
    __syncthreads();  // the shared arrays are reused by the next round
  }
}

// --- host-side launch helpers (instantiated per dtype) ------------------------------------------

template <typename TC, int D, int BS, bool kMma>
constexpr int decode_smem_bytes() {
  using Sh = DecodeShape<TC, D, BS>;
  return Sh::kRingBytes + Sh::kBarBytes + Sh::kTableBytes + Sh::kWarps * BS * 4 +
         Sh::kWarps * (kMma ? 16 : 1) * (D + 2) * 4;
}

template <typename T, typename TC, int D, int BS, bool kMma>
cudaError_t ensure_smem_attr() {
  static unsigned done = 0;  // bit d: set on device d
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 32 && ((__atomic_load_n(&done, __ATOMIC_ACQUIRE) >> dev) & 1u)) return cudaSuccess;
  e = cudaFuncSetAttribute(reinterpret_cast<const void*>(&decode_kernel<T, TC, D, BS, kMma>),
                           cudaFuncAttributeMaxDynamicSharedMemorySize, decode_smem_bytes<TC, D, BS, kMma>());
  if (e == cudaSuccess && dev < 32) __atomic_fetch_or(&done, 1u << dev, __ATOMIC_RELEASE);
  return e;
}

template <typename T, typename TC, int D, int BS, bool kMma>
int decode_ctas_per_sm_t() {
  if (ensure_smem_attr<T, TC, D, BS, kMma>() != cudaSuccess) return 0;
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, &decode_kernel<T, TC, D, BS, kMma>,
                                                    DecodeShape<TC, D, BS>::kWarps * 32,
                                                    decode_smem_bytes<TC, D, BS, kMma>()) != cudaSuccess)
    return 0;
  return n;
}

template <typename T, typename TC, int D, int BS, bool kMma>
cudaError_t launch_decode_t(const DecodeParams& p, int grid, cudaStream_t stream, int* launches) {
  *launches = 0;
  cudaError_t e = ensure_smem_attr<T, TC, D, BS, kMma>();
  if (e != cudaSuccess) return e;
  e = launch_pdl(decode_kernel<T, TC, D, BS, kMma>, dim3(grid), dim3(DecodeShape<TC, D, BS>::kWarps * 32),
                 decode_smem_bytes<TC, D, BS, kMma>(), stream, p);
  if (e != cudaSuccess) return e;
  *launches = 1;
  e = launch_pdl(decode_merge_kernel<T, D, kMma>, dim3(p.num_seqs * p.units), dim3(kMergeWarps * 32), 0, stream, p);
  if (e != cudaSuccess) return e;
  *launches = 2;
  return cudaSuccess;
}

// fp32 caches use the CUDA-core math only; 16-bit and FP8 caches both kinds.
template <typename T, typename TC, int D, int BS>
int ctas_for(DecodeKind kind) {
  if constexpr (sizeof(T) == 4) {
    return decode_ctas_per_sm_t<T, TC, D, BS, false>();
  } else {
    return kind == DecodeKind::kMma ? decode_ctas_per_sm_t<T, TC, D, BS, true>()
                                    : decode_ctas_per_sm_t<T, TC, D, BS, false>();
  }
}

template <typename T, typename TC, int D, int BS>
cudaError_t launch_for(const DecodeParams& p, DecodeKind kind, int grid, cudaStream_t s, int* n) {
  if constexpr (sizeof(T) == 4) {
    return launch_decode_t<T, TC, D, BS, false>(p, grid, s, n);
  } else {
    return kind == DecodeKind::kMma ? launch_decode_t<T, TC, D, BS, true>(p, grid, s, n)
                                    : launch_decode_t<T, TC, D, BS, false>(p, grid, s, n);
  }
}

template <typename T, typename TC>
int decode_ctas_per_sm_dispatch(int head_size, int block_size, DecodeKind kind) {
  if (head_size == 64 && block_size == 16) return ctas_for<T, TC, 64, 16>(kind);
  if (head_size == 64 && block_size == 32) return ctas_for<T, TC, 64, 32>(kind);
  if (head_size == 128 && block_size == 16) return ctas_for<T, TC, 128, 16>(kind);
  if (head_size == 128 && block_size == 32) return ctas_for<T, TC, 128, 32>(kind);
  return 0;
}

template <typename T, typename TC>
cudaError_t launch_decode_dispatch(int head_size, int block_size, const DecodeParams& p, DecodeKind kind, int grid,
                                   cudaStream_t s, int* n) {
  if (head_size == 64 && block_size == 16) return launch_for<T, TC, 64, 16>(p, kind, grid, s, n);
  if (head_size == 64 && block_size == 32) return launch_for<T, TC, 64, 32>(p, kind, grid, s, n);
  if (head_size == 128 && block_size == 16) return launch_for<T, TC, 128, 16>(p, kind, grid, s, n);
  if (head_size == 128 && block_size == 32) return launch_for<T, TC, 128, 32>(p, kind, grid, s, n);
  return cudaErrorInvalidValue;
}

}  // namespace pa
