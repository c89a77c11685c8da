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
//   * Tensor-core math (16-bit and FP8 caches, >= 2 query heads per kv head): the
//     query heads of one kv head are the 8-wide side of m16n8k16 tiles, tokens
//     and head dims the 16-row side (S^T = K Q^T, O^T += V^T P^T), so one K/V read
//     serves all of them and a kv head with up to 8 query heads wastes no
//     tensor-core work.  K and V come straight from the stage with ldmatrix; P
//     stays in registers, split into a rounded 16-bit high part and the rounded
//     remainder so P V keeps ~16 significant bits.
//   * The fused step (pa_decode_step) writes each sequence's new token as part of
//     decode.  Every warp stores its share of the tokens to the pool while its
//     first stages are in flight, and nothing waits for those stores: the token's
//     K and V rows also ride along with the TMA copy of the sequence's last block
//     into a side buffer beside the stage, and the warp that waits on that stage
//     puts the token into its slot of the stage, whatever the copy saw of the slot
//     in the pool.  The write costs no kernel of its own.
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

template <typename T, int D, int BS, int kMode>
struct DecodeShape {
  static constexpr int kElem = sizeof(T);
  static constexpr int kX = 16 / kElem;         // elements per 16-byte K group
  static constexpr int kTile = D * BS * kElem;  // bytes of one K (or V) tile
  static constexpr int kWarps = decode_warps(2 * kTile, kMode);
  static constexpr int kStages = decode_stages(2 * kTile, kMode);
  static constexpr int kRingBytes = kWarps * kStages * 2 * kTile;
  static constexpr int kBarBytes = (kWarps * kStages + 2) * 8;  // the ring's, then one nothing completes (+pad)
  // per-sequence tables: lengths, block prefix, warp sums
  // the cost-weighted prefix of the shared-prefix schedule ([S + 1] ints) is read only
  // while the warps find their ranges, before any copy is issued: it borrows the fused
  // step's side buffers where they are large enough, else it has room of its own here
  static constexpr int kWpreBytes = ((kMaxSeqsPerLaunch + 1) * 4 + 15) / 16 * 16;
  static constexpr int kSideStageBytes = 2 * D * (kElem < 2 ? 2 : kElem);
  static constexpr bool kWpreInSide = kWarps * kStages * kSideStageBytes >= kWpreBytes;
  static constexpr int kTableBytes =
      (kMaxSeqsPerLaunch + (kMaxSeqsPerLaunch + 1) + 2 * kWarps + 3 + 2 * kMaxSeqsPerLaunch) * 4 +
      (kWpreInSide ? 0 : kWpreBytes);
  // score row and running state per warp
  static constexpr int kRows = kMode ? 8 * kMode : 1;
  static constexpr int kStateBytes = kWarps * BS * 4 + kWarps * kRows * (D + 2) * 4;
  // the fused step: a sequence's new K and V rows land beside the stage of its last block
  static constexpr int kSideOffset = (kRingBytes + kBarBytes + kTableBytes + kStateBytes + 127) / 128 * 128;
  // (the rows come in the query's dtype: 16-bit for an FP8 pool, the pool's own otherwise)
  static constexpr int kSideStage = 2 * D * (kElem < 2 ? 2 : kElem);
  static constexpr int kSmemBytes = kSideOffset + kWarps * kStages * kSideStage;
  static_assert(kSmemBytes <= 227 * 1024, "shared memory per CTA");
  static_assert(kSideStage == kSideStageBytes, "side stage");
  // the regions after the tables hold float2 / float4 accesses: keep every region 16-byte aligned
  static_assert(kRingBytes % 16 == 0 && kBarBytes % 16 == 0 && kTableBytes % 16 == 0 && kStateBytes % 16 == 0,
                "shared-memory regions must stay 16-byte aligned");
};

// Wait for block i's stage.  On timeout record the error and drain the copies
// still in flight, the timed-out stage's included (each with its own bounded
// wait), so none lands after exit.  With test_ns > 0 (the timeout-path test), the
// warp's first wait is made on `never`, an mbarrier nothing completes, for test_ns
// nanoseconds: it runs out as a real timeout would, while the drains keep their
// normal limit, so every copy issued still lands before the warp stops.
template <int STAGES>
__device__ __forceinline__ bool wait_stage(uint64_t* bars, uint64_t* never, unsigned long long test_ns, int i, int n,
                                           unsigned* err, int lane) {
  const int st = i % STAGES;
  const bool ok =
      __all_sync(0xffffffffu, (test_ns && i == 0) ? mbar_wait_bounded(never, 0, test_ns)
                                                  : mbar_wait_bounded(&bars[st], (i / STAGES) & 1, kWaitLimitNs));
  if (!ok) {
    if (lane == 0) set_error(err, kErrTimeout);
    for (int j = i; j < n && j < i + STAGES; ++j)
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
// The query heads of one head unit (up to 8 * NH) against the tokens of a block,
// with the tiles transposed so that tokens and head dims take the 16-row side of
// the m16n8k16 shape and the query heads its 8-column side:
//     S^T [tokens x heads] = K [tokens x dims] Q^T [dims x heads]
//     O^T [dims x heads]  += V^T [dims x tokens] P^T [tokens x heads]
// K and V^T are A operands read straight from the stage with ldmatrix (a K-pool
// row holds 16 bytes of dims of one token, a V-pool row the tokens of one dim);
// Q^T stays in registers for the whole segment.  A kv head with at most 8 query
// heads fills one 8-column tile, so no tensor-core work goes to padding rows.
// P^T comes from S^T's accumulators through movmatrix (8x8 transposes): for bf16
// operands split into a rounded high part and the rounded remainder, so that P V
// keeps ~16 significant bits; for fp16 operands one rounded part (11 bits).
//
// T is the query / output type; TC is the cache element type: T itself (the
// operands are then T), or FP8 E4M3.  An FP8 cache is widened in registers to
// fp16 operands (every E4M3 value is an fp16 number; the hardware converts two
// codes per instruction), whatever T is: bf16 queries are brought to fp16 with a
// power-of-two scale per head, chosen from the head's largest |q| so that every
// element keeps its 8 significant bits, and the scale is taken back out of that
// head's scores.  A 16-byte ldmatrix row holds 16 codes and each thread receives
// 4 consecutive ones, which must become the (k, k+1) and (k+8, k+9) operand
// pairs: the dims of Q^T are permuted to match within each 16-dim k-step, and
// the token rows of K are loaded in the order perm(), so that S^T's rows line up
// with the permuted token columns of V^T.
//
// Only the 8-column tiles that hold query rows run (nt_ of them; a unit of up to 8
// heads in a 16-column kernel uses one): block() dispatches to the tile count once.
//
// kEarly (16-bit caches): block() is preceded by fetch(), which reads every K and
// V fragment of the block out of the stage into registers, so the kernel can
// refill the stage before the math instead of after it.
// 2^x by the hardware's approximate exponential, one instruction (|relative error|
// below 2^-22, results below 2^-126 flushed to 0, 2^-inf = 0): the P of a block and
// the rescale factors, which are rounded to 16 bits (P) or enter fp32 sums
__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

template <typename T, typename TC, int D, int BS, int NH, bool kEarly>
struct MmaMath {
  static constexpr int MT = BS / 16;  // 16-token tiles of a block
  static constexpr int KS = D / 16;   // 16-dim k-steps of S^T, and 16-dim row tiles of O^T
  static constexpr bool kFp8 = sizeof(TC) == 1;
  using OT = std::conditional_t<kFp8, __half, T>;  // tensor-core operand type
  static constexpr bool kRescaleQ = kFp8 && !std::is_same<T, __half>::value;
  // P^T in one rounded part for fp16 operands (11 significant bits, the operands' own
  // precision); for bf16 a rounded high part and the rounded remainder (~16 bits),
  // since one bf16 part (8 bits) can exceed the error bound on short sequences
  static constexpr bool kSplitP = !std::is_same<OT, __half>::value;
  static_assert(!(kEarly && kFp8), "early release is for 16-bit caches");
  static constexpr bool kFetch = kEarly;
  static constexpr int FM = kEarly ? MT : 1, FK = kEarly ? KS : 1;

  // Token (within a 16-token tile) of row r of S^T, which is also k-index r of P^T.
  __device__ __forceinline__ static int perm(int r) {
    return kFp8 ? 4 * ((r & 7) >> 1) + (r & 1) + 2 * (r >> 3) : r;
  }

  int nt_;                 // 8-column tiles in use (rows 0..nh-1): the others are skipped
  uint32_t qb[KS][NH][2];  // Q^T B fragments
  float acc[KS][NH][4];    // O^T accumulators
  uint32_t kf[FM][FK][4], vf[FM][FK][4];  // the block's K and V^T A fragments (kEarly)
  float m_[NH][2], l_[NH][2];  // running max (log2 units) and lane-partial sum of heads 8n + 2t4 + {0, 1}
  float hs_[NH][2];            // score factor (scale * log2 e, over the q scale) of heads 8n + 2t4 + {0, 1}
  uint32_t k_lane_off, v_lane_off;
  int g, t4, tok0, tok1;   // tok0 / tok1: tokens of this lane's S^T rows g and g + 8

  __device__ __forceinline__ void init(int lane, float*) {
    g = lane >> 2;
    t4 = lane & 3;
    tok0 = perm(g);
    tok1 = perm(g + 8);
    const int mi = lane >> 3, mr = lane & 7;  // ldmatrix: this lane addresses row mr of matrix mi
    if (kFp8) {
      // K: matrix mi = (16-dim chunk mi >> 1, token rows 8 (mi & 1) ..); V: 8 dims of 16 tokens
      k_lane_off = ((mi >> 1) * BS + perm((mi & 1) * 8 + mr)) * 16;
      v_lane_off = (mi * 8 + mr) * BS;
    } else {
      // K: matrix mi = (8-dim chunk mi >> 1, tokens 8 (mi & 1) ..); V: dims 8 (mi & 1) .., tokens 8 (mi >> 1) ..
      k_lane_off = ((mi >> 1) * BS + (mi & 1) * 8 + mr) * 16;
      v_lane_off = ((mi & 1) * 8 + mr) * (BS * 2) + (mi >> 1) * 16;
    }
  }

  __device__ __forceinline__ void reset() {
#pragma unroll
    for (int ks = 0; ks < KS; ++ks)
#pragma unroll
      for (int n = 0; n < NH; ++n) acc[ks][n][0] = acc[ks][n][1] = acc[ks][n][2] = acc[ks][n][3] = 0.f;
#pragma unroll
    for (int n = 0; n < NH; ++n) {
      m_[n][0] = m_[n][1] = -INFINITY;
      l_[n][0] = l_[n][1] = 0.f;
    }
  }

  // B fragments of query rows 0..nh-1, zero past nh, and the rows' score factors.
  // Row h is head h % group of sequence h / group: q points at the first row and
  // seq_stride is the distance between sequences (the rows of one unit, h < group,
  // are consecutive heads; a shared segment stacks the units of its members).
  __device__ __forceinline__ void load_q(const T* q, int nh, float scale_log2, int group, long long seq_stride) {
    nt_ = NH == 1 ? 1 : min(NH, (nh + 7) >> 3);
#pragma unroll
    for (int n = 0; n < NH; ++n) {
      const int h = 8 * n + g;
      const T* qh = q + (h / group) * seq_stride + (h % group) * D;
#pragma unroll
      for (int ks = 0; ks < KS; ++ks) {
        // operand k = 2t4, 2t4+1 and 2t4+8, 2t4+9 read dims d0, d0+1 and d1, d1+1
        const int d0 = ks * 16 + (kFp8 ? 4 * t4 : 2 * t4);
        const int d1 = kFp8 ? d0 + 2 : d0 + 8;
        qb[ks][n][0] = h < nh ? __ldg(reinterpret_cast<const unsigned int*>(qh + d0)) : 0u;
        qb[ks][n][1] = h < nh ? __ldg(reinterpret_cast<const unsigned int*>(qh + d1)) : 0u;
      }
      hs_[n][0] = hs_[n][1] = scale_log2;
      if constexpr (kRescaleQ) {
        // head g's largest |q| over the four lanes that hold its dims
        float mx = 0.f;
#pragma unroll
        for (int ks = 0; ks < KS; ++ks)
#pragma unroll
          for (int i = 0; i < 2; ++i) {
            const float2 v = unpack2<T>(qb[ks][n][i]);
            mx = fmaxf(mx, fmaxf(fabsf(v.x), fabsf(v.y)));
          }
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
        // 2^e with mx * 2^e in [2^13, 2^14): far from fp16's overflow, and any
        // element within 2^-27 of the largest stays a normal fp16 number
        int e = 0;
        if (mx > 0.f) {
          int ex;
          frexpf(mx, &ex);  // mx = f 2^ex, f in [0.5, 1)
          e = 14 - ex;
        }
        e = e > 120 ? 120 : e < -120 ? -120 : e;
        const float up = ldexpf(1.f, e);
#pragma unroll
        for (int ks = 0; ks < KS; ++ks)
#pragma unroll
          for (int i = 0; i < 2; ++i) {
            const float2 v = unpack2<T>(qb[ks][n][i]);
            qb[ks][n][i] = pack2<__half>(v.x * up, v.y * up);
          }
        // the factors of heads 2t4 and 2t4 + 1 of this tile (held by lanes 8 t4 and 8 t4 + 4)
        const float down = scale_log2 * ldexpf(1.f, -e);
        hs_[n][0] = __shfl_sync(0xffffffffu, down, 8 * t4);
        hs_[n][1] = __shfl_sync(0xffffffffu, down, 8 * t4 + 4);
      }
    }
  }

  // Read the block's K and V^T fragments out of the stage (kEarly only).
  __device__ __forceinline__ void fetch(unsigned char* stage, int tile_bytes) {
    if constexpr (kEarly) {
      const uint32_t kb = smem_addr(stage), vb = kb + tile_bytes;
#pragma unroll
      for (int mt = 0; mt < MT; ++mt)
#pragma unroll
        for (int ks = 0; ks < KS; ++ks)
          ldsm_x4(kb + k_lane_off + (2 * ks * BS + 16 * mt) * 16, kf[mt][ks][0], kf[mt][ks][1], kf[mt][ks][2],
                  kf[mt][ks][3]);
#pragma unroll
      for (int kk = 0; kk < MT; ++kk)
#pragma unroll
        for (int dm = 0; dm < KS; ++dm)
          ldsm_x4(vb + v_lane_off + dm * 16 * (BS * 2) + kk * 32, vf[kk][dm][0], vf[kk][dm][1], vf[kk][dm][2],
                  vf[kk][dm][3]);
    }
  }

  // Operand fragments of two k-steps from four ldmatrix registers of E4M3 codes:
  // registers 0, 1 (rows 0-7, 8-15 of the first k-step) and 2, 3 (the second).
  __device__ __forceinline__ static void widen(const uint32_t (&r)[4], uint32_t (&a0)[4], uint32_t (&a1)[4]) {
    e4m3x4_to_f16x2(r[0], a0[0], a0[2]);
    e4m3x4_to_f16x2(r[1], a0[1], a0[3]);
    e4m3x4_to_f16x2(r[2], a1[0], a1[2]);
    e4m3x4_to_f16x2(r[3], a1[1], a1[3]);
  }

  // Column (query row) masks of a shared segment: the member each of this lane's
  // columns belongs to; a block counts only for the members whose own table holds it.
  int col_member_[NH][2];
  __device__ __forceinline__ void set_columns(int group) {
#pragma unroll
    for (int n = 0; n < NH; ++n)
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) col_member_[n][hh] = (8 * n + 2 * t4 + hh) / group;
  }

  // One block: `rem` valid tokens; `live` has bit i set for every member i whose
  // columns take part (all ones outside shared segments).
  __device__ __forceinline__ void block(unsigned char* stage, int tile_bytes, int rem, float scale_log2,
                                        uint32_t live = 0xffffffffu) {
    if (NH == 1 || nt_ == NH)
      block_t<NH>(stage, tile_bytes, rem, scale_log2, live);
    else
      block_t<1>(stage, tile_bytes, rem, scale_log2, live);
  }

  // block() over the first NT 8-column tiles.
  template <int NT>
  __device__ __forceinline__ void block_t(unsigned char* stage, int tile_bytes, int rem, float scale_log2,
                                          uint32_t live) {
    const uint32_t kb = smem_addr(stage), vb = kb + tile_bytes;
    // S^T = K Q^T for the block's BS tokens, the even and the odd 16-dim k-steps in two
    // accumulators (two dependent chains of KS/2 MMAs, added at the end)
    float sc[MT][NH][4], so[MT][NH][4];
#pragma unroll
    for (int mt = 0; mt < MT; ++mt)
#pragma unroll
      for (int n = 0; n < NH; ++n)
#pragma unroll
        for (int c = 0; c < 4; ++c) sc[mt][n][c] = so[mt][n][c] = 0.f;
#pragma unroll
    for (int mt = 0; mt < MT; ++mt) {
      if constexpr (kFp8) {
#pragma unroll
        for (int kp = 0; kp < KS / 2; ++kp) {
          uint32_t r[4];  // (chunk 2kp, rows 0-7), (2kp, rows 8-15), (2kp+1, rows 0-7), (2kp+1, rows 8-15)
          ldsm_x4(kb + k_lane_off + (2 * kp * BS + 16 * mt) * 16, r[0], r[1], r[2], r[3]);
          uint32_t a0[4], a1[4];
          widen(r, a0, a1);
#pragma unroll
          for (int n = 0; n < NT; ++n) {
            mma_16816<OT>(sc[mt][n], a0, qb[2 * kp][n][0], qb[2 * kp][n][1]);
            mma_16816<OT>(so[mt][n], a1, qb[2 * kp + 1][n][0], qb[2 * kp + 1][n][1]);
          }
        }
      } else {
#pragma unroll
        for (int ks = 0; ks < KS; ++ks) {
          uint32_t a[4];
          if constexpr (kEarly) {
#pragma unroll
            for (int i = 0; i < 4; ++i) a[i] = kf[kEarly ? mt : 0][kEarly ? ks : 0][i];
          } else {
            ldsm_x4(kb + k_lane_off + (2 * ks * BS + 16 * mt) * 16, a[0], a[1], a[2], a[3]);
          }
#pragma unroll
          for (int n = 0; n < NT; ++n)
            mma_16816<OT>((ks & 1) ? so[mt][n] : sc[mt][n], a, qb[ks][n][0], qb[ks][n][1]);
        }
      }
#pragma unroll
      for (int n = 0; n < NT; ++n)
#pragma unroll
        for (int c = 0; c < 4; ++c) sc[mt][n][c] += so[mt][n][c];
    }
    // Online softmax update per head (column), log2 domain; tokens past the sequence
    // (and every token, for a column whose member does not take this block) get -inf.
    bool col_ok[NH][2];
#pragma unroll
    for (int n = 0; n < NH; ++n)
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) col_ok[n][hh] = (live >> col_member_[n][hh]) & 1u;
    float mx[NH][2];
#pragma unroll
    for (int n = 0; n < NH; ++n) mx[n][0] = mx[n][1] = -INFINITY;
#pragma unroll
    for (int mt = 0; mt < MT; ++mt)
#pragma unroll
      for (int n = 0; n < NT; ++n) {
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const int tok = 16 * mt + ((c >> 1) ? tok1 : tok0);
          const float v = sc[mt][n][c] * hs_[n][c & 1];
          sc[mt][n][c] = (tok < rem && col_ok[n][c & 1]) ? v : -INFINITY;
          mx[n][c & 1] = fmaxf(mx[n][c & 1], sc[mt][n][c]);
        }
      }
    // mref: the reference the exponentials are taken against; 0 while a column has
    // seen no score at all (then every term is 2^-inf = 0, never -inf - -inf)
    float corr[NH][2], ps[NH][2], mref[NH][2];
#pragma unroll
    for (int n = 0; n < NH; ++n)
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        corr[n][h] = 1.f;
        ps[n][h] = 0.f;
        mref[n][h] = 0.f;
        if (n >= NT) continue;
        float v = mx[n][h];
        v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 4));
        v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 8));
        v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 16));
        const float mn = fmaxf(m_[n][h], v);
        mref[n][h] = mn == -INFINITY ? 0.f : mn;
        corr[n][h] = ex2_approx(m_[n][h] - mref[n][h]);
        m_[n][h] = mn;
      }
#pragma unroll
    for (int mt = 0; mt < MT; ++mt)
#pragma unroll
      for (int n = 0; n < NT; ++n) {
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          sc[mt][n][c] = ex2_approx(sc[mt][n][c] - mref[n][c & 1]);
          ps[n][c & 1] += sc[mt][n][c];
        }
      }
#pragma unroll
    for (int n = 0; n < NH; ++n) {
      l_[n][0] = l_[n][0] * corr[n][0] + ps[n][0];
      l_[n][1] = l_[n][1] * corr[n][1] + ps[n][1];
    }
    // rescale O only when some column's maximum moved (a factor of exactly 1 changes nothing)
    bool moved = false;
#pragma unroll
    for (int n = 0; n < NT; ++n) moved |= corr[n][0] != 1.f || corr[n][1] != 1.f;
    if (__any_sync(0xffffffffu, moved)) {
#pragma unroll
      for (int ks = 0; ks < KS; ++ks)
#pragma unroll
        for (int n = 0; n < NT; ++n) {
          acc[ks][n][0] *= corr[n][0];
          acc[ks][n][1] *= corr[n][1];
          acc[ks][n][2] *= corr[n][0];
          acc[ks][n][3] *= corr[n][1];
        }
    }
    // O^T += V^T P^T, one 16-token k-step per 16-token tile of S^T.
#pragma unroll
    for (int kk = 0; kk < MT; ++kk) {
      uint32_t bh[NH][2], bl[NH][2];
#pragma unroll
      for (int n = 0; n < NH; ++n)
#pragma unroll
        for (int r = 0; r < 2; ++r) {  // S^T rows 0-7, then rows 8-15
          if (n >= NT) break;
          const float x = sc[kk][n][2 * r], y = sc[kk][n][2 * r + 1];
          const uint32_t hi = pack2<OT>(x, y);
          bh[n][r] = movmatrix_trans(hi);
          if constexpr (kSplitP) {
            const float2 back = unpack2<OT>(hi);
            bl[n][r] = movmatrix_trans(pack2<OT>(x - back.x, y - back.y));
          }
        }
      if constexpr (kFp8) {
#pragma unroll
        for (int dp = 0; dp < KS / 2; ++dp) {
          uint32_t r[4];  // dims 32dp + 0-7, 8-15, 16-23, 24-31; tokens 16kk .. 16kk+15
          ldsm_x4(vb + v_lane_off + 32 * dp * BS + 16 * kk, r[0], r[1], r[2], r[3]);
          uint32_t a0[4], a1[4];
          widen(r, a0, a1);
#pragma unroll
          for (int n = 0; n < NT; ++n) {
            mma_16816<OT>(acc[2 * dp][n], a0, bh[n][0], bh[n][1]);
            mma_16816<OT>(acc[2 * dp + 1][n], a1, bh[n][0], bh[n][1]);
            if constexpr (kSplitP) {
              mma_16816<OT>(acc[2 * dp][n], a0, bl[n][0], bl[n][1]);
              mma_16816<OT>(acc[2 * dp + 1][n], a1, bl[n][0], bl[n][1]);
            }
          }
        }
      } else {
#pragma unroll
        for (int dm = 0; dm < KS; ++dm) {
          uint32_t a[4];
          if constexpr (kEarly) {
#pragma unroll
            for (int i = 0; i < 4; ++i) a[i] = vf[kEarly ? kk : 0][kEarly ? dm : 0][i];
          } else {
            ldsm_x4(vb + v_lane_off + dm * 16 * (BS * 2) + kk * 32, a[0], a[1], a[2], a[3]);
          }
#pragma unroll
          for (int n = 0; n < NT; ++n) {
            mma_16816<OT>(acc[dm][n], a, bh[n][0], bh[n][1]);
            if constexpr (kSplitP) mma_16816<OT>(acc[dm][n], a, bl[n][0], bl[n][1]);
          }
        }
      }
    }
  }

  // Complete the sums over the eight lanes that share a head.
  __device__ __forceinline__ void finish() {
#pragma unroll
    for (int n = 0; n < NH; ++n)
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        float v = l_[n][h];
        v += __shfl_xor_sync(0xffffffffu, v, 4);
        v += __shfl_xor_sync(0xffffffffu, v, 8);
        v += __shfl_xor_sync(0xffffffffu, v, 16);
        l_[n][h] = v;
      }
  }

  // out heads 0..nh-1 (row stride D) = oscale * acc / l, rounded to T; transposed
  // back to head-major through movmatrix so each lane stores pairs of dims.
  __device__ __forceinline__ void store_out(T* out, int nh, float oscale) const {
#pragma unroll
    for (int n = 0; n < NH; ++n) {
      const float i0 = oscale / l_[n][0], i1 = oscale / l_[n][1];
      const int h = 8 * n + g;
#pragma unroll
      for (int ks = 0; ks < KS; ++ks) {
        const uint32_t x0 = movmatrix_trans(pack2<T>(acc[ks][n][0] * i0, acc[ks][n][1] * i1));
        const uint32_t x1 = movmatrix_trans(pack2<T>(acc[ks][n][2] * i0, acc[ks][n][3] * i1));
        if (h < nh) {
          *reinterpret_cast<uint32_t*>(out + h * D + ks * 16 + 2 * t4) = x0;
          *reinterpret_cast<uint32_t*>(out + h * D + ks * 16 + 8 + 2 * t4) = x1;
        }
      }
    }
  }

  // Partial result of heads 0..nh-1: o = oscale * acc / l (fp32, row stride D), (m, l).
  __device__ __forceinline__ void store_partial(float* po, float* pml, int nh, float oscale) const {
#pragma unroll
    for (int n = 0; n < NH; ++n)
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        const int h = 8 * n + 2 * t4 + hh;
        if (h >= nh) continue;
        const float inv = oscale / l_[n][hh];
#pragma unroll
        for (int ks = 0; ks < KS; ++ks) {
          po[h * D + ks * 16 + g] = acc[ks][n][hh] * inv;
          po[h * D + ks * 16 + 8 + g] = acc[ks][n][2 + hh] * inv;
        }
        if (g == 0) *reinterpret_cast<float2*>(pml + 2 * h) = make_float2(m_[n][hh], l_[n][hh]);
      }
  }

  // Merge this partition's result (m, l, o = acc / l) into the warp's running
  // state (M, W, O) in shared memory: M' = max(M, m), O' = O 2^(M - M') + l 2^(m - M') o,
  // W' = W 2^(M - M') + l 2^(m - M').  so: [8 NH][D], sml: [8 NH][2].
  __device__ __forceinline__ void fold(float* so, float* sml, bool first) const {
    float M[NH][2], Wt[NH][2];
#pragma unroll
    for (int n = 0; n < NH; ++n)
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        const int h = 8 * n + 2 * t4 + hh;
        M[n][hh] = first ? -INFINITY : sml[2 * h];
        Wt[n][hh] = first ? 0.f : sml[2 * h + 1];
      }
    __syncwarp();
#pragma unroll
    for (int n = 0; n < NH; ++n)
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        const int h = 8 * n + 2 * t4 + hh;
        const float mn = fmaxf(M[n][hh], m_[n][hh]);
        const float mr = mn == -INFINITY ? 0.f : mn;  // a column with no score yet: both factors 0
        const float fo = exp2f(M[n][hh] - mr), fp = exp2f(m_[n][hh] - mr);  // l 2^(m - M') times o = acc / l
        if (g == 0) *reinterpret_cast<float2*>(sml + 2 * h) = make_float2(mn, Wt[n][hh] * fo + l_[n][hh] * fp);
#pragma unroll
        for (int ks = 0; ks < KS; ++ks)
#pragma unroll
          for (int r = 0; r < 2; ++r) {
            float* o = so + h * D + ks * 16 + 8 * r + g;
            *o = (first ? 0.f : *o) * fo + fp * acc[ks][n][2 * r + hh];
          }
      }
    __syncwarp();
  }

  // Take the running state as this piece's (m, l, acc): acc = O, l = W.
  __device__ __forceinline__ void load_state(const float* so, const float* sml) {
#pragma unroll
    for (int n = 0; n < NH; ++n)
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        const int h = 8 * n + 2 * t4 + hh;
        m_[n][hh] = sml[2 * h];
        l_[n][hh] = sml[2 * h + 1];
#pragma unroll
        for (int ks = 0; ks < KS; ++ks)
#pragma unroll
          for (int r = 0; r < 2; ++r) acc[ks][n][2 * r + hh] = so[h * D + ks * 16 + 8 * r + g];
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

  static constexpr bool kFetch = false;
  __device__ __forceinline__ void fetch(unsigned char*, int) {}

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

  __device__ __forceinline__ void load_q(const T* q, int, float, int, long long) {
    const T* qh = q + half * NGH * X;
#pragma unroll
    for (int k = 0; k < NGH * X; ++k) qv[k] = DType<T>::to_f32(qh[k]);
  }

  __device__ __forceinline__ void set_columns(int) {}

  __device__ __forceinline__ void block(unsigned char* stage, int tile_bytes, int rem, float scale_log2,
                                        uint32_t = 0xffffffffu) {
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

// --- the fused step: the new token ---------------------------------------------------------------

// The E4M3 codes of x / scale, the division correctly rounded in fp32, the
// conversion round-to-nearest-even and saturating -- the write path's conversion,
// so the fused step stores and decodes the very codes the separate write stores.
template <typename TS>
__device__ __forceinline__ uint4 e4m3_codes16(const TS* src, float scale) {
  uint32_t w[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    uint32_t packed = 0;
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      const float a = __fdiv_rn(DType<TS>::to_f32(src[4 * i + 2 * j]), scale);
      const float b = __fdiv_rn(DType<TS>::to_f32(src[4 * i + 2 * j + 1]), scale);
      packed |= (__nv_cvt_float2_to_fp8x2(make_float2(a, b), __NV_SATFINITE, __NV_E4M3) & 0xffffu) << (16 * j);
    }
    w[i] = packed;
  }
  return make_uint4(w[0], w[1], w[2], w[3]);
}
template <typename TS>
__device__ __forceinline__ unsigned char e4m3_code(TS x, float scale) {
  return static_cast<unsigned char>(
      __nv_cvt_float_to_fp8(__fdiv_rn(DType<TS>::to_f32(x), scale), __NV_SATFINITE, __NV_E4M3));
}

// The fused step's new token into an FP8 stage: the side buffer holds the K and V rows
// in the query dtype T; they are quantised as the write path quantises them.
template <typename T, int D, int BS>
__device__ __forceinline__ void inject_token_e4m3(unsigned char* stage, int tile_bytes, const unsigned char* side,
                                                  int off, float k_scale, float v_scale, int lane) {
  constexpr int VPL = D / 32;
  const T* sk = reinterpret_cast<const T*>(side);
  const T* sv = sk + D;
  unsigned char* v = stage + tile_bytes;
  if (lane < D / 16) {
    T e[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) e[i] = sk[lane * 16 + i];
    *reinterpret_cast<uint4*>(stage + (lane * BS + off) * 16) = e4m3_codes16<T>(e, k_scale);
  }
#pragma unroll
  for (int i = 0; i < VPL; ++i) v[(lane + 32 * i) * BS + off] = e4m3_code<T>(sv[lane + 32 * i], v_scale);
  __syncwarp();
}

// The fused step's new token of a (sequence, kv head) -- its K and V rows, copied
// by TMA into `side` with the stage of the sequence's last block -- into that
// stage at slot `off` (K tile [D/X][BS][X]: 16 bytes per X-group, D/X <= 32 of
// them; V tile [D][BS]: one element per dim).
template <typename TC, int D, int BS>
__device__ __forceinline__ void inject_token(unsigned char* stage, int tile_bytes, const unsigned char* side, int off,
                                             int lane) {
  constexpr int X = 16 / static_cast<int>(sizeof(TC)), VPL = D / 32;
  const TC* sv = reinterpret_cast<const TC*>(side + D * sizeof(TC));
  TC* v = reinterpret_cast<TC*>(stage + tile_bytes);
  uint4 g;
  TC e[VPL];
  if (lane < D / X) g = reinterpret_cast<const uint4*>(side)[lane];
#pragma unroll
  for (int i = 0; i < VPL; ++i) e[i] = sv[lane + 32 * i];
  if (lane < D / X) *reinterpret_cast<uint4*>(stage + (lane * BS + off) * 16) = g;
#pragma unroll
  for (int i = 0; i < VPL; ++i) v[(lane + 32 * i) * BS + off] = e[i];
  __syncwarp();
}

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


// Shared prefixes: the clusters and the work of each sequence (see DecodeParams).
// On entry nb[k] holds the blocks of sequence tid * PER + k; on exit its blocks of
// work per unit -- a leader's: its cluster's shared segment plus its own blocks;
// anyone's own blocks: those past the ones it shares -- and s_info[], s_lead[]
// the packed layout.
//   runs: consecutive valid sequences with equal prefix_group; each run is cut
//   into clusters of `members` consecutive sequences, the first the leader;
//   sh(m) = prefix_blocks[m] limited to [0, its blocks - 1] (the last block of a
//   sequence stays its own: the fused step writes it) and to B, the second largest
//   of them (blocks past B are held by one member only); in a cluster of one, 0;
//   the cluster's shared segment is its first B blocks, read through the table of
//   the member with the largest prefix_blocks (the donor).
// wt[k] receives the cost of the sequence's work per unit (see kSegCost).
// s_pre and s_red are scratch here.
template <int PER>
__device__ __forceinline__ void shared_layout(const DecodeParams& p, int* s_pre, int* s_info, int* s_lead,
                                              int* s_red, int (&nb)[PER], int (&wt)[PER], int tid, int warp,
                                              int lane) {
  const int S = p.num_seqs, M = p.members;
#pragma unroll
  for (int k = 0; k < PER; ++k) {
    const int i = tid * PER + k;
    if (i < S) s_pre[i] = nb[k];
  }
  __syncthreads();
  // link: sequence i continues the run of i - 1; kept in bit 30 of s_info[i] (beside sh) until the
  // leaders have sized their clusters, so that they read shared memory only
  constexpr int kLinkBit = 1 << 30, kShMask = (1 << kInfoOffBits) - 1;
  int c0[PER], run = -1;  // the start of the run of each sequence (-1: before this thread's first)
#pragma unroll
  for (int k = 0; k < PER; ++k) {
    const int i = tid * PER + k;
    bool link = false;
    int sh = 0;
    if (i < S && nb[k] > 0) {
      const int gi = __ldg(p.prefix_group + i), pb = __ldg(p.prefix_blocks + i);
      link = i > 0 && s_pre[i - 1] > 0 && __ldg(p.prefix_group + i - 1) == gi;
      sh = max(0, min(pb, nb[k] - 1));
    }
    if (i < S) s_info[i] = sh | (link ? kLinkBit : 0);
    if (!link) run = i;
    c0[k] = run;
  }
  int incl = run;  // run starts seen up to this thread: a running maximum
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int x = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl = max(incl, x);
  }
  if (lane == 31) s_red[warp] = incl;
  __syncthreads();
  int before = __shfl_up_sync(0xffffffffu, incl, 1);
  if (lane == 0) before = -1;
  for (int w = 0; w < warp; ++w) before = max(before, s_red[w]);
#pragma unroll
  for (int k = 0; k < PER; ++k)
    if (c0[k] < 0) c0[k] = before;
  __syncthreads();  // every sh and link is in s_info
  // the cluster of a leader: its size (the run continues while the links do), B and the donor
  int size_[PER];
#pragma unroll
  for (int k = 0; k < PER; ++k) {
    const int i = tid * PER + k;
    size_[k] = 0;
    if (i >= S || (i - c0[k]) % M != 0) continue;
    int size = 1;
    while (i + size < S && size < M && (s_info[i + size] & kLinkBit)) ++size;
    size_[k] = size;
  }
  __syncthreads();  // every leader has read the links
#pragma unroll
  for (int k = 0; k < PER; ++k) {
    const int i = tid * PER + k, size = size_[k];
    if (size == 0) continue;
    // B: the second largest sh (blocks past it are held by one member only: its own);
    // the donor: a member with the largest sh, whose table holds all B blocks
    int top = 0, B = 0, donor = 0;
    if (size > 1)
      for (int m = 0; m < size; ++m) {
        const int sh = s_info[i + m] & kShMask;
        if (sh > top) {
          B = top;
          top = sh;
          donor = m;
        } else if (sh > B) {
          B = sh;
        }
      }
    // clusters are disjoint: only this thread writes the entries of this one
    for (int m = 0; m < size; ++m) {
      const int sh = min(s_info[i + m] & kShMask, B);
      s_info[i + m] = sh | (m << kInfoOffBits) | (m == 0 ? (size - 1) << 27 : 0);
    }
    s_lead[i] = B | (donor << kInfoOffBits);
  }
  __syncthreads();
#pragma unroll
  for (int k = 0; k < PER; ++k) {
    const int i = tid * PER + k;
    wt[k] = 0;
    if (i < S && nb[k] > 0) {
      const int B = info_member(s_info[i]) == 0 ? info_off(s_lead[i]) : 0, own = nb[k] - info_off(s_info[i]);
      nb[k] = B + own;
      wt[k] = (B > 0 ? kSegCost + kSharedCost * B : 0) + kSegCost + kOwnCost * own;
    }
  }
  __syncthreads();  // s_pre and s_red are rewritten by the prefix sums that follow
}

// grid = resident CTAs (persistent); kDecodeWarps independent warps per CTA.
// kMode: 0 = CUDA-core math, 1 or 2 = tensor-core math over 8 or 16 query heads per unit.
template <typename T, typename TC, int D, int BS, int kMode>
__global__ void __launch_bounds__(DecodeShape<TC, D, BS, kMode>::kWarps * 32, 1)
    decode_kernel(const DecodeParams p) {
  using Sh = DecodeShape<TC, D, BS, kMode>;
  constexpr int kDecodeWarps = Sh::kWarps;
  constexpr bool kMma = kMode != 0;
  // Early stage release: 16-bit caches in 8-warp CTAs whose fragments of a block fit in 64 registers.
  constexpr bool kEarly = kMma && sizeof(TC) == 2 && kDecodeWarps == 8 && D * BS <= 128 * 16;
  using Math = std::conditional_t<kMma, MmaMath<T, TC, D, BS, (kMode > 0 ? kMode : 1), kEarly>,
                                  SimtMath<T, TC, D, BS>>;
  constexpr int TILE = Sh::kTile, STAGES = Sh::kStages;
  extern __shared__ __align__(128) unsigned char smem[];

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  unsigned char* ring = smem + warp * STAGES * 2 * TILE;
  unsigned char* side = smem + Sh::kSideOffset + warp * STAGES * Sh::kSideStage;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + Sh::kRingBytes) + warp * STAGES;
  uint64_t* never = reinterpret_cast<uint64_t*>(smem + Sh::kRingBytes) + kDecodeWarps * STAGES;
  int* s_len = reinterpret_cast<int*>(smem + Sh::kRingBytes + Sh::kBarBytes);
  int* s_pre = s_len + kMaxSeqsPerLaunch;                 // [S + 1] block prefix per unit
  int* s_wsum = s_pre + kMaxSeqsPerLaunch + 1;             // [2 warps]: per-warp sums of the prefix scans
  int* s_info = s_wsum + 2 * kDecodeWarps + 3;             // [S] cluster layout (shared prefixes)
  int* s_lead = s_info + kMaxSeqsPerLaunch;                // [S] a leader's shared segment and donor
  // [S + 1] cost-weighted prefix per unit (shared prefixes; see DecodeShape::kWpreBytes)
  int* s_wpre = Sh::kWpreInSide ? reinterpret_cast<int*>(smem + Sh::kSideOffset) : s_lead + kMaxSeqsPerLaunch;
  float* pw = reinterpret_cast<float*>(smem + Sh::kRingBytes + Sh::kBarBytes + Sh::kTableBytes) + warp * BS;
  // running state of this warp's piece across caller partitions (see fold)
  constexpr int kRows = kMma ? 8 * kMode : 1;
  float* st_o = reinterpret_cast<float*>(smem + Sh::kRingBytes + Sh::kBarBytes + Sh::kTableBytes) +
                kDecodeWarps * BS + warp * kRows * (D + 2);
  float* st_ml = st_o + kRows * D;

  if (lane == 0) {
    for (int st = 0; st < STAGES; ++st) mbar_init(&bars[st], 1);
    if (warp == 0) mbar_init(never, 1);  // visible to the other warps after the table prologue's barriers
    fence_barrier_init();
  }
  __syncwarp();
  griddep_launch_dependents();

  // Per-sequence tables: length (0 when outside [1, max_seq_len]) and prefix sums
  // of the blocks of work per unit.  Each thread scans PER consecutive sequences.
  // They come from seq_lens and the prefix groups, which no kernel of this library
  // writes, so they are built while the previous kernel in the stream may still be
  // running (see griddep_wait below).
  const int S = p.num_seqs, U = p.units, PB = p.part_blocks;
  const bool shared = kMma && p.shared;
  {
    constexpr int PER = (kMaxSeqsPerLaunch + kDecodeWarps * 32 - 1) / (kDecodeWarps * 32);
    int nb[PER], wt[PER];
#pragma unroll
    for (int k = 0; k < PER; ++k) {
      const int i = tid * PER + k;
      int L = i < S ? __ldg(p.seq_lens + i) : 0;
      if (L < 1 || L > p.max_seq_len) L = 0;
      if (i < S) s_len[i] = L;
      nb[k] = (L + BS - 1) / BS;
    }
    if (shared) {
      shared_layout<PER>(p, s_pre, s_info, s_lead, s_wsum, nb, wt, tid, warp, lane);
    } else {
#pragma unroll
      for (int k = 0; k < PER; ++k) wt[k] = nb[k] > 0 ? kSegCost + kOwnCost * nb[k] : 0;
    }
    // exclusive prefix sums over the sequences of the blocks (into s_pre) and of the cost
    // (into s_wpre) of each one's work per unit, in one pass
    int sb = 0, sw = 0;
#pragma unroll
    for (int k = 0; k < PER; ++k) {
      sb += nb[k];
      sw += wt[k];
    }
    int ib = sb, iw = sw;  // inclusive warp scans
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int xb = __shfl_up_sync(0xffffffffu, ib, o), xw = __shfl_up_sync(0xffffffffu, iw, o);
      if (lane >= o) {
        ib += xb;
        iw += xw;
      }
    }
    if (lane == 31) {
      s_wsum[warp] = ib;
      s_wsum[kDecodeWarps + warp] = iw;
    }
    __syncthreads();
    int ob = ib - sb, ow = iw - sw;
    for (int w = 0; w < warp; ++w) {
      ob += s_wsum[w];
      ow += s_wsum[kDecodeWarps + w];
    }
#pragma unroll
    for (int k = 0; k < PER; ++k) {
      const int i = tid * PER + k;
      if (i <= S) {
        s_pre[i] = ob;
        s_wpre[i] = ow;
      }
      ob += nb[k];
      ow += wt[k];
    }
    if (tid == blockDim.x - 1) {  // the totals (also covers S == kMaxSeqsPerLaunch)
      s_pre[S] = ob;
      s_wpre[S] = ow;
    }
    __syncthreads();
  }
  // segment ids: one per (sequence, unit), or two with shared prefixes (the shared part, then the own part)
  auto seg_id = [&](int s, int u, int part) { return shared ? 2 * (s * U + u) + part : s * U + u; };
  // blocks of sequence s's shared segment (s a leader), else 0
  auto shared_len = [&](int s) { return info_member(s_info[s]) == 0 ? info_off(s_lead[s]) : 0; };

  // Everything from here on may touch memory the previous kernel in the stream
  // writes (the pools, the output, the workspace a previous call's merge still reads).
  griddep_wait();

  // Sequences outside the contract: record the error, zero their rows, mark their
  // segments as needing no merge.  One CTA does it, and hands the cluster layout
  // to the merge kernel.
  if (blockIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      if (s_len[s] != 0) continue;
      if (tid == 0) set_error(p.err, kErrSeqLen);
      T* out = static_cast<T*>(p.out) + (long long)s * p.num_heads * D;
      for (int i = tid; i < p.num_heads * D; i += blockDim.x) out[i] = DType<T>::from_f32(0.f);
      for (int u = tid; u < U; u += blockDim.x) p.seg_first[seg_id(s, u, 1)] = -1;
    }
    if (shared)
      for (int s = tid; s < S; s += blockDim.x) {
        p.seq_info[s] = s_info[s];
        p.seq_info[S + s] = s_lead[s];
      }
  }

  const int W = gridDim.x * kDecodeWarps;
  const int w = blockIdx.x * kDecodeWarps + warp;

  // The fused step's pool writes: item i = (sequence, kv head) of the launch goes
  // to warp i mod W.  A batch of items is loaded before any of it is stored (the
  // stores may alias the loads as far as the compiler knows).  Nothing in this
  // launch reads these slots from the pool afterwards: decode takes the tokens
  // from the side buffers (see issue), so the stores need no ordering.
  auto write_tokens_e4m3 = [&]() {  // an FP8 pool: rows in T, quantised as the write path does
    constexpr int VPL = D / 32;
    const long long tile_bytes = (long long)D * BS;
    unsigned char* kc = static_cast<unsigned char*>(const_cast<void*>(p.k_cache));
    unsigned char* vc = static_cast<unsigned char*>(const_cast<void*>(p.v_cache));
    const int items = S * p.num_kv_heads;
    for (int i = w; i < items; i += W) {
      const int s2 = i / p.num_kv_heads, h = i - s2 * p.num_kv_heads, L2 = s_len[s2];
      if (L2 == 0) continue;
      const int blk = __ldg(p.block_tables + (long long)s2 * p.max_blocks_per_seq + (L2 - 1) / BS);
      if (blk < 0 || blk >= p.num_blocks) continue;  // recorded when decode reads the block
      const long long tile = (long long)blk * p.num_kv_heads + h;
      const int off = (L2 - 1) % BS;
      const T* key = static_cast<const T*>(p.new_key) + (long long)i * D;
      const T* value = static_cast<const T*>(p.new_value) + (long long)i * D;
      T e[16], vv[VPL];
      if (lane < D / 16) {
#pragma unroll
        for (int j = 0; j < 16; ++j) e[j] = key[lane * 16 + j];
      }
#pragma unroll
      for (int j = 0; j < VPL; ++j) vv[j] = value[lane + 32 * j];
      if (lane < D / 16)
        *reinterpret_cast<uint4*>(kc + tile * tile_bytes + (lane * BS + off) * 16) = e4m3_codes16<T>(e, p.write_k_scale);
#pragma unroll
      for (int j = 0; j < VPL; ++j)
        vc[tile * tile_bytes + (long long)(lane + 32 * j) * BS + off] = e4m3_code<T>(vv[j], p.write_v_scale);
    }
  };
  auto write_tokens = [&]() {
    if constexpr (sizeof(TC) == 1) {
      write_tokens_e4m3();
      return;
    }
    constexpr int X = 16 / static_cast<int>(sizeof(TC)), VPL = D / 32, kBatch = 4;
    const long long tile_bytes = (long long)D * BS * sizeof(TC);
    unsigned char* kc = static_cast<unsigned char*>(const_cast<void*>(p.k_cache));
    unsigned char* vc = static_cast<unsigned char*>(const_cast<void*>(p.v_cache));
    const int items = S * p.num_kv_heads;
    for (int i0 = w; i0 < items; i0 += kBatch * W) {
      uint4 kv[kBatch];
      TC vv[kBatch][VPL];
      long long tile[kBatch];
      int off[kBatch];
#pragma unroll
      for (int b = 0; b < kBatch; ++b) {
        const int i = i0 + b * W;
        tile[b] = -1;
        if (i >= items) continue;
        const int s2 = i / p.num_kv_heads, h = i - s2 * p.num_kv_heads, L2 = s_len[s2];
        if (L2 == 0) continue;
        const int blk = __ldg(p.block_tables + (long long)s2 * p.max_blocks_per_seq + (L2 - 1) / BS);
        if (blk < 0 || blk >= p.num_blocks) continue;  // recorded when decode reads the block
        tile[b] = (long long)blk * p.num_kv_heads + h;
        off[b] = (L2 - 1) % BS;
        const TC* key = static_cast<const TC*>(p.new_key) + (long long)i * D;
        const TC* value = static_cast<const TC*>(p.new_value) + (long long)i * D;
        if (lane < D / X) kv[b] = __ldg(reinterpret_cast<const uint4*>(key) + lane);
#pragma unroll
        for (int e = 0; e < VPL; ++e) vv[b][e] = value[lane + 32 * e];
      }
#pragma unroll
      for (int b = 0; b < kBatch; ++b) {
        if (tile[b] < 0) continue;
        if (lane < D / X) *reinterpret_cast<uint4*>(kc + tile[b] * tile_bytes + (lane * BS + off[b]) * 16) = kv[b];
        TC* vt = reinterpret_cast<TC*>(vc + tile[b] * tile_bytes);
#pragma unroll
        for (int e = 0; e < VPL; ++e) vt[(lane + 32 * e) * BS + off[b]] = vv[b][e];
      }
    }
  };

  // This warp's range of the T blocks of work: an equal share of their cost (blocks,
  // shared blocks and segments weighted as kSegCost says).
  const long long T_all = (long long)s_pre[S] * U;
  long long start, end;
  {
    const long long Tw = (long long)s_wpre[S] * U;
    // the first block whose cost starts at or after t
    auto block_at = [&](long long t) -> long long {
      if (t >= Tw) return T_all;
      int lo = 0, hi = S - 1;
      while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if ((long long)s_wpre[mid] * U <= t) lo = mid;
        else hi = mid - 1;
      }
      const int s = lo, wl = s_wpre[s + 1] - s_wpre[s], nbl = s_pre[s + 1] - s_pre[s];
      const long long r = t - (long long)s_wpre[s] * U;
      const int u = static_cast<int>(r / wl), rr = static_cast<int>(r - (long long)u * wl);
      // a unit's cost: [segment, shared blocks] (a leader with a shared part), segment, own blocks
      const int B = shared ? shared_len(s) : 0;
      const int wS = B > 0 ? kSegCost + kSharedCost * B : 0;
      const int j = rr < wS ? max(0, rr - kSegCost + kSharedCost - 1) / kSharedCost
                            : B + max(0, rr - wS - kSegCost + kOwnCost - 1) / kOwnCost;
      return (long long)s_pre[s] * U + (long long)u * nbl + j;
    };
    const long long qt = Tw / W, rt = Tw % W;
    start = block_at(w * qt + (w * rt) / W);
    end = block_at((w + 1) * qt + ((w + 1) * rt) / W);
    __syncthreads();  // every warp has its range: the side buffers may now receive copies
  }
  const int len = static_cast<int>(end - start);
  if (len <= 0) {
    if (p.fused) write_tokens();
    return;
  }

  // Table lookups: lane i resolves work position start + 32 * group + i: the
  // physical block, and kvh | sequence << 16 | (last block of the sequence) << 30.
  const int32_t* __restrict__ bt = p.block_tables;
  auto fetch = [&](int group, int& phys, int& kvh) {
    const long long gpos = start + 32LL * group + lane;
    phys = 0;
    kvh = 0;
    if (gpos < end) {
      int s, u, j, h0, nh;
      locate(gpos, s_pre, S, U, s, u, j);
      unit_heads<kMma>(p, u, kvh, h0, nh);
      bool in_shared = false;
      int row = s;  // the table the block is read through
      if (shared) {  // position j of the unit's work -> the logical block
        const int B = shared_len(s);
        in_shared = j < B;
        if (in_shared) row = s + info_member(s_lead[s]);
        else j = info_off(s_info[s]) + j - B;
      }
      phys = __ldg(bt + (long long)row * p.max_blocks_per_seq + j);
      if (in_shared) {  // every member that takes this block must hold it at the same place
        const int k = info_size(s_info[s]);
        for (int m = 0; m < k; ++m)
          if (j < info_off(s_info[s + m]) && __ldg(bt + (long long)(s + m) * p.max_blocks_per_seq + j) != phys)
            set_error(p.err, kErrShared);
      }
      const bool last_blk = !in_shared && j == (s_len[s] + BS - 1) / BS - 1;
      kvh |= (s << 16) | (static_cast<int>(last_blk) << 30);
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
    const int tag = __shfl_sync(0xffffffffu, kvh_cur, k & 31);
    const int kvh = tag & 0xffff;
    if (phys < 0 || phys >= p.num_blocks) {  // out-of-pool entry: record it, read block 0 instead
      if (lane == 0) set_error(p.err, kErrBlockId);
      phys = 0;
    }
    if (lane == 0) {
      const int st = k % STAGES;
      unsigned char* dst = ring + st * 2 * TILE;
      const long long tile = (long long)phys * p.num_kv_heads + kvh;
      const bool with_token = p.fused && (tag >> 30);
      mbar_arrive_expect_tx(
          &bars[st], 2 * TILE + (with_token ? 2 * D * static_cast<int>(sizeof(TC) == 1 ? sizeof(T) : sizeof(TC)) : 0));
      bulk_copy_g2s(dst, static_cast<const unsigned char*>(p.k_cache) + tile * TILE, TILE, &bars[st]);
      bulk_copy_g2s(dst + TILE, static_cast<const unsigned char*>(p.v_cache) + tile * TILE, TILE, &bars[st]);
      if (with_token) {  // the new token's K and V rows of (sequence, kv head)
        constexpr int kRowBytes = D * static_cast<int>(sizeof(TC) == 1 ? sizeof(T) : sizeof(TC));
        const long long row = ((long long)((tag >> 16) & 0x3fff) * p.num_kv_heads + kvh) * kRowBytes;
        unsigned char* sd = side + st * Sh::kSideStage;
        bulk_copy_g2s(sd, static_cast<const unsigned char*>(p.new_key) + row, kRowBytes, &bars[st]);
        bulk_copy_g2s(sd + kRowBytes, static_cast<const unsigned char*>(p.new_value) + row, kRowBytes, &bars[st]);
      }
    }
  };
  for (int k = 0; k < STAGES && k < len; ++k) issue(k);
  if (p.fused) write_tokens();  // while the first stages are in flight

  // The compute cursor walks the same positions in order.  Its segment is
  // (cs, cu, part); cj is the logical block, running from jstart to jend.
  Math math;
  math.init(lane, pw);
  math.set_columns(p.group);
  int cs, cu, cj;
  locate(start, s_pre, S, U, cs, cu, cj);
  int part = 1;
  if (shared) {  // position cj of the unit's work: in the shared part, or past it in the own part
    const int B = shared_len(cs);
    if (cj < B) part = 0;
    else cj = info_off(s_info[cs]) + cj - B;
  }
  int L = 0, nblk = 0, kvh = 0, h0 = 0, nh = 0, seg = 0, jstart = 0, jend = 0, j0 = cj;
  int my_off = 0;          // lane m < cluster size: the first own block of member m (shared part)
  bool direct_ok = true;   // a whole segment may go straight to the output
  bool folded = false;     // earlier partitions of this piece are in the running state
  auto enter = [&]() {
    L = s_len[cs];
    nblk = (L + BS - 1) / BS;
    unit_heads<kMma>(p, cu, kvh, h0, nh);
    jstart = 0;
    jend = nblk;
    direct_ok = true;
    if (shared) {
      const int v = s_info[cs];
      if (part == 0) {  // the cluster's common blocks, for the query rows of all its members
        const int k = info_size(v);
        nh = k * p.group;
        jend = shared_len(cs);
        my_off = lane < k ? info_off(s_info[cs + lane]) : 0;
        direct_ok = false;
      } else {          // this sequence's own blocks; merged with its shared part when it has one
        jstart = info_off(v);
        direct_ok = jstart == 0;
      }
    }
    seg = seg_id(cs, cu, part);
    math.reset();
    math.load_q(static_cast<const T*>(p.q) + ((long long)cs * p.num_heads + h0) * D, nh, p.scale_log2, p.group,
                (long long)p.num_heads * D);
  };
  enter();

  for (int k = 0; k < len; ++k) {
    if (!wait_stage<STAGES>(bars, never, p.test_wait_ns, k, len, p.err, lane)) break;
    unsigned char* stage = ring + (k % STAGES) * 2 * TILE;
    // valid tokens in this block (>= 1); a shared block is full for every member that takes it
    const int rem = part == 0 ? BS : L - cj * BS;
    if (p.fused && part != 0 && cj == nblk - 1)  // the sequence's new token: from the step's input, not the pool
    {
      if constexpr (sizeof(TC) == 1)
        inject_token_e4m3<T, D, BS>(stage, TILE, side + (k % STAGES) * Sh::kSideStage, (L - 1) % BS,
                                    p.write_k_scale, p.write_v_scale, lane);
      else
        inject_token<TC, D, BS>(stage, TILE, side + (k % STAGES) * Sh::kSideStage, (L - 1) % BS, lane);
    }
    if (rem < BS) zero_tail_v<TC, D, BS>(stage + TILE, rem, lane);
    if constexpr (Math::kFetch) {  // the block's fragments are in registers: refill the stage now
      math.fetch(stage, TILE);
      __syncwarp();
      if (k + STAGES < len) {
        fence_proxy_async_smem();
        issue(k + STAGES);
      }
    }
    // the members whose tables hold this block (every column outside shared parts)
    const uint32_t live = (shared && part == 0) ? __ballot_sync(0xffffffffu, cj < my_off) : 0xffffffffu;
    math.block(stage, TILE, rem, p.scale_log2, live);
    ++cj;
    const bool seg_end = cj == jend, last = k + 1 == len;
    if (seg_end || last) {  // the end of a piece
      math.finish();
      if (folded) {  // close the last caller partition and take the merged state
        math.fold(st_o, st_ml, false);
        math.load_state(st_o, st_ml);
        folded = false;
      }
      if (j0 == jstart && seg_end && direct_ok) {  // the whole segment: straight to the output
        math.store_out(static_cast<T*>(p.out) + ((long long)cs * p.num_heads + h0) * D, nh, p.out_scale);
        if (lane == 0) p.seg_first[seg] = -1;
      } else {
        // pieces start only at warp and segment boundaries, so this slot is unique
        const long long slot = (long long)w + seg;
        math.store_partial(p.part_o + slot * p.rows * D, p.part_ml + slot * p.rows * 2, nh, p.out_scale);
        if (lane == 0) {
          p.part_tag[slot] = make_int2(seg, static_cast<int>(p.epoch));
          if (j0 == jstart) p.seg_first[seg] = static_cast<int>(slot);
          if (seg_end) p.seg_last[seg] = static_cast<int>(slot);
        }
      }
      if (!last) {
        if (part == 0) {  // the shared part is followed by the leader's own part of the unit
          part = 1;
          cj = info_off(s_info[cs]);
        } else {
          if (++cu == U) {
            cu = 0;
            do {
              ++cs;
            } while (s_pre[cs + 1] == s_pre[cs]);
          }
          cj = 0;
          if (shared) {
            part = shared_len(cs) > 0 ? 0 : 1;
            cj = part == 0 ? 0 : info_off(s_info[cs]);
          }
        }
        enter();
        j0 = cj;
      }
    } else if (cj % PB == 0) {  // a caller partition ends inside this piece: fold it
      math.finish();
      math.fold(st_o, st_ml, !folded);
      folded = true;
      math.reset();
    }
    if constexpr (!Math::kFetch) {
      __syncwarp();
      if (k + STAGES < len) {
        fence_proxy_async_smem();
        issue(k + STAGES);
      }
    }
  }
}

// --- merge of pieces --------------------------------------------------------------------------------
//
// One warp per output row (sequence, query head); kMergeRows rows per CTA.  The
// row's pieces are the slots of its own segment and, with shared prefixes, those of
// its cluster's shared part (where the member's rows sit at row offset
// member * group).  Lane i reads the tag and (m, l) of piece i of a chunk of up to
// 32, together with the first batch of the chunk's partial outputs (each lane D/32
// consecutive head dims; 32 registers' worth), so a chunk of 8 pieces costs one trip
// to L2; the chunk's
// maximum and weights come from warp shuffles,
//     m_c = max m_p,  w_p = l_p 2^(m_p - m_c),  l_c = sum w_p,  o_c = sum w_p o_p.  Chunks fold into a running
// (M, L, O) with the same rule; the row is O / L.  Slots whose tag is not (their
// segment, this launch's epoch) weigh nothing and are never read into a sum:
// when the grid has more warps than blocks of work, a warp with an empty range
// leaves its slot inside a segment's range unwritten.  A piece whose rows saw no
// block (a member that holds fewer shared blocks than the piece covers) has
// m = -inf and weighs nothing too.
constexpr int kMergeRows = 8;

//
// kWide (launches whose segments are cut into many pieces, e.g. a few very long
// sequences): one CTA per row instead, its warps taking equal runs of the row's
// pieces, and warp 0 folding their results from shared memory, so that no warp
// walks a long list of pieces alone.
template <typename T, int D, bool kMma, bool kWide>
__global__ void __launch_bounds__(kMergeRows * 32, 2) decode_merge_kernel(const DecodeParams p) {
  constexpr int CPL = D / 32;  // head dims per lane
  using Vec = std::conditional_t<CPL == 4, float4, float2>;
  __shared__ __align__(16) float s_o[kWide ? kMergeRows : 1][D];
  __shared__ float s_m[kMergeRows], s_l[kMergeRows];
  griddep_wait();
  griddep_launch_dependents();
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const long long row = kWide ? (long long)blockIdx.x : (long long)blockIdx.x * kMergeRows + warp;
  if (row >= (long long)p.num_seqs * p.num_heads) return;  // (wide: the whole CTA)
  const int s = static_cast<int>(row / p.num_heads), h = static_cast<int>(row - (long long)s * p.num_heads);
  // the head unit of h and h's row within it
  int u, r;
  if (kMma) {
    const int kvh = h / p.group, hh = h - kvh * p.group;
    u = kvh * ((p.group + 15) >> 4) + (hh >> 4);
    r = hh & 15;
  } else {
    u = h;
    r = 0;
  }
  const int b = s * p.units + u;
  const bool shared = kMma && p.shared;
  const int own = shared ? 2 * b + 1 : b;
  int first = p.seg_first[own], last = p.seg_last[own];
  const bool own_ok = first >= 0 && last >= first && last < p.num_slots;
  if (!own_ok && first >= 0) return;  // an aborted launch
  if (!own_ok) {                      // the own part went straight to the output
    first = 0;
    last = -1;
  }
  // the cluster's shared part, if this sequence takes any of its blocks
  int sfirst = 0, slast = -1, srow = 0, sseg = -1;
  if (shared) {
    const int v = p.seq_info[s], mi = info_member(v);
    if (info_off(v) > 0) {  // its leader is s - mi
      sseg = 2 * ((s - mi) * p.units + u);
      sfirst = p.seg_first[sseg];
      slast = p.seg_last[sseg];
      srow = mi * p.group;
      if (sfirst < 0 || slast < sfirst || slast >= p.num_slots) slast = sfirst - 1;  // (an aborted launch)
    }
  }
  const int Ks = slast - sfirst + 1;
  const int K = Ks + (last - first + 1);
  if (K <= 0) return;  // (wide: the whole CTA, every warp computed the same)
  // the pieces this warp folds
  const int lo = kWide ? (K * warp) / kMergeRows : 0, hi = kWide ? (K * (warp + 1)) / kMergeRows : K;
  const int ep = static_cast<int>(p.epoch);
  // piece i: the offset of its row in the partial arrays, and the segment that must have written it
  const long long at_s = (long long)sfirst * p.rows + srow + r, at_o = (long long)(first - Ks) * p.rows + r;
  auto piece = [&](int i, long long& at, int& seg) {
    at = (i < Ks ? at_s : at_o) + (long long)i * p.rows;
    seg = i < Ks ? sseg : own;
  };

  float RM = -INFINITY, RL = 0.f, RO[CPL];
#pragma unroll
  for (int c = 0; c < CPL; ++c) RO[c] = 0.f;
  constexpr int kBatch = 32 / CPL;  // partial outputs in flight per lane (32 registers)
  for (int c0 = lo; c0 < hi; c0 += 32) {
    const int n = min(32, hi - c0);
    // the tags and (m, l) of the chunk and the first batch of its partial outputs, all in flight at once
    float m = -INFINITY, l = 0.f;
    int2 tag = make_int2(-1, 0);
    int sg_mine = -1;
    float2 ml = make_float2(0.f, 0.f);
    if (lane < n) {
      long long at;
      piece(c0 + lane, at, sg_mine);
      tag = p.part_tag[at / p.rows];
      ml = *reinterpret_cast<const float2*>(p.part_ml + at * 2);
    }
    Vec ov[kBatch];
#pragma unroll
    for (int i = 0; i < kBatch; ++i)
      if (i < n) {
        long long at;
        int sg;
        piece(c0 + i, at, sg);
        ov[i] = *reinterpret_cast<const Vec*>(p.part_o + at * D + CPL * lane);
      }
    if (lane < n && tag.x == sg_mine && tag.y == ep) {
      m = ml.x;
      l = ml.y;
    }
    float mc = m;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) mc = fmaxf(mc, __shfl_xor_sync(0xffffffffu, mc, o));
    const float w = m == -INFINITY ? 0.f : l * exp2f(m - mc);
    float lc = w;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) lc += __shfl_xor_sync(0xffffffffu, lc, o);
    float oc[CPL];
#pragma unroll
    for (int c = 0; c < CPL; ++c) oc[c] = 0.f;
    for (int i0 = 0; i0 < n; i0 += kBatch) {
      if (i0 > 0) {  // the next batch of partial outputs
#pragma unroll
        for (int i = 0; i < kBatch; ++i)
          if (i0 + i < n) {
            long long at;
            int sg;
            piece(c0 + i0 + i, at, sg);
            ov[i] = *reinterpret_cast<const Vec*>(p.part_o + at * D + CPL * lane);
          }
      }
#pragma unroll
      for (int i = 0; i < kBatch; ++i) {
        const float wi = __shfl_sync(0xffffffffu, w, (i0 + i) & 31);
        if (i0 + i < n && wi > 0.f) {  // a slot no piece wrote in this launch holds anything (NaN too)
          const float* v = reinterpret_cast<const float*>(&ov[i]);
#pragma unroll
          for (int c = 0; c < CPL; ++c) oc[c] = fmaf(wi, v[c], oc[c]);
        }
      }
    }
    if (lc > 0.f) {
      const float mn = fmaxf(RM, mc);
      const float fa = exp2f(RM - mn), fb = exp2f(mc - mn);
      RL = RL * fa + lc * fb;
#pragma unroll
      for (int c = 0; c < CPL; ++c) RO[c] = RO[c] * fa + fb * oc[c];
      RM = mn;
    }
  }
  if constexpr (kWide) {  // warp 0 folds the warps' results
    if (lane == 0) {
      s_m[warp] = RM;
      s_l[warp] = RL;
    }
#pragma unroll
    for (int c = 0; c < CPL; ++c) s_o[warp][CPL * lane + c] = RO[c];
    __syncthreads();
    if (warp != 0) return;
    RM = -INFINITY;
    RL = 0.f;
#pragma unroll
    for (int c = 0; c < CPL; ++c) RO[c] = 0.f;
    for (int j = 0; j < kMergeRows; ++j) {
      if (!(s_l[j] > 0.f)) continue;
      const float mn = fmaxf(RM, s_m[j]);
      const float fa = exp2f(RM - mn), fb = exp2f(s_m[j] - mn);
      RL = RL * fa + s_l[j] * fb;
#pragma unroll
      for (int c = 0; c < CPL; ++c) RO[c] = RO[c] * fa + fb * s_o[j][CPL * lane + c];
      RM = mn;
    }
  }
  const float il = 1.f / RL;
  T* out = static_cast<T*>(p.out) + row * D + CPL * lane;
#pragma unroll
  for (int c = 0; c < CPL; ++c) out[c] = DType<T>::from_f32(RO[c] * il);
}

// --- host-side launch helpers (instantiated per dtype) ------------------------------------------

template <typename TC, int D, int BS, int kMode>
constexpr int decode_smem_bytes() {
  return DecodeShape<TC, D, BS, kMode>::kSmemBytes;
}

template <typename T, typename TC, int D, int BS, int kMode>
cudaError_t ensure_smem_attr() {
  static unsigned done = 0;  // bit d: set on device d
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 32 && ((__atomic_load_n(&done, __ATOMIC_ACQUIRE) >> dev) & 1u)) return cudaSuccess;
  e = cudaFuncSetAttribute(reinterpret_cast<const void*>(&decode_kernel<T, TC, D, BS, kMode>),
                           cudaFuncAttributeMaxDynamicSharedMemorySize, decode_smem_bytes<TC, D, BS, kMode>());
  if (e == cudaSuccess && dev < 32) __atomic_fetch_or(&done, 1u << dev, __ATOMIC_RELEASE);
  return e;
}

template <typename T, typename TC, int D, int BS, int kMode>
int decode_ctas_per_sm_t() {
  if (ensure_smem_attr<T, TC, D, BS, kMode>() != cudaSuccess) return 0;
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, &decode_kernel<T, TC, D, BS, kMode>,
                                                    DecodeShape<TC, D, BS, kMode>::kWarps * 32,
                                                    decode_smem_bytes<TC, D, BS, kMode>()) != cudaSuccess)
    return 0;
  return n;
}

template <typename T, typename TC, int D, int BS, int kMode>
cudaError_t launch_decode_t(const DecodeParams& p, int grid, cudaStream_t stream, int* launches) {
  *launches = 0;
  cudaError_t e = ensure_smem_attr<T, TC, D, BS, kMode>();
  if (e != cudaSuccess) return e;
  e = launch_pdl(decode_kernel<T, TC, D, BS, kMode>, dim3(grid), dim3(DecodeShape<TC, D, BS, kMode>::kWarps * 32),
                 decode_smem_bytes<TC, D, BS, kMode>(), stream, p);
  if (e != cudaSuccess) return e;
  *launches = 1;
  // rows whose segments average 16 pieces or more (a few very long sequences) take a CTA each
  const long long rows = (long long)p.num_seqs * p.num_heads;
  const long long segs = (long long)p.num_seqs * p.units;
  const bool wide = (long long)grid * DecodeShape<TC, D, BS, kMode>::kWarps >= 16 * segs;
  if (wide)
    e = launch_pdl(decode_merge_kernel<T, D, (kMode != 0), true>, dim3(static_cast<unsigned>(rows)),
                   dim3(kMergeRows * 32), 0, stream, p);
  else
    e = launch_pdl(decode_merge_kernel<T, D, (kMode != 0), false>,
                   dim3(static_cast<unsigned>((rows + kMergeRows - 1) / kMergeRows)), dim3(kMergeRows * 32), 0, stream,
                   p);
  if (e != cudaSuccess) return e;
  *launches = 2;
  return cudaSuccess;
}

// fp32 caches use the CUDA-core math only; 16-bit and FP8 caches both kinds.
template <typename T, typename TC, int D, int BS>
int ctas_for(DecodeKind kind) {
  if constexpr (sizeof(T) == 4) {
    return decode_ctas_per_sm_t<T, TC, D, BS, 0>();
  } else {
    switch (kind) {
      case DecodeKind::kMma8: return decode_ctas_per_sm_t<T, TC, D, BS, 1>();
      case DecodeKind::kMma16: return decode_ctas_per_sm_t<T, TC, D, BS, 2>();
      default: return decode_ctas_per_sm_t<T, TC, D, BS, 0>();
    }
  }
}

template <typename T, typename TC, int D, int BS>
cudaError_t launch_for(const DecodeParams& p, DecodeKind kind, int grid, cudaStream_t s, int* n) {
  if constexpr (sizeof(T) == 4) {
    return launch_decode_t<T, TC, D, BS, 0>(p, grid, s, n);
  } else {
    switch (kind) {
      case DecodeKind::kMma8: return launch_decode_t<T, TC, D, BS, 1>(p, grid, s, n);
      case DecodeKind::kMma16: return launch_decode_t<T, TC, D, BS, 2>(p, grid, s, n);
      default: return launch_decode_t<T, TC, D, BS, 0>(p, grid, s, n);
    }
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
