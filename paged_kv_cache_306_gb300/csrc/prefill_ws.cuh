// prefill_ws.cuh -- chunked prefill on tcgen05 with warp specialisation.
//
// Causal attention of each sequence's chunk of new query tokens over its paged
// cache (what is computed: see prefill.cu), on sm_103a's tcgen05 MMAs with the
// accumulators in tensor memory (TMEM).  A query tile is 128 rows -- (token,
// query head) pairs of one kv head, head fastest -- which are TMEM lanes
// 0..127; keys are taken 64 at a time (a chunk).  A CTA owns a PAIR of
// consecutive tiles of one (sequence, kv head): both read the same keys, so each
// chunk of K and V is copied once and feeds the MMAs of both tiles, and while
// the tensor cores work for one tile the softmax of the other runs.  The phases
// run in different warps that hand over through mbarriers:
//
//   * warp 8, one thread: the TMA copies of chunk c, through two tensor maps: K
//     into K buffer c % 4 once both tiles' S of chunk c - 4 have read it, V into V
//     buffer c % 4 once both tiles' P V of chunk c - 4 have read it, each on its own
//     mbarrier, so S waits only for K and the V copies are well ahead.  K: the pool seen
//     as rows of 16 keys x 8 dims (one 256-byte run of a K tile [D/8][bs][8]); one
//     tile::gather4 load per 8-dim chunk fetches the rows of the chunk's 64 keys
//     (from up to four blocks anywhere in the pool) and lands them as [64][8]:
//     the K operand of S = Q K^T becomes [D/8][64 keys][8], core matrices with one
//     uniform stride, so S is one MMA of N = 64 per 16 dims (a block-by-block S
//     of N = bs took four times the MMAs and was the largest cost).  V: the pool
//     seen as rows of bs keys (one dim of a V tile [D][bs]); each [D rows x 8 keys]
//     box lands as [D][8], one 8-key group of the [key/8][D][8] layout the P V MMA
//     reads.  No re-layout pass.
//   * warp 9, one thread: for each chunk c, S_A(c) and S_B(c) = Q K^T into each
//     tile's TMEM columns S[c % 2] (once chunk c has landed and that tile's
//     P V(c - 2), which read P from those columns, is done), then O_A += P V(c - 1)
//     and O_B += P V(c - 1) with P read from TMEM; each group is committed to
//     mbarriers.  Tile A's softmax of chunk c thus runs under S_B(c), the P V of
//     chunk c - 1 and the S of chunk c + 1 of both tiles.
//   * warps 0..3 (tile A) and 4..7 (tile B), one thread per row: the softmax of
//     S(c).  P = exp2(s - m) goes back into the row's own S
//     columns as rounded 16-bit high and low parts (two per 32-bit column).  The
//     running maximum moves only when it grows by more than 2^8; then the row's O
//     is rescaled in TMEM after P V(c - 1) has finished (rare).  In the last chunk
//     tile A's threads zero the V of keys past the sequence (or past the blocks
//     loaded) in shared memory first: P is 0 there, but 0 * NaN would poison O.
//     A tile whose rows end before the pair's last chunks sees scores of -inf
//     there (P = 0).
//
// TMEM: per tile two S/P column groups of 64 and O (D <= 128 columns) in 256, all
// 512 columns for the pair; one CTA per SM.
// Every wait is bounded (1 s of %globaltimer); a thread that gives up records
// PA_DEVERR_TIMEOUT and raises a CTA-wide abort flag that makes every other wait
// give up at once; the threads that issued copies or MMAs then wait (bounded)
// for them before TMEM is freed.
#pragma once

#include <cuda.h>

#include "pa_device.cuh"
#include "pa_launch.h"
#include "tc_ops.cuh"

namespace pa {
namespace ws {

using tc::commit;
using tc::elect_one;
using tc::fence_after;
using tc::fence_before;
using tc::idesc;
using tc::ld32;
using tc::mma;
using tc::sdesc;
using tc::st32;

constexpr int kRows = 128;  // query rows per tile (= TMEM lanes)
constexpr int kKeys = 64;   // keys per chunk
constexpr int kSoftmaxThreads = 128;  // per tile
constexpr int kProducerWarp = 8, kMmaWarp = 9;
constexpr int kThreads = 10 * 32;
constexpr int kKStages = 4, kVStages = 4;
constexpr uint64_t kWaitNs = 1000000000ull;

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

// tcgen05 MMA with the A operand in TMEM (row i in lane i, two 16-bit K elements per column)
__device__ __forceinline__ void mma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b, uint32_t id, bool accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.u32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b), "r"(id), "r"((uint32_t)accumulate));
}

// 64 consecutive fp32 columns of this thread's TMEM lane: two loads, one wait
__device__ __forceinline__ void ld64(uint32_t taddr, float (&v)[64]) {
  uint32_t r[64];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%64];\n\t"
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%32,%33,%34,%35,%36,%37,%38,%39,%40,%41,%42,%43,%44,%45,%46,%47,"
      "%48,%49,%50,%51,%52,%53,%54,%55,%56,%57,%58,%59,%60,%61,%62,%63}, [%65];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
        "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
        "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31]),
        "=r"(r[32]), "=r"(r[33]), "=r"(r[34]), "=r"(r[35]), "=r"(r[36]), "=r"(r[37]), "=r"(r[38]), "=r"(r[39]),
        "=r"(r[40]), "=r"(r[41]), "=r"(r[42]), "=r"(r[43]), "=r"(r[44]), "=r"(r[45]), "=r"(r[46]), "=r"(r[47]),
        "=r"(r[48]), "=r"(r[49]), "=r"(r[50]), "=r"(r[51]), "=r"(r[52]), "=r"(r[53]), "=r"(r[54]), "=r"(r[55]),
        "=r"(r[56]), "=r"(r[57]), "=r"(r[58]), "=r"(r[59]), "=r"(r[60]), "=r"(r[61]), "=r"(r[62]), "=r"(r[63])
      : "r"(taddr), "r"(taddr + 32)
      : "memory");
#pragma unroll
  for (int i = 0; i < 64; ++i) v[i] = __uint_as_float(r[i]);
}

// 2^x by the hardware's approximate exponential (|relative error| below 2^-22; 2^-inf = 0)
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// 2-D tensor-map copy global -> shared (box at element coordinates x, y)
__device__ __forceinline__ void tma_2d_g2s(void* dst, const CUtensorMap* map, int x, int y, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
          smem_addr(dst)),
      "l"(map), "r"(x), "r"(y), "r"(smem_addr(bar))
      : "memory");
}

// tile::gather4 tensor-map copy: four rows (element row indices rows[0..3]) of a 2-D
// map whose box is one row high, landing one after another in shared memory
__device__ __forceinline__ void tma_gather4_g2s(void* dst, const CUtensorMap* map, const int (&rows)[4], uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile::gather4.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, "
      "%4, %5, %6}], [%7];" ::"r"(smem_addr(dst)),
      "l"(map), "r"(0), "r"(rows[0]), "r"(rows[1]), "r"(rows[2]), "r"(rows[3]), "r"(smem_addr(bar))
      : "memory");
}

// A bounded wait that also gives up at once when another thread of the CTA has
// given up (*abort set); a thread that times out sets *abort and records the error.
__device__ __forceinline__ bool wait_or_abort(uint64_t* bar, uint32_t parity, volatile int* abort, unsigned* err,
                                              uint64_t limit_ns = kWaitNs) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  while (true) {
#pragma unroll 1
    for (int i = 0; i < 32; ++i)
      if (mbar_try_wait(bar, parity)) return true;
    if (*abort) return false;
    if (global_timer_ns() - t0 > limit_ns) {
      *abort = 1;
      set_error(err, kErrTimeout);
      return false;
    }
  }
}

// The pair of rank `rank` (0-based) in the order of decreasing length -- the chunks
// of keys it reads -- ties by sequence, kv head and pair index; so the longest
// pairs of the whole launch start first and the short ones fill the tail.  Every
// thread of the CTA takes part (thread t owns sequences t * kPer ..).  Tile j of
// sequence s covers rows 128 j .. of its n * G rows and reads chunks
// 0 .. (ctx + (row_hi - 1) / G) / 64, non-decreasing in j; pair k holds tiles 2k and
// 2k + 1 (if there is one) and reads what its last tile reads.  So the tiles of s
// reading >= x chunks are a suffix j >= j0 in closed form, the pairs reading >= x
// are those from j0 / 2 on, and the rank-th pair is found by a binary search on x.
// Writes (sequence, kv head, pair) to out; returns false when rank is past the pairs.
__device__ bool pick_pair(const PrefillParams& p, int rank, int* red, int* out) {
  constexpr int kPer = (kMaxSeqsPerLaunch + kThreads - 1) / kThreads;
  constexpr int kWarpsTotal = kThreads / 32;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int G = p.group, Hkv = p.num_kv_heads;
  int ctx[kPer], rows[kPer], nt[kPer];
  bool bad = false;
#pragma unroll
  for (int i = 0; i < kPer; ++i) {
    const int s = tid * kPer + i;
    ctx[i] = rows[i] = nt[i] = 0;
    if (s < p.num_seqs) {
      const int L = __ldg(p.seq_lens + s), a = __ldg(p.query_start_loc + s), b = __ldg(p.query_start_loc + s + 1);
      const int n = b - a;
      if (L < 1 || L > p.max_seq_len || a < 0 || b > p.num_query_tokens || n < 0 || n > L) {
        bad = true;
      } else {
        ctx[i] = L - n;
        rows[i] = n * G;
        nt[i] = (rows[i] + kRows - 1) / kRows;
      }
    }
  }
  if (bad && blockIdx.x == 0) set_error(p.err, kErrSeqLen);
  // pairs of owned sequence i that read >= x chunks
  auto cnt = [&](int i, int x) -> int {
    const long long need = (long long)G * (64LL * (x - 1) - ctx[i]) + 1;  // rows a tile must reach
    if (nt[i] == 0 || need > rows[i]) return 0;
    const int j0 = need <= 1 ? 0 : static_cast<int>((need + kRows - 1) / kRows - 1);  // first tile reading >= x
    return (nt[i] + 1) / 2 - j0 / 2;
  };
  int buf = 0;
  auto reduce = [&](int v, bool take_max) -> int {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const int u = __shfl_xor_sync(0xffffffffu, v, o);
      v = take_max ? max(v, u) : v + u;
    }
    buf ^= 1;
    if (lane == 0) red[buf * 16 + warp] = v;
    __syncthreads();
    int t = 0;
#pragma unroll
    for (int w = 0; w < kWarpsTotal; ++w) t = take_max ? max(t, red[buf * 16 + w]) : t + red[buf * 16 + w];
    return t;
  };
  int local = 0, longest = 0;
#pragma unroll
  for (int i = 0; i < kPer; ++i) {
    local += (nt[i] + 1) / 2;
    if (nt[i]) longest = max(longest, (ctx[i] + (rows[i] - 1) / G) / 64 + 1);
  }
  if ((long long)Hkv * reduce(local, false) <= rank) return false;
  int lo = 1, hi = reduce(longest, true);  // C(lo) > rank
  while (lo < hi) {
    const int mid = (lo + hi + 1) / 2;
    local = 0;
#pragma unroll
    for (int i = 0; i < kPer; ++i) local += cnt(i, mid);
    if ((long long)Hkv * reduce(local, false) > rank) lo = mid;
    else hi = mid - 1;
  }
  // rank among the pairs of exactly lo chunks, ordered by (sequence, kv head, pair)
  local = 0;
#pragma unroll
  for (int i = 0; i < kPer; ++i) local += cnt(i, lo + 1);
  const long long r = rank - (long long)Hkv * reduce(local, false);
  int e[kPer], mine = 0;
#pragma unroll
  for (int i = 0; i < kPer; ++i) {
    e[i] = cnt(i, lo) - cnt(i, lo + 1);
    mine += e[i];
  }
  int incl = mine;  // inclusive scan over threads (sequence order)
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int u = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += u;
  }
  buf ^= 1;
  if (lane == 31) red[buf * 16 + warp] = incl;
  __syncthreads();
  long long before = incl - mine;
  for (int w = 0; w < warp; ++w) before += red[buf * 16 + w];
  before *= Hkv;
#pragma unroll
  for (int i = 0; i < kPer; ++i) {
    const long long span = (long long)Hkv * e[i];
    if (r >= before && r < before + span) {
      const int q = static_cast<int>(r - before);
      out[0] = tid * kPer + i;
      out[1] = q / e[i];
      out[2] = (nt[i] + 1) / 2 - cnt(i, lo) + q % e[i];
    }
    before += span;
  }
  __syncthreads();
  return true;
}

template <typename T, int D, int BS>
struct Shape {
  static constexpr int kTile = D * BS * 2;                 // one block's K (or V) tile
  static constexpr int kBlocks = kKeys / BS;               // blocks per chunk
  static constexpr int kQTile = kRows * D * 2;             // one tile's Q, core-matrix layout
  static constexpr int kKBytes = kKeys * D * 2;  // a chunk's K as [D/8][64][8]
  static constexpr int kVBytes = kKeys * D * 2;  // a chunk's V as [key/8][D][8]
  static constexpr int kOffK = 2 * kQTile;                  // K ring
  static constexpr int kOffV = kOffK + kKStages * kKBytes;  // V ring
  static constexpr int kOffBar = kOffV + kVStages * kVBytes;
  // fullk[K], fullv[V], kfree[K], vfree[V], per tile sfull[2], pfull[2], pvdone[2], never
  static constexpr int kNumBars = 2 * kKStages + 2 * kVStages + 2 * 6 + 1;
  static constexpr int kOffRed = kOffBar + kNumBars * 8 + 32;  // [2][16] ints: block reductions
  // more than half an SM's shared memory, so one CTA per SM: it takes all of TMEM
  static constexpr int kSmem = kOffRed + 2 * 16 * 4 > 116 * 1024 ? kOffRed + 2 * 16 * 4 : 116 * 1024;
  static constexpr int kTmemCols = 512;  // tile X at 256 X: S/P[0] 0..63, S/P[1] 64..127, O 128..128+D
};

template <typename T, int D, int BS>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_ws_kernel(const PrefillParams p, const __grid_constant__ CUtensorMap tmap_k,
                      const __grid_constant__ CUtensorMap tmap_v) {
  using Sh = Shape<T, D, BS>;
  static_assert(Sh::kSmem > 114 * 1024, "two CTAs on one SM would contend for TMEM");
  extern __shared__ __align__(1024) unsigned char smem[];
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + Sh::kOffBar);
  uint64_t* fullk = bars;                   // [kKStages] K buffer landed (TMA bytes)
  uint64_t* fullv = fullk + kKStages;       // [kVStages] V buffer landed (TMA bytes)
  uint64_t* kfree = fullv + kVStages;       // [kKStages] both tiles' S read the K buffer (commit)
  uint64_t* vfree = kfree + kKStages;       // [kVStages] both tiles' P V read the V buffer (commit)
  uint64_t* tbars = vfree + kVStages;       // per tile X at 6 X: sfull[2], pfull[2], pvdone[2]
  uint64_t* never = tbars + 12;             // nothing completes it: the timeout-path test waits on it
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(bars + Sh::kNumBars);
  int* s_pair = reinterpret_cast<int*>(s_tmem + 1);                     // sequence, kv head, pair (or -1)
  volatile int* s_abort = reinterpret_cast<volatile int*>(s_pair + 3);  // a thread gave up
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  // S in TMEM, the K buffer read (commit); P in TMEM, O rescaled, V tail zeroed (128 arrivals);
  // P V done: P's columns and O free (commit)
  auto sfull = [&](int X, int i) { return tbars + 6 * X + i; };
  auto pfull = [&](int X, int i) { return tbars + 6 * X + 2 + i; };
  auto pvdone = [&](int X, int i) { return tbars + 6 * X + 4 + i; };

  griddep_launch_dependents();
  griddep_wait();

  // ---- which pair: the longest first over the whole launch
  const bool has_pair = pick_pair(p, static_cast<int>(blockIdx.x), reinterpret_cast<int*>(smem + Sh::kOffRed), s_pair);
  if (tid == 0) {
    if (!has_pair) s_pair[0] = -1;
    *s_abort = 0;
    for (int i = 0; i < kKStages; ++i) {
      mbar_init(&fullk[i], 1);
      mbar_init(&kfree[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      for (int X = 0; X < 2; ++X) {
        mbar_init(sfull(X, i), 1);
        mbar_init(pfull(X, i), kSoftmaxThreads);
        mbar_init(pvdone(X, i), 1);
      }
    }
    for (int i = 0; i < kVStages; ++i) {
      mbar_init(&fullv[i], 1);
      mbar_init(&vfree[i], 1);
    }
    mbar_init(never, 1);
    fence_barrier_init();
  }
  __syncthreads();
  const int s = s_pair[0];
  if (s < 0) return;  // no pair for this CTA (before any TMEM is taken)
  const int kvh = s_pair[1], pair = s_pair[2];
  const int G = p.group;
  const int L = p.seq_lens[s], tok0 = p.query_start_loc[s], n = p.query_start_loc[s + 1] - tok0;
  const int rows = n * G, pair_lo = 2 * pair * kRows, pair_hi = min(rows, pair_lo + 2 * kRows);
  const bool two = pair_lo + kRows < rows;    // the pair has a tile B
  const int ctx = L - n;
  const int p_max = ctx + (pair_hi - 1) / G;  // last position any row of the pair has
  const int nblk = p_max / BS + 1;            // blocks holding keys 0..p_max
  const int nchunks = (p_max + kKeys) / kKeys;

  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_addr(s_tmem)),
                 "r"(Sh::kTmemCols));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  // the softmax threads' tile and row; Q of both tiles into shared memory (core matrices: 8 rows x 16 bytes)
  const int X = tid >= kSoftmaxThreads ? 1 : 0;  // (softmax threads only)
  const int r = tid & (kRows - 1), row = pair_lo + X * kRows + r;
  const bool valid = row < pair_hi;
  if (tid < 2 * kSoftmaxThreads) {
    unsigned char* sQ = smem + X * Sh::kQTile;
    const T* q = static_cast<const T*>(p.q) +
                 ((long long)(tok0 + (valid ? row / G : 0)) * p.num_heads + (long long)kvh * G + (valid ? row % G : 0)) * D;
#pragma unroll
    for (int c = 0; c < D / 8; ++c) {
      const uint4 v = valid ? __ldg(reinterpret_cast<const uint4*>(q) + c) : make_uint4(0, 0, 0, 0);
      *reinterpret_cast<uint4*>(sQ + (r / 8) * (D / 8) * 128 + c * 128 + (r % 8) * 16) = v;
    }
  }
  fence_proxy_async_smem();  // Q's generic stores before the MMAs read it
  fence_before();
  __syncthreads();
  fence_after();
  const uint32_t tmem = *s_tmem;
  auto wait = [&](uint64_t* bar, int parity) { return wait_or_abort(bar, parity, s_abort, p.err); };
  int issued_k = 0, issued_v = 0;  // chunks whose K (V) copies the producer issued

  if (warp < 8) {
    // ================= softmax: tile X, row r, all keys of each chunk =================
    if (X == 0 || two) {
      const uint32_t tbase = tmem + 256 * X;
      const uint32_t t_o = tbase + 2 * kKeys;
      const int pos = valid ? ctx + row / G : ctx + (pair_hi - 1) / G;  // a padding row behaves as a real one
      const int kz = min(L, nblk * BS);  // first key whose V must read as zero
      const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
      const float sl2 = p.scale_log2;
      float m = -INFINITY, l = 0.f;
      bool ok = true;
      for (int c = 0; c < nchunks; ++c) {
        const int sb = c & 1;
        // tcgen05.ld / st are warp-collective (.sync.aligned): every branch around them
        // is taken by the whole warp, so each wait's outcome is agreed across the warp
        if (!__all_sync(0xffffffffu, wait(sfull(X, sb), (c >> 1) & 1))) {
          ok = false;
          break;
        }
        fence_after();
        const uint32_t t_s = tbase + lane_base + sb * kKeys;
        float sv[kKeys];
        ld64(t_s, sv);
        const int lim = pos - c * kKeys;  // keys 0..lim of the chunk are visible to the row
        if (lim < kKeys - 1) {           // the diagonal chunk (or past it): hide the later keys
#pragma unroll
          for (int j = 0; j < kKeys; ++j)
            if (j > lim) sv[j] = -INFINITY;
        }
        // the row maximum of the raw scores, as a tree (scale > 0 keeps the order)
        float mx;
        {
          float t[8];
#pragma unroll
          for (int i = 0; i < 8; ++i) t[i] = sv[i];
#pragma unroll
          for (int j = 8; j < kKeys; ++j) t[j & 7] = fmaxf(t[j & 7], sv[j]);
          mx = fmaxf(fmaxf(fmaxf(t[0], t[1]), fmaxf(t[2], t[3])), fmaxf(fmaxf(t[4], t[5]), fmaxf(t[6], t[7]))) * sl2;
        }
        float corr = 1.f;
        const bool move = mx > m + 8.f;
        if (move) {
          corr = m == -INFINITY ? 0.f : exp2f(m - mx);
          m = mx;
          l *= corr;
        }
        // O holds P V up to chunk c - 1 once that group is done: rescale the row if the maximum moved
        // (the whole warp takes the branch when one of its rows needs it; the others scale by 1)
        const bool rescale = c > 0 && move && corr != 1.f;
        if (__any_sync(0xffffffffu, rescale)) {
          if (!__all_sync(0xffffffffu, wait(pvdone(X, (c - 1) & 1), ((c - 1) >> 1) & 1))) {
            ok = false;
            break;
          }
          fence_after();
          const float f = rescale ? corr : 1.f;
#pragma unroll
          for (int c0 = 0; c0 < D; c0 += 32) {
            float o[32];
            ld32(t_o + lane_base + c0, o);
#pragma unroll
            for (int j = 0; j < 32; ++j) o[j] *= f;
            st32(t_o + lane_base + c0, o);
          }
        }
        // P into the row's S columns: high parts in 0..31, low parts in 32..63
        {
          float hi[32], lo[32];
          float ps[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
          for (int j = 0; j < 32; ++j) {  // P = 2^(scale * s - m), s = -inf gives 0
            const float x0 = ex2(fmaf(sv[2 * j], sl2, -m)), x1 = ex2(fmaf(sv[2 * j + 1], sl2, -m));
            ps[j & 3] += x0 + x1;
            const uint32_t h = pack2<T>(x0, x1);
            const float2 back = unpack2<T>(h);
            hi[j] = __uint_as_float(h);
            lo[j] = __uint_as_float(pack2<T>(x0 - back.x, x1 - back.y));
          }
          st32(t_s, hi);
          st32(t_s + 32, lo);
          l += (ps[0] + ps[1]) + (ps[2] + ps[3]);
        }
        // the last chunk: V of keys past the sequence (or past the blocks loaded) reads as
        // zero; tile A's threads clear it before either tile's P V of the chunk is issued
        if (X == 0 && c == nchunks - 1 && kz < (c + 1) * kKeys) {
          if (!__all_sync(0xffffffffu, wait(&fullv[c % kVStages], (c / kVStages) & 1))) {
            ok = false;
            break;
          }
          unsigned char* vbase = smem + Sh::kOffV + (c % kVStages) * Sh::kVBytes;
          const int k0 = kz - c * kKeys, cnt = (kKeys - k0) * D;
          for (int i = tid; i < cnt; i += kSoftmaxThreads) {
            const int kk = k0 + i / D, d = i % D;
            *reinterpret_cast<T*>(vbase + (kk / 8) * (D * 16) + d * 16 + (kk % 8) * 2) = DType<T>::from_f32(0.f);
          }
          fence_proxy_async_smem();
        }
        fence_before();
        mbar_arrive(pfull(X, sb));
      }
      if (__all_sync(0xffffffffu, ok && wait(pvdone(X, (nchunks - 1) & 1), ((nchunks - 1) >> 1) & 1))) {
        fence_after();
        const float inv = 1.f / l;
        T* out = static_cast<T*>(p.out) +
                 ((long long)(tok0 + (valid ? row / G : 0)) * p.num_heads + (long long)kvh * G + (valid ? row % G : 0)) *
                     D;
#pragma unroll
        for (int c0 = 0; c0 < D; c0 += 32) {
          float o[32];
          ld32(t_o + lane_base + c0, o);
          if (valid) {
#pragma unroll
            for (int j = 0; j < 32; j += 8) {
              uint4 w;
              w.x = pack2<T>(o[j] * inv, o[j + 1] * inv);
              w.y = pack2<T>(o[j + 2] * inv, o[j + 3] * inv);
              w.z = pack2<T>(o[j + 4] * inv, o[j + 5] * inv);
              w.w = pack2<T>(o[j + 6] * inv, o[j + 7] * inv);
              *reinterpret_cast<uint4*>(out + c0 + j) = w;
            }
          }
        }
      }
    }
  } else if (warp == kProducerWarp) {
    // ================= TMA copies of chunk c =================
    if (lane == 0) {
      const int32_t* bt = p.block_tables + (long long)s * p.max_blocks_per_seq;
      int phys[Sh::kBlocks];
      auto load_table = [&](int c) {
#pragma unroll
        for (int b = 0; b < Sh::kBlocks; ++b) {
          const int gb = c * Sh::kBlocks + b;
          phys[b] = gb < nblk ? __ldg(bt + gb) : -1;
        }
      };
      load_table(0);
      bool ok = true;
      for (int c = 0; c < nchunks; ++c) {
        const int kb = c % kKStages;
        if (c >= kKStages && !wait(&kfree[kb], ((c - kKStages) / kKStages) & 1)) {  // both tiles' S read it
          ok = false;
          break;
        }
        unsigned char* sk = smem + Sh::kOffK + kb * Sh::kKBytes;
        const int vb = c % kVStages;
        unsigned char* sv_ = smem + Sh::kOffV + vb * Sh::kVBytes;
        int nv = 0;
        long long tl[Sh::kBlocks];
#pragma unroll
        for (int b = 0; b < Sh::kBlocks; ++b) {
          int ph = phys[b];
          if (c * Sh::kBlocks + b < nblk) {
            ++nv;
            if (ph < 0 || ph >= p.num_blocks) {
              set_error(p.err, kErrBlockId);
              ph = 0;
            }
          } else {
            ph = phys[0] < 0 || phys[0] >= p.num_blocks ? 0 : phys[0];  // a block past the keys: any rows do
          }
          tl[b] = (long long)ph * p.num_kv_heads + kvh;
        }
        mbar_arrive_expect_tx(&fullk[kb], Sh::kKBytes);
        // K: per 8-dim chunk dc, the rows (16 keys each) of the chunk's 64 keys
#pragma unroll
        for (int dc = 0; dc < D / 8; ++dc) {
          int rw[4];
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const int b = (16 * q) / BS, h = (16 * q) % BS / 16;
            rw[q] = static_cast<int>((tl[b] * (D / 8) + dc) * (BS / 16) + h);
          }
          tma_gather4_g2s(sk + dc * (kKeys * 16), &tmap_k, rw, &fullk[kb]);
        }
        issued_k = c + 1;
        if (c >= kVStages && !wait(&vfree[vb], ((c - kVStages) / kVStages) & 1)) {  // both tiles' P V read it
          ok = false;
          break;
        }
        mbar_arrive_expect_tx(&fullv[vb], nv * Sh::kTile);
        // V: per block and 8-key group, [D][8]
#pragma unroll
        for (int b = 0; b < Sh::kBlocks; ++b) {
          if (c * Sh::kBlocks + b >= nblk) continue;
#pragma unroll
          for (int g = 0; g < BS / 8; ++g)  // V rows tl*D .. tl*D+D-1, keys 8g .. 8g+7 of the block
            tma_2d_g2s(sv_ + ((b * BS) / 8 + g) * (D * 16), &tmap_v, g * 8, static_cast<int>(tl[b] * D),
                       &fullv[vb]);
        }
        issued_v = c + 1;
        load_table(c + 1);  // lands while this chunk is in flight
      }
      (void)ok;
    }
  } else {
    // ================= MMA issue: S of both tiles for chunk c, then their P V(c - 1) =================
    // The whole warp runs the loop and the waits (so the loop state and the descriptors
    // stay warp-uniform); one elected lane issues the MMAs and the commits.
    constexpr uint32_t kIdS = idesc<T>(kRows, kKeys), kIdO = idesc<T>(kRows, D);
    const int ntiles = two ? 2 : 1;
    const bool leader = elect_one();
    // descriptors of the first Q tile, K buffer and V buffer; a step moves the address
    // field (bits 0..13, 16-byte units), which stays below 2^14 for any shared address
    const uint64_t dq0 = sdesc(smem_addr(smem), 128, (D / 8) * 128);
    const uint64_t dk0 = sdesc(smem_addr(smem + Sh::kOffK), kKeys * 16, 128);
    const uint64_t dv0 = sdesc(smem_addr(smem + Sh::kOffV), D * 16, 128);
    auto wait_all = [&](uint64_t* bar, int parity) { return __all_sync(0xffffffffu, wait(bar, parity)); };
    uint64_t* last_bar = nullptr;  // the last barrier a commit was issued to, and its phase
    int last_par = 0;
    auto commit_to = [&](uint64_t* bar, int parity) {
      if (leader) commit(bar);
      __syncwarp();
      last_bar = bar;
      last_par = parity;
    };
    // the timeout-path test: the first wait runs out on `never` (no MMA issued yet);
    // the producer then drains its copies with the normal limit
    bool ok = __all_sync(0xffffffffu, !p.test_wait_ns || wait_or_abort(never, 0, s_abort, p.err, p.test_wait_ns));
    for (int c = 0; c <= nchunks && ok; ++c) {
      if (c < nchunks) {
        const int sb = c & 1, kb = c % kKStages;
        ok = wait_all(&fullk[kb], (c / kKStages) & 1);
        for (int Xm = 0; Xm < ntiles && ok; ++Xm) {
          if (c >= 2 && !(ok = wait_all(pvdone(Xm, sb), ((c - 2) >> 1) & 1))) break;  // P(c-2) read from S[sb]
          fence_after();
          if (leader) {
            const uint64_t da = dq0 + Xm * (Sh::kQTile >> 4), db = dk0 + kb * (Sh::kKBytes >> 4);
#pragma unroll
            for (int ks = 0; ks < D / 16; ++ks)
              mma(tmem + 256 * Xm + sb * kKeys, da + ks * 16, db + ks * (2 * kKeys), kIdS, ks > 0);
          }
          commit_to(sfull(Xm, sb), (c >> 1) & 1);
        }
        if (!ok) break;
        commit_to(&kfree[kb], (c / kKStages) & 1);
      }
      if (c >= 1) {
        const int c1 = c - 1, sb = c1 & 1;
        const int vb = c1 % kVStages;
        if (!(ok = wait_all(&fullv[vb], (c1 / kVStages) & 1))) break;
        for (int Xm = 0; Xm < ntiles && ok; ++Xm) {
          if (!(ok = wait_all(pfull(Xm, sb), (c1 >> 1) & 1))) break;
          fence_after();
          if (leader) {
            const uint64_t db = dv0 + vb * (Sh::kVBytes >> 4);
            const uint32_t tb = tmem + 256 * Xm;
#pragma unroll
            for (int part = 0; part < 2; ++part) {
#pragma unroll
              for (int kk = 0; kk < kKeys / 16; ++kk)
                mma_ts(tb + 2 * kKeys, tb + sb * kKeys + part * 32 + kk * 8, db + kk * (2 * D), kIdO,
                       c1 > 0 || part > 0 || kk > 0);
            }
          }
          commit_to(pvdone(Xm, sb), (c1 >> 1) & 1);
        }
        if (!ok) break;
        commit_to(&vfree[vb], (c1 / kVStages) & 1);
      }
    }
    // MMAs committed but maybe not finished: a commit tracks every earlier MMA of the
    // issuing thread, so the last commit's barrier covers them all
    if (!ok && last_bar != nullptr) mbar_wait_bounded(last_bar, last_par, kWaitNs / 8);
  }

  fence_before();
  __syncthreads();
  // After an abort (whoever raised it, before or after the producer's loop ended) no
  // consumer waits for the copies still landing: the producer waits (bounded) for the
  // last chunks it issued, so nothing lands after the CTA exits.
  if (*s_abort && warp == kProducerWarp && lane == 0) {
    for (int c = issued_k - kKStages; c < issued_k; ++c)
      if (c >= 0) mbar_wait_bounded(&fullk[c % kKStages], (c / kKStages) & 1, kWaitNs / 8);
    for (int c = issued_v - kVStages; c < issued_v; ++c)
      if (c >= 0) mbar_wait_bounded(&fullv[c % kVStages], (c / kVStages) & 1, kWaitNs / 8);
  }
  if (warp == 0) {
    fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(Sh::kTmemCols));
  }
}

}  // namespace ws
}  // namespace pa
