// prefill_ws.cuh -- chunked prefill on tcgen05 with warp specialisation.
//
// Causal attention of each sequence's chunk of new query tokens over its paged
// cache (what is computed: see prefill.cu), on sm_103a's tcgen05 MMAs with the
// accumulators in tensor memory (TMEM).  A CTA owns a
// tile of 128 query rows -- (token, query head) pairs of one kv head, head
// fastest -- which are TMEM lanes 0..127, and takes keys 64 at a time.  The
// phases of a chunk run in different warps that hand over through mbarriers, so
// the copies, the MMAs and the softmax of neighbouring chunks overlap:
//
//   * warp 4, one thread: the TMA copies of chunk c, through two tensor maps: K
//     into K buffer c % 2 once S of chunk c - 2 has read it, V into V buffer c % 3
//     once P V of chunk c - 3 has read it (V is needed last), each on its own
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
//   * warp 5, one thread: S(c) = Q K^T into TMEM columns S[c % 2] (once chunk c
//     has landed and P V(c - 2), which read P from those columns, is done), then
//     O += P V(c - 1) with P read from TMEM; each group is committed to mbarriers.
//   * warps 0..3, one thread per row: the softmax of S(c) while the tensor cores
//     run P V(c - 1) and S(c + 1).  P = exp2(s - m) goes back into the row's own S
//     columns as rounded 16-bit high and low parts (two per 32-bit column).  The
//     running maximum moves only when it grows by more than 2^8; then the row's O
//     is rescaled in TMEM after P V(c - 1) has finished (rare).  In the last chunk
//     the V of keys past the sequence (or past the blocks loaded) is zeroed in
//     shared memory first: P is 0 there, but 0 * NaN would poison O.
//
// At under 113 KiB of shared memory and 256 TMEM columns, two CTAs share an SM.
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
using tc::fence_after;
using tc::fence_before;
using tc::idesc;
using tc::ld32;
using tc::mma;
using tc::sdesc;
using tc::st32;

constexpr int kRows = 128;  // query rows per CTA (= TMEM lanes)
constexpr int kKeys = 64;   // keys per chunk
constexpr int kSoftmaxThreads = 128;
constexpr int kProducerWarp = 4, kMmaWarp = 5;
constexpr int kThreads = 6 * 32;
constexpr int kVStages = 3;
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

// The tile of rank `rank` (0-based) in the order of decreasing length -- the chunks of
// keys it reads -- ties by sequence, kv head and tile index; so the longest tiles of
// the whole launch start first and the short ones fill the tail.  Every thread of
// the CTA takes part (thread t owns sequences t * kPer ..); tile j of sequence s
// covers rows 128 j .. of its n * G rows and reads chunks 0 .. (ctx + (row_hi - 1) / G) / 64,
// which is non-decreasing in j, so the tiles of s reading >= x chunks are a suffix
// in j counted in closed form, and the rank-th tile is found by a binary search on x.
// Writes (sequence, kv head, tile) to out; returns false when rank is past the tiles.
__device__ bool pick_tile(const PrefillParams& p, int rank, int* red, int* out) {
  constexpr int kPer = (kMaxSeqsPerLaunch + kThreads - 1) / kThreads;
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
  // tiles of owned sequence i that read >= x chunks
  auto cnt = [&](int i, int x) -> int {
    const long long need = (long long)G * (64LL * (x - 1) - ctx[i]) + 1;  // rows the tile must reach
    if (nt[i] == 0 || need > rows[i]) return 0;
    if (need <= 1) return nt[i];
    return nt[i] - static_cast<int>((need + kRows - 1) / kRows - 1);
  };
  int buf = 0;
  auto reduce = [&](int v, bool take_max) -> int {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const int u = __shfl_xor_sync(0xffffffffu, v, o);
      v = take_max ? max(v, u) : v + u;
    }
    buf ^= 1;
    if (lane == 0) red[buf * 8 + warp] = v;
    __syncthreads();
    int t = take_max ? 0 : 0;
#pragma unroll
    for (int w = 0; w < kThreads / 32; ++w) t = take_max ? max(t, red[buf * 8 + w]) : t + red[buf * 8 + w];
    return t;
  };
  int local = 0, longest = 0;
#pragma unroll
  for (int i = 0; i < kPer; ++i) {
    local += nt[i];
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
  // rank among the tiles of exactly lo chunks, ordered by (sequence, kv head, tile)
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
  if (lane == 31) red[buf * 8 + warp] = incl;
  __syncthreads();
  long long before = incl - mine;
  for (int w = 0; w < warp; ++w) before += red[buf * 8 + w];
  before *= Hkv;
#pragma unroll
  for (int i = 0; i < kPer; ++i) {
    const long long span = (long long)Hkv * e[i];
    if (r >= before && r < before + span) {
      const int q = static_cast<int>(r - before);
      out[0] = tid * kPer + i;
      out[1] = q / e[i];
      out[2] = nt[i] - cnt(i, lo) + q % e[i];
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
  static constexpr int kQBytes = kRows * D * 2;            // Q, core-matrix layout
  static constexpr int kKBytes = kKeys * D * 2;  // a chunk's K as [D/8][64][8]
  static constexpr int kVBytes = kKeys * D * 2;  // a chunk's V as [key/8][D][8]
  static constexpr int kOffK = kQBytes;          // K ring: 2 buffers
  static constexpr int kOffV = kOffK + 2 * kKBytes;  // V ring: 3 buffers (V is read last)
  static constexpr int kOffBar = kOffV + kVStages * kVBytes;
  static constexpr int kNumBars = 2 + kVStages + 2 + 2 + 2 + kVStages + 1;  // the last: nothing completes it
  static constexpr int kOffRed = kOffBar + kNumBars * 8 + 32;  // [2][8] ints: block reductions
  static constexpr int kSmem = kOffRed + 2 * 8 * 4;            // <= 113 KiB: two CTAs per SM
  static constexpr int kTmemCols = 256;  // S/P[0]: 0..63, S/P[1]: 64..127, O: 128..128+D
};

template <typename T, int D, int BS>
__global__ void __launch_bounds__(kThreads, 2)
    prefill_ws_kernel(const PrefillParams p, const __grid_constant__ CUtensorMap tmap_k,
                      const __grid_constant__ CUtensorMap tmap_v) {
  using Sh = Shape<T, D, BS>;
  extern __shared__ __align__(1024) unsigned char smem[];
  unsigned char* sQ = smem;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + Sh::kOffBar);
  uint64_t* fullk = bars;                   // [2] K buffer landed (TMA bytes)
  uint64_t* fullv = fullk + 2;              // [kVStages] V buffer landed (TMA bytes)
  uint64_t* sfull = fullv + kVStages;       // [2] S in TMEM, the K buffer read (commit)
  uint64_t* pfull = sfull + 2;              // [2] P in TMEM, O rescaled and V tail zeroed where needed (128 arrivals)
  uint64_t* pvdone = pfull + 2;             // [2] P V done: P's columns and O are free (commit)
  uint64_t* vfree = pvdone + 2;             // [kVStages] P V done with the V buffer (commit)
  uint64_t* never = vfree + kVStages;       // nothing completes it: the timeout-path test waits on it
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(bars + Sh::kNumBars);
  int* s_tile = reinterpret_cast<int*>(s_tmem + 1);                     // sequence, kv head, tile (or -1)
  volatile int* s_abort = reinterpret_cast<volatile int*>(s_tile + 3);  // a thread gave up
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  griddep_launch_dependents();
  griddep_wait();

  // ---- which tile: the longest first over the whole launch
  const bool has_tile = pick_tile(p, static_cast<int>(blockIdx.x), reinterpret_cast<int*>(smem + Sh::kOffRed), s_tile);
  if (tid == 0) {
    if (!has_tile) s_tile[0] = -1;
    *s_abort = 0;
    for (int i = 0; i < 2; ++i) {
      mbar_init(&fullk[i], 1);
      mbar_init(&sfull[i], 1);
      mbar_init(&pfull[i], kSoftmaxThreads);
      mbar_init(&pvdone[i], 1);
    }
    for (int i = 0; i < kVStages; ++i) {
      mbar_init(&fullv[i], 1);
      mbar_init(&vfree[i], 1);
    }
    mbar_init(never, 1);
    fence_barrier_init();
  }
  __syncthreads();
  const int s = s_tile[0];
  if (s < 0) return;  // no tile for this CTA (before any TMEM is taken)
  const int kvh = s_tile[1], tile = s_tile[2];
  const int G = p.group;
  const int L = p.seq_lens[s], tok0 = p.query_start_loc[s], n = p.query_start_loc[s + 1] - tok0;
  const int rows = n * G, row_lo = tile * kRows, row_hi = min(rows, row_lo + kRows);
  const int ctx = L - n;
  const int p_max = ctx + (row_hi - 1) / G;  // last position any row of the tile has
  const int nblk = p_max / BS + 1;            // blocks holding keys 0..p_max
  const int nchunks = (p_max + kKeys) / kKeys;

  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_addr(s_tmem)),
                 "r"(Sh::kTmemCols));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  // the softmax threads' rows; Q into shared memory (core matrices: 8 rows x 16 bytes)
  const int r = tid & (kRows - 1), row = row_lo + r;
  const bool valid = row < row_hi;
  if (tid < kSoftmaxThreads) {
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
  const uint32_t t_o = tmem + 2 * kKeys;
  auto wait = [&](uint64_t* bar, int parity) { return wait_or_abort(bar, parity, s_abort, p.err); };
  int issued_k = 0, issued_v = 0;  // chunks whose K (V) copies the producer issued

  if (warp < 4) {
    // ================= softmax: row r, all keys of each chunk =================
    const int pos = valid ? ctx + row / G : p_max;  // a padding row behaves as the last real one
    const int kz = min(L, nblk * BS);               // first key whose V must read as zero
    const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
    const float sl2 = p.scale_log2;
    float m = -INFINITY, l = 0.f;
    bool ok = true;
    for (int c = 0; c < nchunks; ++c) {
      const int sb = c & 1;
      // tcgen05.ld / st are warp-collective (.sync.aligned): every branch around them
      // is taken by the whole warp, so each wait's outcome is agreed across the warp
      if (!__all_sync(0xffffffffu, wait(&sfull[sb], (c >> 1) & 1))) {
        ok = false;
        break;
      }
      fence_after();
      const uint32_t t_s = tmem + lane_base + sb * kKeys;
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
        if (!__all_sync(0xffffffffu, wait(&pvdone[(c - 1) & 1], ((c - 1) >> 1) & 1))) {
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
      // the last chunk: V of keys past the sequence (or past the blocks loaded) reads as zero
      if (c == nchunks - 1 && kz < (c + 1) * kKeys) {
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
      mbar_arrive(&pfull[sb]);
    }
    if (__all_sync(0xffffffffu, ok && wait(&pvdone[(nchunks - 1) & 1], ((nchunks - 1) >> 1) & 1))) {
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
  } else if (warp == kProducerWarp) {
    // ================= TMA copies of chunk c into stage c % 2 =================
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
        const int sb = c & 1;
        if (c >= 2 && !wait(&sfull[sb], ((c - 2) >> 1) & 1)) {  // S(c-2) is done with the stage's K
          ok = false;
          break;
        }
        unsigned char* sk = smem + Sh::kOffK + sb * Sh::kKBytes;
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
        mbar_arrive_expect_tx(&fullk[sb], Sh::kKBytes);
        // K: per 8-dim chunk dc, the rows (16 keys each) of the chunk's 64 keys
#pragma unroll
        for (int dc = 0; dc < D / 8; ++dc) {
          int rw[4];
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const int b = (16 * q) / BS, h = (16 * q) % BS / 16;
            rw[q] = static_cast<int>((tl[b] * (D / 8) + dc) * (BS / 16) + h);
          }
          tma_gather4_g2s(sk + dc * (kKeys * 16), &tmap_k, rw, &fullk[sb]);
        }
        issued_k = c + 1;
        if (c >= kVStages && !wait(&vfree[vb], ((c - kVStages) / kVStages) & 1)) {  // P V(c-3) read the buffer
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
    }
  } else {
    // ================= MMA issue: S(c), then O += P V(c - 1) =================
    if (lane == 0) {
      constexpr uint32_t kIdS = idesc<T>(kRows, kKeys), kIdO = idesc<T>(kRows, D);
      // the timeout-path test: the first wait runs out on `never` (no MMA issued yet);
      // the producer then drains its copies with the normal limit
      bool ok = !p.test_wait_ns || wait_or_abort(never, 0, s_abort, p.err, p.test_wait_ns);
      int last_s = -1, last_pv = -1;  // last groups committed
      for (int c = 0; c <= nchunks && ok; ++c) {
        if (c < nchunks) {
          const int sb = c & 1;
          ok = wait(&fullk[sb], (c >> 1) & 1);
          if (ok && c >= 2) ok = wait(&pvdone[sb], ((c - 2) >> 1) & 1);  // P(c-2) read from S[sb]
          if (!ok) break;
          fence_after();
          const unsigned char* st = smem + Sh::kOffK + sb * Sh::kKBytes;
#pragma unroll
          for (int ks = 0; ks < D / 16; ++ks) {
            const uint64_t da = sdesc(smem_addr(sQ) + ks * 256, 128, (D / 8) * 128);
            const uint64_t db = sdesc(smem_addr(st) + ks * 2 * (kKeys * 16), kKeys * 16, 128);
            mma(tmem + sb * kKeys, da, db, kIdS, ks > 0);
          }
          commit(&sfull[sb]);
          last_s = c;
        }
        if (c >= 1) {
          const int c1 = c - 1, sb = c1 & 1;
          const int vb = c1 % kVStages;
          if (!(ok = wait(&pfull[sb], (c1 >> 1) & 1) && wait(&fullv[vb], (c1 / kVStages) & 1))) break;
          fence_after();
          const uint32_t sV = smem_addr(smem + Sh::kOffV + vb * Sh::kVBytes);
#pragma unroll
          for (int part = 0; part < 2; ++part) {
#pragma unroll
            for (int kk = 0; kk < kKeys / 16; ++kk) {
              const uint64_t db = sdesc(sV + kk * 2 * (D * 16), D * 16, 128);
              mma_ts(t_o, tmem + sb * kKeys + part * 32 + kk * 8, db, kIdO, c1 > 0 || part > 0 || kk > 0);
            }
          }
          commit(&pvdone[sb]);
          commit(&vfree[vb]);
          last_pv = c1;
        }
      }
      if (!ok) {  // MMAs committed but maybe not finished: wait (bounded) for the last of each kind
        if (last_s >= 0) mbar_wait_bounded(&sfull[last_s & 1], (last_s >> 1) & 1, kWaitNs / 8);
        if (last_pv >= 0) mbar_wait_bounded(&pvdone[last_pv & 1], (last_pv >> 1) & 1, kWaitNs / 8);
      }
    }
  }

  fence_before();
  __syncthreads();
  // After an abort (whoever raised it, before or after the producer's loop ended) no
  // consumer waits for the copies still landing: the producer waits (bounded) for the
  // last chunks it issued, so nothing lands after the CTA exits.
  if (*s_abort && warp == kProducerWarp && lane == 0) {
    for (int c = issued_k - 2; c < issued_k; ++c)
      if (c >= 0) mbar_wait_bounded(&fullk[c & 1], (c >> 1) & 1, kWaitNs / 8);
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
