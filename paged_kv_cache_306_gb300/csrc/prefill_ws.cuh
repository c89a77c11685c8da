// prefill_ws.cuh -- chunked prefill on tcgen05 with warp specialisation.
//
// Causal attention of each sequence's chunk of new query tokens over its paged
// cache (what is computed: see prefill.cu), on sm_103a's tcgen05 MMAs with the
// accumulators in tensor memory (TMEM).  A query tile is 128 rows -- (token,
// query head) pairs of one kv head, head fastest -- which are TMEM lanes
// 0..127; keys are taken 128 at a time (a chunk).  A CTA owns a PAIR of
// consecutive tiles A and B of one (sequence, kv head): both read the same keys,
// so each chunk of K and V is copied once and feeds the MMAs of both tiles.  The
// two tiles take turns: while the softmax of one runs, the tensor cores run the
// other's P V and its next S (ping-pong).  The phases run in different warps that
// hand over through mbarriers:
//
//   * warp 8: the TMA copies of chunk c, K into K buffer c % 2 once both tiles' S
//     of chunk c - 2 have read it, V into V buffer c % 2 once both tiles' P V of
//     chunk c - 2 have read it, each on its own mbarrier.  K: the pool seen as rows
//     of 16 keys x 8 dims (one 256-byte run of a K tile [D/8][bs][8]); lane i issues
//     the i-th tile::gather4 load (one per 8-dim slice and 64 keys), which fetches
//     four such rows from blocks anywhere in the pool and lands them as [64][8]: the
//     K operand of S = Q K^T is [D/8][128 keys][8], core matrices with one uniform
//     stride, so S is one MMA of N = 128 per 16 dims.  V: lane b issues one box per
//     block, the (block, kv head) tile [D][bs] with the 32-byte (bs 16) or 64-byte
//     (bs 32) swizzle, which is the K-major operand layout of P V with the same
//     swizzle: no re-layout pass.  (V was first copied as [D x 8-key] boxes of
//     16-byte rows, 16 per chunk, whose copies held the K gathers back, and then
//     with cp.async from two warps of its own.)
//   * warp 9: the MMAs, in the order P V_A(c), S_A(c + 1), P V_B(c), S_B(c + 1): a
//     tile's S(c + 1) overwrites the P(c) its P V(c) reads and is issued right behind
//     it (the MMAs of one thread run in issue order).  The whole warp runs the loop
//     and the waits; one elected lane issues the MMAs and commits them to mbarriers.
//   * warps 0..3 (tile A) and 4..7 (tile B), one thread per row: the softmax of
//     S(c).  P = exp2(s - m) goes back into the row's own S columns as 16-bit
//     values, two per 32-bit column: the 16 columns of keys 16 k .. 16 k + 15
//     become 8 columns of P rounded to fp16 or, for bf16, 8 columns of rounded high
//     parts and 8 of low parts (~16 significant bits; P V is then two MMA groups).
//     The running maximum moves only when it grows by more than 2^8; then the row's O is rescaled in TMEM (P V(c - 1) is done by
//     then: S(c) was issued after it).  In the last chunk tile A's threads zero the
//     V of keys past the sequence (or past the blocks loaded) in shared memory
//     first: P is 0 there, but 0 * NaN would poison O.  A tile whose rows end
//     before the pair's last chunk sees scores of -inf there (P = 0).
//
// TMEM: tile X at column 256 X: S/P in 0..127, O (D <= 128 columns) from 128; all
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
constexpr int kKeys = 128;  // keys per chunk
constexpr int kSoftmaxThreads = 128;  // per tile
constexpr int kCopyWarp = 8, kMmaWarp = 9;
// A cluster of two CTAs on two SMs takes a unit of four consecutive tiles of one
// (sequence, kv head), a pair per CTA; each CTA copies half of every chunk of K and V
// with TMA multicast into both, so each SM fetches half of the bytes its MMAs read.
constexpr int kCluster = 2, kUnitTiles = 2 * kCluster;
constexpr uint16_t kClusterMask = (1u << kCluster) - 1;
constexpr int kThreads = 10 * 32;
constexpr int kKStages = 2, kVStages = 2;
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

// 128 consecutive fp32 columns of this thread's TMEM lane: four loads, one wait (in one
// statement, so no use of the registers can be scheduled before the wait)
__device__ __forceinline__ void ld128(uint32_t taddr, float (&v)[128]) {
  uint32_t r[128];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%128];\n\t"
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%32,%33,%34,%35,%36,%37,%38,%39,%40,%41,%42,%43,%44,%45,%46,%47,"
      "%48,%49,%50,%51,%52,%53,%54,%55,%56,%57,%58,%59,%60,%61,%62,%63}, [%129];\n\t"
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%64,%65,%66,%67,%68,%69,%70,%71,%72,%73,%74,%75,%76,%77,%78,%79,"
      "%80,%81,%82,%83,%84,%85,%86,%87,%88,%89,%90,%91,%92,%93,%94,%95}, [%130];\n\t"
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%96,%97,%98,%99,%100,%101,%102,%103,%104,%105,%106,%107,%108,%109,%110,%111,"
      "%112,%113,%114,%115,%116,%117,%118,%119,%120,%121,%122,%123,%124,%125,%126,%127}, [%131];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
        "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
        "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31]),
        "=r"(r[32]), "=r"(r[33]), "=r"(r[34]), "=r"(r[35]), "=r"(r[36]), "=r"(r[37]), "=r"(r[38]), "=r"(r[39]),
        "=r"(r[40]), "=r"(r[41]), "=r"(r[42]), "=r"(r[43]), "=r"(r[44]), "=r"(r[45]), "=r"(r[46]), "=r"(r[47]),
        "=r"(r[48]), "=r"(r[49]), "=r"(r[50]), "=r"(r[51]), "=r"(r[52]), "=r"(r[53]), "=r"(r[54]), "=r"(r[55]),
        "=r"(r[56]), "=r"(r[57]), "=r"(r[58]), "=r"(r[59]), "=r"(r[60]), "=r"(r[61]), "=r"(r[62]), "=r"(r[63]),
        "=r"(r[64]), "=r"(r[65]), "=r"(r[66]), "=r"(r[67]), "=r"(r[68]), "=r"(r[69]), "=r"(r[70]), "=r"(r[71]),
        "=r"(r[72]), "=r"(r[73]), "=r"(r[74]), "=r"(r[75]), "=r"(r[76]), "=r"(r[77]), "=r"(r[78]), "=r"(r[79]),
        "=r"(r[80]), "=r"(r[81]), "=r"(r[82]), "=r"(r[83]), "=r"(r[84]), "=r"(r[85]), "=r"(r[86]), "=r"(r[87]),
        "=r"(r[88]), "=r"(r[89]), "=r"(r[90]), "=r"(r[91]), "=r"(r[92]), "=r"(r[93]), "=r"(r[94]), "=r"(r[95]),
        "=r"(r[96]), "=r"(r[97]), "=r"(r[98]), "=r"(r[99]), "=r"(r[100]), "=r"(r[101]), "=r"(r[102]), "=r"(r[103]),
        "=r"(r[104]), "=r"(r[105]), "=r"(r[106]), "=r"(r[107]), "=r"(r[108]), "=r"(r[109]), "=r"(r[110]), "=r"(r[111]),
        "=r"(r[112]), "=r"(r[113]), "=r"(r[114]), "=r"(r[115]), "=r"(r[116]), "=r"(r[117]), "=r"(r[118]), "=r"(r[119]),
        "=r"(r[120]), "=r"(r[121]), "=r"(r[122]), "=r"(r[123]), "=r"(r[124]), "=r"(r[125]), "=r"(r[126]), "=r"(r[127])
      : "r"(taddr), "r"(taddr + 32), "r"(taddr + 64), "r"(taddr + 96)
      : "memory");
#pragma unroll
  for (int i = 0; i < 128; ++i) v[i] = __uint_as_float(r[i]);
}

// 16 consecutive 32-bit columns of this thread's TMEM lane; no wait (wait_st before
// the columns are handed over)
__device__ __forceinline__ void st16(uint32_t taddr, const uint32_t (&v)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(
          taddr),
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]), "r"(v[9]),
      "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15])
      : "memory");
}
__device__ __forceinline__ void st8(uint32_t taddr, const uint32_t (&v)[8]) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"r"(taddr), "r"(v[0]),
               "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7])
               : "memory");
}
__device__ __forceinline__ void wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// 2^x by the hardware's approximate exponential (|relative error| below 2^-22; 2^-inf = 0)
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Shared-memory matrix descriptor (tcgen05), K-major with the 32-byte (mode 6) or
// 64-byte (mode 4) swizzle: rows of 32 or 64 bytes, sbo = the distance between groups
// of 8 rows; the leading offset is unused when one MMA's K extent fits a row.
__device__ __forceinline__ uint64_t sdesc_swizzled(uint32_t addr, uint32_t sbo, uint32_t mode) {
  return (uint64_t)((addr >> 4) & 0x3FFF) | ((uint64_t)1 << 16) | ((uint64_t)((sbo >> 4) & 0x3FFF) << 32) |
         ((uint64_t)1 << 46) | ((uint64_t)mode << 61);
}

// tile::gather4 tensor-map copy: four rows (element row indices rows[0..3]) of a 2-D
// map whose box is one row high, landing one after another at the same offset of
// shared memory in every CTA of the cluster in `mask`, each signalling its own
// mbarrier at `bar`'s offset
__device__ __forceinline__ void tma_gather4_mc(void* dst, const CUtensorMap* map, const int (&rows)[4], uint64_t* bar,
                                               uint16_t mask) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile::gather4.mbarrier::complete_tx::bytes.multicast::cluster "
      "[%0], [%1, {%2, %3, %4, %5, %6}], [%7], %8;" ::"r"(smem_addr(dst)),
      "l"(map), "r"(0), "r"(rows[0]), "r"(rows[1]), "r"(rows[2]), "r"(rows[3]), "r"(smem_addr(bar)), "h"(mask)
      : "memory");
}

// 2-D tensor-map copy (box at element coordinates x, y) into every CTA of `mask`, as above
__device__ __forceinline__ void tma_2d_mc(void* dst, const CUtensorMap* map, int x, int y, uint64_t* bar,
                                          uint16_t mask) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.multicast::cluster [%0], "
      "[%1, {%2, %3}], [%4], %5;" ::"r"(smem_addr(dst)),
      "l"(map), "r"(x), "r"(y), "r"(smem_addr(bar)), "h"(mask)
      : "memory");
}

// One arrival on the mbarrier at `bar`'s offset in every CTA of `mask` once every
// earlier MMA of this thread has completed
__device__ __forceinline__ void commit_mc(uint64_t* bar, uint16_t mask) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(
          smem_addr(bar)),
      "h"(mask)
      : "memory");
}

__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

// Every thread of both CTAs of the cluster: the mbarrier inits (and any shared-memory
// writes before it) are visible cluster-wide afterwards
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
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

// The unit of rank `rank` (0-based) in the order of decreasing length -- the chunks
// of keys it reads -- ties by sequence, kv head and unit index; so the longest
// units of the whole launch start first and the short ones fill the tail.  A unit
// is kUnitTiles consecutive tiles of one (sequence, kv head), the work of one
// cluster.  Every thread of the CTA takes part (thread t owns sequences
// t * kPer ..).  Tile j of sequence s covers rows 128 j .. of its n * G rows and
// reads chunks 0 .. (ctx + (row_hi - 1) / G) / 128, non-decreasing in j; unit k holds
// tiles kUnitTiles k .. (those that exist) and reads what its last tile reads.  So
// the tiles of s reading >= x chunks are a suffix j >= j0 in closed form, the units
// reading >= x are those from j0 / kUnitTiles on, and the rank-th unit is found by
// a binary search on x.  Writes (sequence, kv head, unit) to out; returns false
// when rank is past the units.
__device__ bool pick_unit(const PrefillParams& p, int rank, int* red, int* out) {
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
  // units of owned sequence i that read >= x chunks
  auto cnt = [&](int i, int x) -> int {
    const long long need = (long long)G * ((long long)kKeys * (x - 1) - ctx[i]) + 1;  // rows a tile must reach
    if (nt[i] == 0 || need > rows[i]) return 0;
    const int j0 = need <= 1 ? 0 : static_cast<int>((need + kRows - 1) / kRows - 1);  // first tile reading >= x
    return (nt[i] + kUnitTiles - 1) / kUnitTiles - j0 / kUnitTiles;
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
    local += (nt[i] + kUnitTiles - 1) / kUnitTiles;
    if (nt[i]) longest = max(longest, (ctx[i] + (rows[i] - 1) / G) / kKeys + 1);
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
  // rank among the units of exactly lo chunks, ordered by (sequence, kv head, unit)
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
      out[2] = (nt[i] + kUnitTiles - 1) / kUnitTiles - cnt(i, lo) + q % e[i];
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
  static constexpr int kKBytes = kKeys * D * 2;  // a chunk's K as [D/8][128][8]
  static constexpr int kVBytes = kKeys * D * 2;  // a chunk's V: kBlocks swizzled tiles [D][bs]
  static constexpr int kOffK = 2 * kQTile;                  // K ring
  static constexpr int kOffV = kOffK + kKStages * kKBytes;  // V ring
  static constexpr int kOffBar = kOffV + kVStages * kVBytes;
  // fullk[K], fullv[V], kfree[K], vfree[V], per tile sfull, pfull, pvdone, never
  static constexpr int kNumBars = 2 * kKStages + 2 * kVStages + 2 * 3 + 1;
  static constexpr int kOffRed = kOffBar + kNumBars * 8 + 32;  // [2][16] ints: block reductions
  // more than half an SM's shared memory, so one CTA per SM: it takes all of TMEM
  static constexpr int kSmem = kOffRed + 2 * 16 * 4 > 116 * 1024 ? kOffRed + 2 * 16 * 4 : 116 * 1024;
  static constexpr int kTmemCols = 512;  // tile X at 256 X: S/P 0..127, O 128..128+D
};

template <typename T, int D, int BS>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_ws_kernel(const PrefillParams p, const __grid_constant__ CUtensorMap tmap_k,
                      const __grid_constant__ CUtensorMap tmap_v) {
  using Sh = Shape<T, D, BS>;
  static_assert(Sh::kSmem > 114 * 1024, "two CTAs on one SM would contend for TMEM");
  static_assert(kKeys % BS == 0, "a chunk is whole blocks");
  // P in one 16-bit part for fp16 (11 significant bits, the operands' own precision); for
  // bf16 a high and a low part (~16 bits), since one bf16 part (8 bits) would add
  // errors as large as the output's own rounding
  constexpr int kParts = std::is_same<T, __half>::value ? 1 : 2;
  extern __shared__ __align__(1024) unsigned char smem[];
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + Sh::kOffBar);
  uint64_t* fullk = bars;                   // [kKStages] K buffer landed (TMA bytes)
  uint64_t* fullv = fullk + kKStages;       // [kVStages] V buffer landed (TMA bytes)
  uint64_t* kfree = fullv + kVStages;       // [kKStages] both CTAs' S read the K buffer (a commit from each)
  uint64_t* vfree = kfree + kKStages;       // [kVStages] both CTAs' P V read the V buffer (a commit from each)
  uint64_t* tbars = vfree + kVStages;       // per tile X at 3 X: sfull, pfull, pvdone
  uint64_t* never = tbars + 6;              // nothing completes it: the timeout-path test waits on it
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(bars + Sh::kNumBars);
  int* s_pair = reinterpret_cast<int*>(s_tmem + 1);                     // sequence, kv head, unit (or -1)
  volatile int* s_abort = reinterpret_cast<volatile int*>(s_pair + 3);  // a thread gave up
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  // S(c) in TMEM (commit); P(c) in TMEM, O rescaled, V tail zeroed (128 arrivals);
  // P V(c) done: P's columns free, O final after the last chunk (commit)
  auto sfull = [&](int X) { return tbars + 3 * X; };
  auto pfull = [&](int X) { return tbars + 3 * X + 1; };
  auto pvdone = [&](int X) { return tbars + 3 * X + 2; };

  griddep_launch_dependents();
  griddep_wait();

  // ---- which unit: the longest first over the whole launch (both CTAs of a cluster pick the same)
  const uint32_t crank = cluster_rank();
  const bool has_unit =
      pick_unit(p, static_cast<int>(blockIdx.x / kCluster), reinterpret_cast<int*>(smem + Sh::kOffRed), s_pair);
  if (tid == 0) {
    if (!has_unit) s_pair[0] = -1;
    *s_abort = 0;
    for (int i = 0; i < kKStages; ++i) {
      mbar_init(&fullk[i], 1);
      mbar_init(&kfree[i], kCluster);
    }
    for (int i = 0; i < kVStages; ++i) {
      mbar_init(&fullv[i], 1);
      mbar_init(&vfree[i], kCluster);
    }
    for (int X = 0; X < 2; ++X) {
      mbar_init(sfull(X), 1);
      mbar_init(pfull(X), kSoftmaxThreads);
      mbar_init(pvdone(X), 1);
    }
    mbar_init(never, 1);
    fence_barrier_init();
  }
  __syncthreads();
  cluster_sync_all();  // both CTAs' mbarriers are initialised before either copies into the other
  const int s = s_pair[0];
  if (s < 0) return;  // no unit for this cluster: both CTAs leave here, before any TMEM is taken
  const int kvh = s_pair[1], unit = s_pair[2];
  const int G = p.group;
  const int L = p.seq_lens[s], tok0 = p.query_start_loc[s], n = p.query_start_loc[s + 1] - tok0;
  // this CTA's pair: tiles kUnitTiles unit + 2 crank and the next (either may be past the rows)
  const int rows = n * G, pair_lo = (kUnitTiles * unit + 2 * static_cast<int>(crank)) * kRows,
            pair_hi = min(rows, pair_lo + 2 * kRows);
  const int ntiles = pair_lo >= rows ? 0 : (pair_lo + kRows < rows ? 2 : 1);  // tiles with rows: A, then B
  // keys: what the unit's last row sees, the same in both CTAs (they share every chunk)
  const int unit_hi = min(rows, (kUnitTiles * unit + kUnitTiles) * kRows);
  const int ctx = L - n;
  const int p_max = ctx + (unit_hi - 1) / G;  // last position any row of the unit has
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
  if (tid < 2 * kSoftmaxThreads) {  // all 16-byte pieces of the row in flight at once, zeros for a padding row
    const uint32_t sq = smem_addr(smem + X * Sh::kQTile + (r / 8) * (D / 8) * 128 + (r % 8) * 16);
    const T* q = static_cast<const T*>(p.q) +
                 ((long long)(tok0 + (valid ? row / G : 0)) * p.num_heads + (long long)kvh * G + (valid ? row % G : 0)) * D;
    const uint32_t nbytes = valid ? 16u : 0u;
#pragma unroll
    for (int c = 0; c < D / 8; ++c)
      asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(sq + c * 128), "l"(q + 8 * c), "r"(nbytes)
                   : "memory");
    asm volatile("cp.async.wait_all;" ::: "memory");
  }
  fence_proxy_async_smem();  // Q's generic stores before the MMAs read it
  fence_before();
  __syncthreads();
  fence_after();
  const uint32_t tmem = *s_tmem;
  int issued_k = 0, issued_v = 0;  // chunks whose K (V) copies warp 8 issued
  auto wait = [&](uint64_t* bar, int parity) { return wait_or_abort(bar, parity, s_abort, p.err); };

  if (warp < 8) {
    // ================= softmax: tile X, row r, all keys of each chunk =================
    if (ntiles > X) {
      const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
      const uint32_t t_s = tmem + 256 * X + lane_base;
      const uint32_t t_o = t_s + kKeys;
      const int pos = valid ? ctx + row / G : ctx + (pair_hi - 1) / G;  // a padding row behaves as a real one
      const int kz = min(L, nblk * BS);  // first key whose V must read as zero
      const float sl2 = p.scale_log2;
      float m = -INFINITY, l = 0.f;
      bool ok = true;
      for (int c = 0; c < nchunks; ++c) {
        // tcgen05.ld / st are warp-collective (.sync.aligned): every branch around them
        // is taken by the whole warp, so each wait's outcome is agreed across the warp
        if (!__all_sync(0xffffffffu, wait(sfull(X), c & 1))) {
          ok = false;
          break;
        }
        fence_after();
        float sv[kKeys];
        ld128(t_s, sv);
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
        // P over the row's S columns, 16 keys at a time: the 16 columns of keys 16 k ..
        // 16 k + 15 become 8 columns of high parts (then, for bf16, 8 of low parts)
        {
          float ps[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
          for (int k = 0; k < kKeys / 16; ++k) {
            uint32_t blk[8 * kParts];
#pragma unroll
            for (int j = 0; j < 8; ++j) {  // P = 2^(scale * s - m), s = -inf gives 0
              const float x0 = ex2(fmaf(sv[16 * k + 2 * j], sl2, -m)), x1 = ex2(fmaf(sv[16 * k + 2 * j + 1], sl2, -m));
              ps[j & 3] += x0 + x1;
              blk[j] = pack2<T>(x0, x1);
              if constexpr (kParts == 2) {
                const float2 back = unpack2<T>(blk[j]);
                blk[8 + j] = pack2<T>(x0 - back.x, x1 - back.y);
              }
            }
            if constexpr (kParts == 2) st16(t_s + 16 * k, blk);
            else st8(t_s + 16 * k, blk);
          }
          wait_st();
          l += (ps[0] + ps[1]) + (ps[2] + ps[3]);
        }
        // O holds P V up to chunk c - 1, finished (S(c) was issued after it): rescale the
        // row if the maximum moved (the whole warp takes the branch when one of its rows
        // needs it; the others scale by 1)
        const bool rescale = c > 0 && move && corr != 1.f;
        if (__any_sync(0xffffffffu, rescale)) {
          const float f = rescale ? corr : 1.f;
#pragma unroll
          for (int c0 = 0; c0 < D; c0 += 32) {
            float o[32];
            ld32(t_o + c0, o);
#pragma unroll
            for (int j = 0; j < 32; ++j) o[j] *= f;
            st32(t_o + c0, o);
          }
        }
        // the last chunk: V of keys past the sequence (or past the blocks loaded) reads as
        // zero; tile A's threads clear it before either tile's P V of the chunk is issued
        if (X == 0 && c == nchunks - 1 && kz < (c + 1) * kKeys) {
          if (!__all_sync(0xffffffffu, wait(&fullv[c % kVStages], (c / kVStages) & 1))) {
            ok = false;
            break;
          }
          // block b's tile [D][bs]: dim d's keys 8 g .. 8 g + 7 are the 16 bytes at d * 2 bs + 16 g
          // within the row, moved by the swizzle (16-byte unit bits xor'ed with bits 7 and up)
          unsigned char* vbase = smem + Sh::kOffV + (c % kVStages) * Sh::kVBytes;
          constexpr int kRow = 2 * BS, kUnits = kRow / 16;
          const int k0 = kz - c * kKeys;  // first key to clear (0 <= k0 < kKeys)
          const int g0 = k0 / 8;          // the 8-key group holding it
          for (int i = tid; i < (kKeys / 8 - g0) * D; i += kSoftmaxThreads) {
            const int g = g0 + i / D, d = i % D;  // keys 8 g .. 8 g + 7 of dim d
            const int a = d * kRow + ((8 * g) % BS) * 2;
            unsigned char* u = vbase + ((8 * g) / BS) * Sh::kTile + (a ^ (((a >> 7) & (kUnits - 1)) << 4));
            if (8 * g >= k0) {
              *reinterpret_cast<uint4*>(u) = make_uint4(0, 0, 0, 0);
            } else {
              for (int k = k0 - 8 * g; k < 8; ++k) *reinterpret_cast<T*>(u + 2 * k) = DType<T>::from_f32(0.f);
            }
          }
          fence_proxy_async_smem();
        }
        fence_before();
        mbar_arrive(pfull(X));
      }
      if (__all_sync(0xffffffffu, ok && wait(pvdone(X), 0))) {  // one phase: the last P V
        fence_after();
        const float inv = 1.f / l;
        T* out = static_cast<T*>(p.out) +
                 ((long long)(tok0 + (valid ? row / G : 0)) * p.num_heads + (long long)kvh * G + (valid ? row % G : 0)) *
                     D;
#pragma unroll
        for (int c0 = 0; c0 < D; c0 += 32) {
          float o[32];
          ld32(t_o + c0, o);
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
  } else if (warp == kCopyWarp) {
    // ================= copies of chunk c (warp 8): K gathers, then V boxes =================
    // This CTA issues its half of the chunk's copies, each into both CTAs of the
    // cluster: lane i the gather4 load crank * kGathers / 2 + i of K (8-dim slice dc,
    // keys 64 h .. 64 h + 63), lane b the V box of the chunk's block b when b % 2 is
    // its rank.  Each CTA's full barriers expect the whole chunk.
    constexpr int kGathers = (D / 8) * (kKeys / 64), kMine = kGathers / kCluster;
    static_assert(kGathers <= 32 && Sh::kBlocks <= 32 && kGathers % kCluster == 0, "one copy per lane");
    const int32_t* bt = p.block_tables + (long long)s * p.max_blocks_per_seq;
    auto phys_of = [&](int c) {  // lane b: the physical block of the chunk's block b (-1 past the keys)
      const int gb = c * Sh::kBlocks + lane;
      return lane < Sh::kBlocks && gb < nblk ? __ldg(bt + gb) : -1;
    };
    const int gi = static_cast<int>(crank) * kMine + lane;  // this lane's gather (lanes < kMine)
    const int dc = gi / (kKeys / 64), h = gi % (kKeys / 64);
    int ph = phys_of(0);  // the next chunk's table entries land while a chunk is in flight
    bool ok = true;
    for (int c = 0; c < nchunks && ok; ++c) {
      const int kb = c % kKStages, vb = c % kVStages;
      const bool live = lane < Sh::kBlocks && c * Sh::kBlocks + lane < nblk;
      const bool bad = ph < 0 || ph >= p.num_blocks;
      if (live && bad) set_error(p.err, kErrBlockId);
      const int ph0 = __shfl_sync(0xffffffffu, bad ? 0 : ph, 0);  // block 0 of a chunk always holds keys
      // a block past the keys: any rows do (S there is masked; its V is not copied)
      const long long tl = (long long)(live ? (bad ? 0 : ph) : ph0) * p.num_kv_heads + kvh;
      const int nlive = __popc(__ballot_sync(0xffffffffu, live));
      int rw[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) {  // the rows (16 keys each) of this lane's 64 keys
        const int key = 64 * h + 16 * q;
        const long long tb = __shfl_sync(0xffffffffu, tl, key / BS);
        rw[q] = static_cast<int>((tb * (D / 8) + dc) * (BS / 16) + (key % BS) / 16);
      }
      if (c >= kKStages &&  // both CTAs' S read the buffer (in both CTAs)
          !(ok = __all_sync(0xffffffffu, wait(&kfree[kb], ((c - kKStages) / kKStages) & 1))))
        break;
      if (lane == 0) mbar_arrive_expect_tx(&fullk[kb], Sh::kKBytes);
      __syncwarp();
      if (lane < kMine)  // lands as [64 keys][8 dims] in the slice's rows, in both CTAs
        tma_gather4_mc(smem + Sh::kOffK + kb * Sh::kKBytes + dc * (kKeys * 16) + h * (64 * 16), &tmap_k, rw,
                       &fullk[kb], kClusterMask);
      issued_k = c + 1;
      if (c >= kVStages &&  // both CTAs' P V read the buffer (in both CTAs)
          !(ok = __all_sync(0xffffffffu, wait(&vfree[vb], ((c - kVStages) / kVStages) & 1))))
        break;
      if (lane == 0) mbar_arrive_expect_tx(&fullv[vb], nlive * Sh::kTile);
      __syncwarp();
      if (live && lane % kCluster == static_cast<int>(crank))  // the (block, kv head) tile [D][bs], swizzled;
        tma_2d_mc(smem + Sh::kOffV + vb * Sh::kVBytes + lane * Sh::kTile, &tmap_v, 0,  // V past the keys is zeroed
                  static_cast<int>(tl * D), &fullv[vb], kClusterMask);                // by the softmax threads
      issued_v = c + 1;
      ph = phys_of(c + 1);
    }
  } else {
    // ================= MMAs (warp 9): P V_A(c), S_A(c + 1), P V_B(c), S_B(c + 1) =================
    // The whole warp runs the loop and the waits (so the loop state and the descriptors
    // stay warp-uniform); one elected lane issues the MMAs and the commits.
    // A CTA without rows (the unit's second pair missing) still frees each buffer
    // for its partner: it commits to the free barriers of both CTAs with no MMA before.
    constexpr uint32_t kIdS = idesc<T>(kRows, kKeys), kIdO = idesc<T>(kRows, D);
    const bool leader = elect_one();
    // descriptors of the first Q tile, K buffer and V buffer; a step moves the address
    // field (bits 0..13, 16-byte units), which stays below 2^14 for any shared address
    const uint64_t dq0 = sdesc(smem_addr(smem), 128, (D / 8) * 128);
    const uint64_t dk0 = sdesc(smem_addr(smem + Sh::kOffK), kKeys * 16, 128);
    // V: one [D][bs] tile per block, rows of 2 bs bytes with the matching swizzle; the keys
    // 16 kk .. 16 kk + 15 are block 16 kk / bs, at byte 2 (16 kk % bs) of its rows
    const uint64_t dv0 = sdesc_swizzled(smem_addr(smem + Sh::kOffV), 8 * BS * 2, BS == 16 ? 6u : 4u);
    auto wait_all = [&](uint64_t* bar, int parity) { return __all_sync(0xffffffffu, wait(bar, parity)); };
    uint64_t* last_bar = nullptr;  // the last barrier a commit was issued to, and its phase
    int last_par = 0;
    auto commit_to = [&](uint64_t* bar, int parity, bool both = false) {  // both: the free barriers of both CTAs
      if (leader) {
        if (both) commit_mc(bar, kClusterMask);
        else commit(bar);
      }
      __syncwarp();
      last_bar = bar;
      last_par = parity;
    };
    auto issue_s = [&](int Xm, int c) {  // S_X(c) = Q_X K(c)^T into X's S columns
      if (leader) {
        const uint64_t da = dq0 + Xm * (Sh::kQTile >> 4), db = dk0 + (c % kKStages) * (Sh::kKBytes >> 4);
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks)
          mma(tmem + 256 * Xm, da + ks * 16, db + ks * (2 * kKeys), kIdS, ks > 0);
      }
      commit_to(sfull(Xm), c & 1);
    };
    auto issue_pv = [&](int Xm, int c) {  // O_X += P_X(c) V(c): high parts, then low parts
      if (leader) {
        const uint64_t db = dv0 + (c % kVStages) * (Sh::kVBytes >> 4);
        const uint32_t tb = tmem + 256 * Xm;
#pragma unroll
        for (int part = 0; part < kParts; ++part) {
#pragma unroll
          for (int kk = 0; kk < kKeys / 16; ++kk)  // keys 16 kk ..: high parts in 8 columns, low in the next 8
            mma_ts(tb + kKeys, tb + 16 * kk + 8 * part,
                   db + (((16 * kk) / BS) * Sh::kTile + ((16 * kk) % BS) * 2) / 16, kIdO, c > 0 || part > 0 || kk > 0);
        }
      }
      if (c == nchunks - 1) commit_to(pvdone(Xm), 0);  // O_X is complete
    };
    // the timeout-path test: the first wait runs out on `never` (no MMA issued yet);
    // the producer then drains its copies with the normal limit
    bool ok = __all_sync(0xffffffffu, !p.test_wait_ns || wait_or_abort(never, 0, s_abort, p.err, p.test_wait_ns));
    if (ok && (ok = wait_all(&fullk[0], 0))) {
      fence_after();
      for (int Xm = 0; Xm < ntiles; ++Xm) issue_s(Xm, 0);
      commit_to(&kfree[0], 0, true);
    }
    for (int c = 0; c < nchunks && ok; ++c) {
      const int vb = c % kVStages, c1 = c + 1;
      if (!(ok = wait_all(&fullv[vb], (c / kVStages) & 1))) break;
      for (int Xm = 0; Xm < ntiles && ok; ++Xm) {
        if (!(ok = wait_all(pfull(Xm), c & 1))) break;  // the softmax wrote P_X(c)
        fence_after();
        issue_pv(Xm, c);
        if (Xm == ntiles - 1) commit_to(&vfree[vb], (c / kVStages) & 1, true);
        if (c1 < nchunks) {
          if (Xm == 0 && !(ok = wait_all(&fullk[c1 % kKStages], (c1 / kKStages) & 1))) break;
          // S_X(c + 1) overwrites the columns P V_X(c) reads, issued right behind it: MMAs
          // of one thread run in issue order, so no wait is needed between the two
          fence_after();
          issue_s(Xm, c1);
          if (Xm == ntiles - 1) commit_to(&kfree[c1 % kKStages], (c1 / kKStages) & 1, true);
        }
      }
      if (ntiles == 0 && ok) {  // no rows: free the buffers for the partner as they land
        commit_to(&vfree[vb], (c / kVStages) & 1, true);
        if (c1 < nchunks) {
          if (!(ok = wait_all(&fullk[c1 % kKStages], (c1 / kKStages) & 1))) break;
          commit_to(&kfree[c1 % kKStages], (c1 / kKStages) & 1, true);
        }
      }
    }
    // The partner's last commits arrive on this CTA's free barriers: wait (bounded) for
    // their final phases, so nothing lands in this CTA's shared memory after it exits.
    if (ok) {
      for (int c = max(0, nchunks - kKStages); c < nchunks; ++c)
        mbar_wait_bounded(&kfree[c % kKStages], (c / kKStages) & 1, kWaitNs / 8);
      for (int c = max(0, nchunks - kVStages); c < nchunks; ++c)
        mbar_wait_bounded(&vfree[c % kVStages], (c / kVStages) & 1, kWaitNs / 8);
    }
    // MMAs committed but maybe not finished: a commit tracks every earlier MMA of the
    // issuing thread, so the last commit's barrier covers them all
    if (!ok && last_bar != nullptr) mbar_wait_bounded(last_bar, last_par, kWaitNs / 8);
  }

  fence_before();
  __syncthreads();
  // After an abort no consumer waits for the copies still landing: warp 8 waits
  // (bounded) for the last chunks it issued, so nothing lands after the CTA exits.
  if (*s_abort && warp == kCopyWarp && lane == 0) {
    for (int c = issued_k - kKStages; c < issued_k; ++c)
      if (c >= 0) mbar_wait_bounded(&fullk[c % kKStages], (c / kKStages) & 1, kWaitNs / 8);
    for (int c = issued_v - kVStages; c < issued_v; ++c)
      if (c >= 0) mbar_wait_bounded(&fullv[c % kVStages], (c / kVStages) & 1, kWaitNs / 8);
  }
  // Neither CTA of the cluster leaves while the other may still copy into it or
  // commit to its barriers (every wait above is bounded, so both arrive here).
  __syncthreads();
  cluster_sync_all();
  if (warp == 0) {
    fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(Sh::kTmemCols));
  }
}

}  // namespace ws
}  // namespace pa
