// prefill_ws.cuh -- chunked prefill on tcgen05 with warp specialisation.
//
// Causal attention of each sequence's chunk of new query tokens over its paged
// cache (what is computed: see prefill.cu), on sm_103a's tcgen05 MMAs with the
// accumulators in tensor memory (TMEM).  A query tile is 128 rows -- (token,
// query head) pairs of one kv head, head fastest -- which are TMEM lanes
// 0..127; keys are taken 128 at a time (a chunk).  A unit is four consecutive
// tiles of one (sequence, kv head); a cluster of two CTAs on two SMs takes a unit
// at a time, each CTA a PAIR of its tiles, A and B.  All four read the same keys,
// so each chunk of K and V is copied once per cluster (half by each CTA, with TMA
// multicast into both) and feeds the MMAs of both tiles of both CTAs.  The two
// tiles of a CTA take turns: while the softmax of one runs, the tensor cores run
// the other's P V and its next S (ping-pong).  The kernel is persistent: as many
// clusters as fit on the GPU at once, each taking units in the order of
// decreasing length until none is left; the K/V rings, the barriers' phases and
// the TMEM columns carry on from one unit to the next, so a unit's first copies,
// its Q and its first S overlap the previous unit's last chunk and its output.
// The phases run in different warps that hand over through mbarriers:
//
//   * warp 10: the unit ring.  It replays a greedy assignment of all units,
//     longest first, each to the cluster with the least work so far, and puts
//     this cluster's units into a ring up to four ahead; each is read by every
//     other warp.
//   * warp 8: the TMA copies of chunk c (counted over all units), K into K buffer
//     c % 2 once both tiles' S of chunk c - 2 have read it, V into V buffer c % 2
//     once both tiles' P V of chunk c - 2 have read it, each on its own mbarrier.  K: the pool seen as rows
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
//     S(c), then the unit's output out of TMEM; during a unit's last chunk they
//     load the next unit's Q (its S(0) waits for it, its first P V for the output).
//     P = exp2(s - m) goes back into the row's own S columns as 16-bit values, two
//     per 32-bit column: the 16 columns of keys 16 k .. 16 k + 15 become 8 columns
//     of P rounded to fp16 or, for bf16, 8 columns of rounded high parts and 8 of
//     low parts (~16 significant bits; P V is then two MMA groups).  The running
//     maximum moves only when it grows by more than 2^8; then the row's O is
//     rescaled in TMEM (P V(c - 1) is done by then: S(c) was issued after it).  In the last chunk tile A's threads zero the
//     V of keys past the sequence (or past the blocks loaded) in shared memory
//     first: P is 0 there, but 0 * NaN would poison O.  A tile whose rows end
//     before the pair's last chunk sees scores of -inf there (P = 0).
//
// TMEM: tile X at column 256 X: S/P in 0..127, O (D <= 128 columns) from 128; all
// 512 columns for the pair; one CTA per SM.  A unit's first P V_X overwrites O_X
// only after the softmax threads have read the previous unit's O_X out.
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
constexpr int kCopyWarp = 8, kMmaWarp = 9, kSchedWarp = 10;
// A cluster of two CTAs on two SMs takes a unit of four consecutive tiles of one
// (sequence, kv head), a pair per CTA; each CTA copies half of every chunk of K and V
// with TMA multicast into both, so each SM fetches half of the bytes its MMAs read.
constexpr int kCluster = 2, kUnitTiles = 2 * kCluster;
constexpr uint16_t kClusterMask = (1u << kCluster) - 1;
constexpr int kThreads = 11 * 32;
// The unit ring: the scheduler warp writes up to kUnitSlots units ahead; each is
// read by the 8 softmax warps, the copy warp and the MMA warp.
constexpr int kUnitSlots = 4, kUnitReaders = 10;
constexpr int kLoadsPerLane = 4;  // the scheduler's greedy assignment: up to 128 clusters
// A unit's fixed cost in chunk periods (its first S and its output; measured ~2.8)
constexpr int kUnitCost = 3;
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

// Packed pairs of fp32 values (low = first) and the paired fp32 operations of sm_100+:
// one instruction for both halves, each rounded as its scalar form
__device__ __forceinline__ uint64_t f2pack(float a, float b) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
  return r;
}
__device__ __forceinline__ float2 f2unpack(uint64_t v) {
  float a, b;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(v));
  return make_float2(a, b);
}
__device__ __forceinline__ uint64_t fma2(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ uint64_t mul2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ uint64_t add2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
// the largest of three (a NaN operand is ignored, as by fmaxf)
__device__ __forceinline__ float max3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

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

// The per-sequence figures unit selection needs, in shared memory (3 kMaxSeqsPerLaunch
// ints): ctx = tokens before the chunk, rows = its n G query rows, and its tiles.
// One warp fills it once per CTA (lane i: sequences i, i + 32, ..) and checks the
// lengths; returns the most chunks any unit reads.
__device__ int build_seq_table(const PrefillParams& p, int* tab) {
  const int lane = threadIdx.x & 31, G = p.group, S = p.num_seqs;
  bool bad = false;
  int longest = 0;
  for (int s = lane; s < S; s += 32) {
    const int L = __ldg(p.seq_lens + s), a = __ldg(p.query_start_loc + s), b = __ldg(p.query_start_loc + s + 1);
    const int n = b - a;
    int ctx = 0, rows = 0, nt = 0;
    if (L < 1 || L > p.max_seq_len || a < 0 || b > p.num_query_tokens || n < 0 || n > L) {
      bad = true;
    } else {
      ctx = L - n;
      rows = n * G;
      nt = (rows + kRows - 1) / kRows;
    }
    tab[s] = ctx;
    tab[kMaxSeqsPerLaunch + s] = rows;
    tab[2 * kMaxSeqsPerLaunch + s] = nt;
    if (nt) longest = max(longest, (ctx + (rows - 1) / G) / kKeys + 1);
  }
  if (bad && blockIdx.x == 0) set_error(p.err, kErrSeqLen);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) longest = max(longest, __shfl_xor_sync(0xffffffffu, longest, o));
  __syncwarp();
  return longest;
}

// Units of sequence s (per kv head) that read >= x chunks of keys, from the table of
// build_seq_table.  Tile j of s covers rows 128 j .. of its n G rows and reads chunks
// 0 .. (ctx + (row_hi - 1) / G) / 128, non-decreasing in j; a unit holds kUnitTiles
// consecutive tiles (those that exist) and reads what its last tile reads.  So the
// tiles reading >= x chunks are a suffix j >= j0 in closed form, and the units
// reading >= x are the last ones, from j0 / kUnitTiles on.
__device__ __forceinline__ int units_reading(const int* tab, int G, int s, int x) {
  const int ctx = tab[s], rows = tab[kMaxSeqsPerLaunch + s], nt = tab[2 * kMaxSeqsPerLaunch + s];
  const long long need = (long long)G * ((long long)kKeys * (x - 1) - ctx) + 1;  // rows a tile must reach
  if (nt == 0 || need > rows) return 0;
  const int j0 = need <= 1 ? 0 : static_cast<int>((need + kRows - 1) / kRows - 1);  // first tile reading >= x
  return (nt + kUnitTiles - 1) / kUnitTiles - j0 / kUnitTiles;
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
  // fullk[K], fullv[V], kfree[K], vfree[V], per tile 5 (sfull, pfull, pvdone, qfull,
  // ofree), ufull[U], uempty[U], never
  static constexpr int kNumBars = 2 * kKStages + 2 * kVStages + 2 * 5 + 2 * kUnitSlots + 1;
  static constexpr int kOffMisc = kOffBar + (kNumBars * 8 + 15) / 16 * 16;  // TMEM address, abort flag
  static constexpr int kOffUnits = kOffMisc + 16;                           // [kUnitSlots] int4: the unit ring
  static constexpr int kOffTab = kOffUnits + kUnitSlots * 16;               // unit selection's table
  static constexpr int kEnd = kOffTab + 3 * kMaxSeqsPerLaunch * 4;
  // more than half an SM's shared memory, so one CTA per SM: it takes all of TMEM
  static constexpr int kSmem = kEnd > 116 * 1024 ? kEnd : 116 * 1024;
  static constexpr int kTmemCols = 512;  // tile X at 256 X: S/P 0..127, O 128..128+D
};

// The figures of one unit that every role needs: the same in every role, and in both
// CTAs of the cluster except for the pair, which is this CTA's.
struct UnitView {
  int s, kvh, L, tok0, pair_lo, pair_hi, ntiles, ctx, nblk, nchunks;
};
template <int BS>
__device__ __forceinline__ UnitView unit_view(const PrefillParams& p, int4 u, uint32_t crank) {
  UnitView v;
  v.s = u.x;
  v.kvh = u.y;
  const int G = p.group;
  v.L = p.seq_lens[v.s];
  v.tok0 = p.query_start_loc[v.s];
  const int n = p.query_start_loc[v.s + 1] - v.tok0, rows = n * G;
  // this CTA's pair: tiles kUnitTiles unit + 2 crank and the next (either may be past the rows)
  v.pair_lo = (kUnitTiles * u.z + 2 * static_cast<int>(crank)) * kRows;
  v.pair_hi = min(rows, v.pair_lo + 2 * kRows);
  v.ntiles = v.pair_lo >= rows ? 0 : (v.pair_lo + kRows < rows ? 2 : 1);  // tiles with rows: A, then B
  // keys: what the unit's last row sees (the same in both CTAs: they share every chunk)
  const int unit_hi = min(rows, (kUnitTiles * u.z + kUnitTiles) * kRows);
  v.ctx = v.L - n;
  const int p_max = v.ctx + (unit_hi - 1) / G;  // last position any row of the unit has
  v.nblk = p_max / BS + 1;                      // blocks holding keys 0..p_max
  v.nchunks = (p_max + kKeys) / kKeys;
  return v;
}

template <typename T, int D, int BS>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_ws_kernel(const PrefillParams p, const __grid_constant__ CUtensorMap tmap_k,
                      const __grid_constant__ CUtensorMap tmap_v) {
  using Sh = Shape<T, D, BS>;
  static_assert(Sh::kSmem > 114 * 1024, "two CTAs on one SM would contend for TMEM");
  static_assert(Sh::kSmem <= 227 * 1024, "shared memory per CTA");
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
  uint64_t* tbars = vfree + kVStages;       // per tile X at 5 X: sfull, pfull, pvdone, qfull, ofree
  uint64_t* ufull = tbars + 10;             // [kUnitSlots] the scheduler wrote the slot
  uint64_t* uempty = ufull + kUnitSlots;    // [kUnitSlots] every reader took the slot
  uint64_t* never = uempty + kUnitSlots;    // nothing completes it: the timeout-path test waits on it
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(smem + Sh::kOffMisc);
  volatile int* s_abort = reinterpret_cast<volatile int*>(s_tmem + 1);  // a thread gave up
  volatile int* s_unit = reinterpret_cast<volatile int*>(smem + Sh::kOffUnits);  // [kUnitSlots][4]
  int* tab = reinterpret_cast<int*>(smem + Sh::kOffTab);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  // S(c) in TMEM (commit); P(c) in TMEM, O rescaled, V tail zeroed (128 arrivals); the
  // unit's last P V done (commit); the next unit's Q in shared memory (128 arrivals);
  // the unit's O read out of TMEM (128 arrivals)
  auto sfull = [&](int X) { return tbars + 5 * X; };
  auto pfull = [&](int X) { return tbars + 5 * X + 1; };
  auto pvdone = [&](int X) { return tbars + 5 * X + 2; };
  auto qfull = [&](int X) { return tbars + 5 * X + 3; };
  auto ofree = [&](int X) { return tbars + 5 * X + 4; };

  griddep_launch_dependents();
  griddep_wait();
  const uint32_t crank = cluster_rank();
  if (tid == 0) {
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
      mbar_init(qfull(X), kSoftmaxThreads);
      mbar_init(ofree(X), kSoftmaxThreads);
    }
    for (int i = 0; i < kUnitSlots; ++i) {
      mbar_init(&ufull[i], 1);
      mbar_init(&uempty[i], kUnitReaders);
    }
    mbar_init(never, 1);
    fence_barrier_init();
  }
  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_addr(s_tmem)),
                 "r"(Sh::kTmemCols));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  fence_before();
  __syncthreads();
  fence_after();
  cluster_sync_all();  // both CTAs' mbarriers are initialised before either copies into the other
  const uint32_t tmem = *s_tmem;
  const int G = p.group;
  int issued_k = 0, issued_v = 0;  // chunks (of all units) whose K (V) copies warp 8 issued
  auto wait = [&](uint64_t* bar, int parity) { return wait_or_abort(bar, parity, s_abort, p.err); };
  // the k-th unit of the ring (the slot's ufull phase k / kUnitSlots); every reader
  // takes it once and frees it with one arrival per warp
  auto take_unit = [&](int k, int4& u) -> bool {
    const int slot = k % kUnitSlots;
    if (!__all_sync(0xffffffffu, wait(&ufull[slot], (k / kUnitSlots) & 1))) return false;
    u = make_int4(s_unit[4 * slot], s_unit[4 * slot + 1], s_unit[4 * slot + 2], 0);
    __syncwarp();
    if (lane == 0) mbar_arrive(&uempty[slot]);
    return true;
  };

  if (warp < 8) {
    // ================= softmax: tile X, row r, all keys of each chunk of each unit =================
    const int X = warp >> 2, r = tid & (kRows - 1);
    const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
    const uint32_t t_s = tmem + 256 * X + lane_base;
    const uint32_t t_o = t_s + kKeys;
    const float sl2 = p.scale_log2;
    const uint32_t sq = smem_addr(smem + X * Sh::kQTile + (r / 8) * (D / 8) * 128 + (r % 8) * 16);
    // this thread's row of Q_X for unit v into shared memory: every 16-byte piece in
    // flight at once, zeros for a padding row (completed and handed over by q_landed)
    auto load_q = [&](const UnitView& v) {
      const int row = v.pair_lo + X * kRows + r;
      const bool valid = row < v.pair_hi;
      const T* q = static_cast<const T*>(p.q) +
                   ((long long)(v.tok0 + (valid ? row / G : 0)) * p.num_heads + (long long)v.kvh * G +
                    (valid ? row % G : 0)) * D;
      const uint32_t nbytes = valid ? 16u : 0u;
#pragma unroll
      for (int c = 0; c < D / 8; ++c)
        asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(sq + c * 128), "l"(q + 8 * c), "r"(nbytes)
                     : "memory");
    };
    auto q_landed = [&]() {  // the Q copies done, visible to the MMAs, handed over
      asm volatile("cp.async.wait_all;" ::: "memory");
      fence_proxy_async_smem();
      mbar_arrive(qfull(X));
    };
    int cx = 0, ux = 0;  // chunks and units this tile had rows in: the phases of its barriers
    int g = 0;           // chunks of all units before this one: the K/V ring positions
    int4 u;
    bool ok = take_unit(0, u);
    UnitView U{};
    if (ok && u.x >= 0) {
      U = unit_view<BS>(p, u, crank);
      if (U.ntiles > X) {
        load_q(U);
        q_landed();
      }
    }
    for (int k = 0; ok && u.x >= 0; ++k) {
      int4 un = make_int4(-1, 0, 0, 0);  // the next unit, taken during this one's last chunk
      UnitView N{};
      auto next = [&]() {
        if (!(ok = take_unit(k + 1, un))) return;
        if (un.x >= 0) {
          N = unit_view<BS>(p, un, crank);
          if (N.ntiles > X) load_q(N);  // Q_X is free: the last S_X of this unit is done
        }
      };
      if (U.ntiles > X) {
        const int row = U.pair_lo + X * kRows + r;
        const bool valid = row < U.pair_hi;
        const int pos = valid ? U.ctx + row / G : U.ctx + (U.pair_hi - 1) / G;  // a padding row behaves as a real one
        const int kz = min(U.L, U.nblk * BS);  // first key whose V must read as zero
        float m = -INFINITY, l = 0.f;
        for (int c = 0; c < U.nchunks; ++c, ++cx) {
          // tcgen05.ld / st are warp-collective (.sync.aligned): every branch around them
          // is taken by the whole warp, so each wait's outcome is agreed across the warp
          if (!(ok = __all_sync(0xffffffffu, wait(sfull(X), cx & 1)))) break;
          fence_after();
          if (c == U.nchunks - 1) {
            next();
            if (!ok) break;
          }
          float sv[kKeys];
          ld128(t_s, sv);
          const int lim = pos - c * kKeys;  // keys 0..lim of the chunk are visible to the row
          if (lim < kKeys - 1) {           // the diagonal chunk (or past it): hide the later keys
#pragma unroll
            for (int j = 0; j < kKeys; ++j)
              if (j > lim) sv[j] = -INFINITY;
          }
          // the row maximum of the raw scores, as a tree of three-input maxima in 8 chains
          // (scale > 0 keeps the order)
          float mx;
          {
            static_assert(kKeys % 16 == 0, "8 chains, two keys a step");
            float t[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) t[i] = fmaxf(sv[i], sv[8 + i]);
#pragma unroll
            for (int j = 16; j < kKeys; j += 16)
#pragma unroll
              for (int i = 0; i < 8; ++i) t[i] = max3(t[i], sv[j + i], sv[j + 8 + i]);
            mx = fmaxf(max3(t[0], t[1], t[2]), max3(max3(t[3], t[4], t[5]), t[6], t[7])) * sl2;
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
            // P = 2^(scale * s - m) (s = -inf gives 0): the scaling of a pair of scores and
            // the row sums in paired fp32 operations
            const uint64_t sl2x2 = f2pack(sl2, sl2), negm2 = f2pack(-m, -m);
            uint64_t ps2[2] = {f2pack(0.f, 0.f), f2pack(0.f, 0.f)};
#pragma unroll
            for (int k2 = 0; k2 < kKeys / 16; ++k2) {
              uint32_t blk[8 * kParts];
#pragma unroll
              for (int j = 0; j < 8; ++j) {
                const float2 y = f2unpack(fma2(f2pack(sv[16 * k2 + 2 * j], sv[16 * k2 + 2 * j + 1]), sl2x2, negm2));
                const float x0 = ex2(y.x), x1 = ex2(y.y);
                ps2[j & 1] = add2(ps2[j & 1], f2pack(x0, x1));
                blk[j] = pack2<T>(x0, x1);
                if constexpr (kParts == 2) {
                  const float2 back = unpack2<T>(blk[j]);
                  blk[8 + j] = pack2<T>(x0 - back.x, x1 - back.y);
                }
              }
              if constexpr (kParts == 2) st16(t_s + 16 * k2, blk);
              else st8(t_s + 16 * k2, blk);
            }
            wait_st();
            const float2 s0 = f2unpack(ps2[0]), s1 = f2unpack(ps2[1]);
            l += (s0.x + s0.y) + (s1.x + s1.y);
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
          if (X == 0 && c == U.nchunks - 1 && kz < (c + 1) * kKeys) {
            const int gc = g + c;
            if (!(ok = __all_sync(0xffffffffu, wait(&fullv[gc % kVStages], (gc / kVStages) & 1)))) break;
            // block b's tile [D][bs]: dim d's keys 8 g .. 8 g + 7 are the 16 bytes at d * 2 bs + 16 g
            // within the row, moved by the swizzle (16-byte unit bits xor'ed with bits 7 and up)
            unsigned char* vbase = smem + Sh::kOffV + (gc % kVStages) * Sh::kVBytes;
            constexpr int kRow = 2 * BS, kUnits = kRow / 16;
            const int k0 = kz - c * kKeys;  // first key to clear (0 <= k0 < kKeys)
            const int g0 = k0 / 8;          // the 8-key group holding it
            for (int i = tid; i < (kKeys / 8 - g0) * D; i += kSoftmaxThreads) {
              const int g8 = g0 + i / D, d = i % D;  // keys 8 g8 .. 8 g8 + 7 of dim d
              const int a = d * kRow + ((8 * g8) % BS) * 2;
              unsigned char* ptr = vbase + ((8 * g8) / BS) * Sh::kTile + (a ^ (((a >> 7) & (kUnits - 1)) << 4));
              if (8 * g8 >= k0) {
                *reinterpret_cast<uint4*>(ptr) = make_uint4(0, 0, 0, 0);
              } else {
                for (int kk = k0 - 8 * g8; kk < 8; ++kk) *reinterpret_cast<T*>(ptr + 2 * kk) = DType<T>::from_f32(0.f);
              }
            }
            fence_proxy_async_smem();
          }
          fence_before();
          mbar_arrive(pfull(X));
        }
        if (!ok) break;
        if (un.x >= 0 && N.ntiles > X) q_landed();  // the next unit's first S_X may go
        // the unit's output: O / l, read out of TMEM (then the columns are free for the
        // next unit's P V), rounded to T, stored as the row's D contiguous elements
        if (!(ok = __all_sync(0xffffffffu, wait(pvdone(X), ux & 1)))) break;
        fence_after();
        const float inv = 1.f / l;
        const uint64_t inv2 = f2pack(inv, inv);
        uint32_t o16[D / 2];
#pragma unroll
        static_assert(D % 64 == 0, "O read 64 columns at a time");
        for (int c0 = 0; c0 < D; c0 += 64) {  // 64 columns per wait
          float o[64];
          ld64(t_o + c0, o);
#pragma unroll
          for (int j = 0; j < 64; j += 2) {
            const float2 v = f2unpack(mul2(f2pack(o[j], o[j + 1]), inv2));
            o16[(c0 + j) / 2] = pack2<T>(v.x, v.y);
          }
        }
        fence_before();
        mbar_arrive(ofree(X));
        if (valid) {
          T* out = static_cast<T*>(p.out) +
                   ((long long)(U.tok0 + row / G) * p.num_heads + (long long)U.kvh * G + row % G) * D;
#pragma unroll
          for (int j = 0; j < D / 8; ++j)
            reinterpret_cast<uint4*>(out)[j] = make_uint4(o16[4 * j], o16[4 * j + 1], o16[4 * j + 2], o16[4 * j + 3]);
        }
        ++ux;
      } else {  // no rows of this tile in the unit: only the next unit's Q
        next();
        if (!ok) break;
        if (un.x >= 0 && N.ntiles > X) q_landed();
      }
      g += U.nchunks;
      u = un;
      U = N;
    }
    asm volatile("cp.async.wait_all;" ::: "memory");  // no Q copy lands after the CTA exits
  } else if (warp == kCopyWarp) {
    // ================= copies (warp 8): K gathers, then V boxes, chunk after chunk of each unit =================
    // This CTA issues its half of each chunk's copies, each into both CTAs of the
    // cluster: lane i the gather4 load crank * kGathers / 2 + i of K (8-dim slice dc,
    // keys 64 h .. 64 h + 63), lane b the V box of the chunk's block b when b % 2 is
    // its rank.  Each CTA's full barriers expect the whole chunk.  Buffer positions run
    // on over the units (g counts the chunks of all units so far).
    constexpr int kGathers = (D / 8) * (kKeys / 64), kMine = kGathers / kCluster;
    static_assert(kGathers <= 32 && Sh::kBlocks <= 32 && kGathers % kCluster == 0, "one copy per lane");
    const int gi = static_cast<int>(crank) * kMine + lane;  // this lane's gather (lanes < kMine)
    const int dc = gi / (kKeys / 64), h = gi % (kKeys / 64);
    bool ok = true;
    int g = 0;
    for (int k = 0; ok; ++k) {
      int4 u;
      if (!(ok = take_unit(k, u)) || u.x < 0) break;
      const UnitView U = unit_view<BS>(p, u, crank);
      const int32_t* bt = p.block_tables + (long long)U.s * p.max_blocks_per_seq;
      auto phys_of = [&](int c) {  // lane b: the physical block of the chunk's block b (-1 past the keys)
        const int gb = c * Sh::kBlocks + lane;
        return lane < Sh::kBlocks && gb < U.nblk ? __ldg(bt + gb) : -1;
      };
      int ph = phys_of(0);  // the next chunk's table entries land while a chunk is in flight
      for (int c = 0; c < U.nchunks; ++c) {
        const int gc = g + c, kb = gc % kKStages, vb = gc % kVStages;
        const bool live = lane < Sh::kBlocks && c * Sh::kBlocks + lane < U.nblk;
        const bool bad = ph < 0 || ph >= p.num_blocks;
        if (live && bad) set_error(p.err, kErrBlockId);
        const int ph0 = __shfl_sync(0xffffffffu, bad ? 0 : ph, 0);  // block 0 of a chunk always holds keys
        // a block past the keys: any rows do (S there is masked; its V is not copied)
        const long long tl = (long long)(live ? (bad ? 0 : ph) : ph0) * p.num_kv_heads + U.kvh;
        const int nlive = __popc(__ballot_sync(0xffffffffu, live));
        int rw[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {  // the rows (16 keys each) of this lane's 64 keys
          const int key = 64 * h + 16 * q;
          const long long tb = __shfl_sync(0xffffffffu, tl, key / BS);
          rw[q] = static_cast<int>((tb * (D / 8) + dc) * (BS / 16) + (key % BS) / 16);
        }
        if (gc >= kKStages &&  // both CTAs' S read the buffer (in both CTAs)
            !(ok = __all_sync(0xffffffffu, wait(&kfree[kb], ((gc - kKStages) / kKStages) & 1))))
          break;
        if (lane == 0) mbar_arrive_expect_tx(&fullk[kb], Sh::kKBytes);
        __syncwarp();
        if (lane < kMine)  // lands as [64 keys][8 dims] in the slice's rows, in both CTAs
          tma_gather4_mc(smem + Sh::kOffK + kb * Sh::kKBytes + dc * (kKeys * 16) + h * (64 * 16), &tmap_k, rw,
                         &fullk[kb], kClusterMask);
        issued_k = gc + 1;
        if (gc >= kVStages &&  // both CTAs' P V read the buffer (in both CTAs)
            !(ok = __all_sync(0xffffffffu, wait(&vfree[vb], ((gc - kVStages) / kVStages) & 1))))
          break;
        if (lane == 0) mbar_arrive_expect_tx(&fullv[vb], nlive * Sh::kTile);
        __syncwarp();
        if (live && lane % kCluster == static_cast<int>(crank))  // the (block, kv head) tile [D][bs], swizzled;
          tma_2d_mc(smem + Sh::kOffV + vb * Sh::kVBytes + lane * Sh::kTile, &tmap_v, 0,  // V past the keys is zeroed
                    static_cast<int>(tl * D), &fullv[vb], kClusterMask);                // by the softmax threads
        issued_v = gc + 1;
        ph = phys_of(c + 1);
      }
      g += U.nchunks;
    }
  } else if (warp == kSchedWarp) {
    // ================= the unit ring (warp 10): this cluster's units =================
    // Every cluster replays the same greedy assignment of all units of the launch:
    // longest first (ties by sequence, kv head, unit), each to the cluster with the
    // least work so far (ties to the lowest index), a unit's work being its chunks +
    // kUnitCost;
    // this cluster's units enter the ring in that order.  Both CTAs of a cluster write
    // the same sequence; a unit with x < 0 ends it.
    const int longest = build_seq_table(p, tab);
    const int cid = blockIdx.x / kCluster, ncl = gridDim.x / kCluster;  // ncl <= 32 kLoadsPerLane
    long long load[kLoadsPerLane];  // work of cluster lane + 32 i
#pragma unroll
    for (int i = 0; i < kLoadsPerLane; ++i) load[i] = lane + 32 * i < ncl ? 0 : LLONG_MAX;
    int k = 0;
    bool ok = true;
    auto push = [&](int s, int kvh, int ui) {  // the next unit of this cluster into the ring
      const int slot = k % kUnitSlots;
      if (k >= kUnitSlots && !__all_sync(0xffffffffu, wait(&uempty[slot], ((k - kUnitSlots) / kUnitSlots) & 1))) {
        ok = false;
        return;
      }
      if (lane == 0) {
        s_unit[4 * slot] = s;
        s_unit[4 * slot + 1] = kvh;
        s_unit[4 * slot + 2] = ui;
        mbar_arrive(&ufull[slot]);  // release: the slot's words before the phase completes
      }
      __syncwarp();
      ++k;
    };
    const int S = p.num_seqs, Hkv = p.num_kv_heads;
    for (int x = longest; x >= 1 && ok; --x) {
      for (int s0 = 0; s0 < S && ok; s0 += 32) {  // lane i: sequence s0 + i's units of exactly x chunks
        const int s = s0 + lane;
        int e = 0, first = 0;
        if (s < S) {
          const int a = units_reading(tab, G, s, x), b = units_reading(tab, G, s, x + 1);
          e = a - b;
          first = (tab[2 * kMaxSeqsPerLaunch + s] + kUnitTiles - 1) / kUnitTiles - a;
        }
        for (unsigned m = __ballot_sync(0xffffffffu, e > 0); m && ok; m &= m - 1) {
          const int src = __ffs(m) - 1;
          const int ee = __shfl_sync(0xffffffffu, e, src), ff = __shfl_sync(0xffffffffu, first, src);
          for (int kvh = 0; kvh < Hkv && ok; ++kvh)
            for (int jj = 0; jj < ee && ok; ++jj) {
              long long best = load[0];
              int bi = lane;
#pragma unroll
              for (int i = 1; i < kLoadsPerLane; ++i)
                if (load[i] < best) {
                  best = load[i];
                  bi = lane + 32 * i;
                }
#pragma unroll
              for (int o = 16; o > 0; o >>= 1) {
                const long long ob = __shfl_xor_sync(0xffffffffu, best, o);
                const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
                if (ob < best || (ob == best && oi < bi)) {
                  best = ob;
                  bi = oi;
                }
              }
              if (bi == cid) push(s0 + src, kvh, ff + jj);
#pragma unroll
              for (int i = 0; i < kLoadsPerLane; ++i)
                if (bi == lane + 32 * i) load[i] += x + kUnitCost;
            }
        }
      }
    }
    if (ok) push(-1, 0, 0);
  } else {
    // ================= MMAs (warp 9): per unit S_X(0), then per chunk P V_A(c), S_A(c + 1), P V_B(c), S_B(c + 1) =================
    // The whole warp runs the loop and the waits (so the loop state and the descriptors
    // stay warp-uniform); one elected lane issues the MMAs and the commits.  A CTA
    // without rows in a unit (the unit's second pair missing) still frees each buffer
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
    int cx[2] = {0, 0}, ux[2] = {0, 0};  // per tile: chunks (S, P V) and units it had rows in
    auto issue_s = [&](int Xm, int gc) {  // S_X = Q_X K(gc)^T into X's S columns
      if (leader) {
        const uint64_t da = dq0 + Xm * (Sh::kQTile >> 4), db = dk0 + (gc % kKStages) * (Sh::kKBytes >> 4);
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks)
          mma(tmem + 256 * Xm, da + ks * 16, db + ks * (2 * kKeys), kIdS, ks > 0);
      }
      commit_to(sfull(Xm), cx[Xm] & 1);
    };
    auto issue_pv = [&](int Xm, int gc, bool first) {  // O_X (+)= P_X V(gc): high parts, then low parts
      if (leader) {
        const uint64_t db = dv0 + (gc % kVStages) * (Sh::kVBytes >> 4);
        const uint32_t tb = tmem + 256 * Xm;
#pragma unroll
        for (int part = 0; part < kParts; ++part) {
#pragma unroll
          for (int kk = 0; kk < kKeys / 16; ++kk)  // keys 16 kk ..: high parts in 8 columns, low in the next 8
            mma_ts(tb + kKeys, tb + 16 * kk + 8 * part,
                   db + (((16 * kk) / BS) * Sh::kTile + ((16 * kk) % BS) * 2) / 16, kIdO, !first || part > 0 || kk > 0);
        }
      }
    };
    // the timeout-path test: the first wait runs out on `never` (no MMA issued yet);
    // the producer then drains its copies with the normal limit
    bool ok = __all_sync(0xffffffffu, !p.test_wait_ns || wait_or_abort(never, 0, s_abort, p.err, p.test_wait_ns));
    int g = 0;  // chunks of all units so far
    for (int k = 0; ok; ++k) {
      int4 u;
      if (!(ok = take_unit(k, u)) || u.x < 0) break;
      const UnitView U = unit_view<BS>(p, u, crank);
      const int nt = U.ntiles, nc = U.nchunks;
      // S of the unit's first chunk, for each tile as soon as its Q has landed (the
      // previous unit's P V run ahead of it on the tensor cores)
      if (!(ok = wait_all(&fullk[g % kKStages], (g / kKStages) & 1))) break;
      for (int Xm = 0; Xm < nt && ok; ++Xm) {
        if (!(ok = wait_all(qfull(Xm), ux[Xm] & 1))) break;
        fence_after();
        issue_s(Xm, g);
      }
      if (!ok) break;
      commit_to(&kfree[g % kKStages], (g / kKStages) & 1, true);
      for (int c = 0; c < nc && ok; ++c) {
        const int gc = g + c, vb = gc % kVStages, g1 = gc + 1;
        if (!(ok = wait_all(&fullv[vb], (gc / kVStages) & 1))) break;
        for (int Xm = 0; Xm < nt && ok; ++Xm) {
          if (!(ok = wait_all(pfull(Xm), cx[Xm] & 1))) break;  // the softmax wrote P_X(c)
          // the first P V of a unit overwrites O_X: the previous unit's O_X is read out
          if (c == 0 && ux[Xm] > 0 && !(ok = wait_all(ofree(Xm), (ux[Xm] - 1) & 1))) break;
          fence_after();
          issue_pv(Xm, gc, c == 0);
          if (Xm == nt - 1) commit_to(&vfree[vb], (gc / kVStages) & 1, true);
          if (c == nc - 1) commit_to(pvdone(Xm), ux[Xm] & 1);  // O_X is complete
          ++cx[Xm];
          if (c + 1 < nc) {
            if (Xm == 0 && !(ok = wait_all(&fullk[g1 % kKStages], (g1 / kKStages) & 1))) break;
            // S_X(c + 1) overwrites the columns P V_X(c) reads, issued right behind it: MMAs
            // of one thread run in issue order, so no wait is needed between the two
            fence_after();
            issue_s(Xm, g1);
            if (Xm == nt - 1) commit_to(&kfree[g1 % kKStages], (g1 / kKStages) & 1, true);
          }
        }
        if (nt == 0 && ok) {  // no rows: free the buffers for the partner as they land
          commit_to(&vfree[vb], (gc / kVStages) & 1, true);
          if (c + 1 < nc) {
            if (!(ok = wait_all(&fullk[g1 % kKStages], (g1 / kKStages) & 1))) break;
            commit_to(&kfree[g1 % kKStages], (g1 / kKStages) & 1, true);
          }
        }
      }
      for (int Xm = 0; Xm < nt; ++Xm) ++ux[Xm];
      g += nc;
    }
    // The partner's last commits arrive on this CTA's free barriers: wait (bounded) for
    // their final phases, so nothing lands in this CTA's shared memory after it exits.
    if (ok) {
      for (int c = max(0, g - kKStages); c < g; ++c)
        mbar_wait_bounded(&kfree[c % kKStages], (c / kKStages) & 1, kWaitNs / 8);
      for (int c = max(0, g - kVStages); c < g; ++c)
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
