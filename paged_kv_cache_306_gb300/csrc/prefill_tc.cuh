// prefill_tc.cuh -- chunked prefill on the 5th-generation tensor cores (tcgen05, TMEM).
//
// Causal attention of each sequence's chunk of new query tokens over its paged
// cache (what is computed: see prefill.cu), on sm_103a's tcgen05 MMA, whose
// accumulators live in tensor memory (TMEM):
//
//   * A CTA of 8 warps owns a tile of 128 query rows -- (token, query head) pairs
//     of one kv head, head fastest -- and TMEM lanes 0..127 are those rows.  Two
//     threads share a row, one from each group of 4 warps (a warp reaches TMEM
//     lanes 32 (warp % 4) ..): each takes half of a chunk's keys in the softmax
//     and half of the head dims in the epilogue; the row maximum and sum are
//     combined through shared memory.
//   * Keys are taken 64 at a time (4 blocks of 16 or 2 of 32).  Their K and V
//     tiles arrive by 1-D bulk copies (TMA unit) into one stage; the next chunk's
//     copies start as soon as the S MMAs have read K and V has been re-laid out,
//     so they run under the softmax and P V.  At under 113 KiB of shared memory
//     two CTAs share an SM, and each one's serial phases fill the other's gaps.  A pool K tile [D/8][bs][8] is already the K-major
//     core-matrix layout the MMA reads (8 keys x 16 bytes per core matrix), so
//     S = Q K^T is issued straight from the stage: one MMA of M=128, N=bs, K=16
//     per block and 16-dim step, into TMEM columns 0..63.
//   * The threads load their S rows from TMEM (tcgen05.ld), apply the causal
//     mask, and update the online softmax; the running maximum is moved only when
//     it grows by more than 2^8, so O (TMEM columns 64..64+D) is rescaled rarely.
//     P = exp2(s - m) goes to shared memory as a rounded 16-bit high part and the
//     rounded remainder (~16 significant bits), K-major core matrices.
//   * V's pool tile [D][bs] has 2*bs-byte rows, not the 16-byte core-matrix rows
//     the MMA needs, so the chunk's V is re-laid out in shared memory as
//     [key/8][D][8] (keys past the sequence zeroed), then O += P V is two MMA
//     groups (P's high and low parts) of M=128, N=D, K=16 per 16 keys.
//   * One elected thread issues every MMA and commits them to mbarriers; every
//     wait is bounded (1 s of %globaltimer); on a timeout the CTA records
//     PA_DEVERR_TIMEOUT, lets its copies in flight land (bounded) and frees TMEM.
#pragma once

#include "pa_device.cuh"
#include "pa_launch.h"

namespace pa {
namespace tc {

constexpr int kRows = 128;     // query rows per CTA (= TMEM lanes)
constexpr int kThreads = 256;  // 8 warps: two threads per row
constexpr int kKeys = 64;      // keys per chunk
constexpr uint64_t kWaitNs = 1000000000ull;

// shared-memory matrix descriptor (tcgen05): K-major, no swizzle; lbo = byte
// distance between core matrices adjacent along K, sbo = along M / N
__device__ __forceinline__ uint64_t sdesc(uint32_t addr, uint32_t lbo, uint32_t sbo) {
  return (uint64_t)((addr >> 4) & 0x3FFF) | ((uint64_t)((lbo >> 4) & 0x3FFF) << 16) |
         ((uint64_t)((sbo >> 4) & 0x3FFF) << 32) | ((uint64_t)1 << 46);
}

// instruction descriptor for kind::f16: fp32 accumulate, A and B of type T, both K-major
template <typename T>
__host__ __device__ constexpr uint32_t idesc(int M, int N) {
  return (1u << 4) | ((std::is_same<T, __nv_bfloat16>::value ? 1u : 0u) << 7) |
         ((std::is_same<T, __nv_bfloat16>::value ? 1u : 0u) << 10) | ((uint32_t)(N >> 3) << 17) |
         ((uint32_t)(M >> 4) << 24);
}

__device__ __forceinline__ void mma(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t id, bool accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.u32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a), "l"(b), "r"(id), "r"((uint32_t)accumulate));
}

__device__ __forceinline__ void commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_addr(bar))
               : "memory");
}

__device__ __forceinline__ void fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// 32 consecutive fp32 columns of this thread's TMEM lane (the load and its wait in one
// statement, so no use of the registers can be scheduled before the wait)
__device__ __forceinline__ void ld32(uint32_t taddr, float (&v)[32]) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
        "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
        "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr)
      : "memory");
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

__device__ __forceinline__ void st32(uint32_t taddr, const float (&v)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
      "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
      "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])), "r"(__float_as_uint(v[3])),
      "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])), "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])),
      "r"(__float_as_uint(v[8])), "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])),
      "r"(__float_as_uint(v[11])), "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])),
      "r"(__float_as_uint(v[14])), "r"(__float_as_uint(v[15])), "r"(__float_as_uint(v[16])),
      "r"(__float_as_uint(v[17])), "r"(__float_as_uint(v[18])), "r"(__float_as_uint(v[19])),
      "r"(__float_as_uint(v[20])), "r"(__float_as_uint(v[21])), "r"(__float_as_uint(v[22])),
      "r"(__float_as_uint(v[23])), "r"(__float_as_uint(v[24])), "r"(__float_as_uint(v[25])),
      "r"(__float_as_uint(v[26])), "r"(__float_as_uint(v[27])), "r"(__float_as_uint(v[28])),
      "r"(__float_as_uint(v[29])), "r"(__float_as_uint(v[30])), "r"(__float_as_uint(v[31]))
      : "memory");
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

template <typename T, int D, int BS>
struct Shape {
  static constexpr int kTile = D * BS * 2;                 // one block's K (or V) tile
  static constexpr int kBlocks = kKeys / BS;               // blocks per chunk
  static constexpr int kQBytes = kRows * D * 2;            // Q, core-matrix layout
  static constexpr int kStageBytes = 2 * kBlocks * kTile;  // K tiles, then V tiles
  static constexpr int kV2Bytes = kKeys * D * 2;           // V re-laid out [key/8][D][8]
  static constexpr int kPBytes = kRows * kKeys * 2;        // P high (then P low)
  static constexpr int kOffStage = kQBytes;
  static constexpr int kOffV2 = kOffStage + kStageBytes;
  static constexpr int kOffP = kOffV2 + kV2Bytes;
  static constexpr int kOffBar = kOffP + 2 * kPBytes;
  static constexpr int kSmem = kOffBar + 8 * 8 + 16;  // <= 113 KiB: two CTAs per SM
  static constexpr int kTmemCols = 256;  // S: 64 columns, O: D columns at 64
};

// grid: one CTA per tile of 128 rows (an upper bound on the tiles; the CTAs past the real ones exit)
template <typename T, int D, int BS>
__global__ void __launch_bounds__(kThreads, 2) prefill_tc_kernel(const PrefillParams p) {
  using Sh = Shape<T, D, BS>;
  extern __shared__ __align__(1024) unsigned char smem[];
  unsigned char* sQ = smem;
  unsigned char* sStage = smem + Sh::kOffStage;
  unsigned char* sV2 = smem + Sh::kOffV2;
  unsigned char* sP = smem + Sh::kOffP;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + Sh::kOffBar);
  uint64_t* s_done = full + 1;
  uint64_t* o_done = full + 2;
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(full + 3);
  int* s_tile = reinterpret_cast<int*>(full + 4);  // sequence, kv head, tile (or -1)
  const int tid = threadIdx.x, warp = tid >> 5;

  griddep_launch_dependents();
  griddep_wait();

  // ---- which tile: walk the sequences' tile counts (tiles of a sequence are taken last first,
  // so the longest ones start early)
  if (tid == 0) {
    const int G = p.group, Hkv = p.num_kv_heads;
    long long t = blockIdx.x;
    int found = -1, fk = 0, fj = 0;
    for (int s = 0; s < p.num_seqs && found < 0; ++s) {
      const int L = p.seq_lens[s], a = p.query_start_loc[s], b = p.query_start_loc[s + 1];
      const int n = b - a;
      if (L < 1 || L > p.max_seq_len || a < 0 || b > p.num_query_tokens || n < 0 || n > L) {
        if (blockIdx.x == 0) set_error(p.err, kErrSeqLen);
        continue;
      }
      const long long tiles = (long long)((n * G + kRows - 1) / kRows);
      if (t < tiles * Hkv) {
        found = s;
        fk = static_cast<int>(t / tiles);
        fj = static_cast<int>(tiles - 1 - t % tiles);
      } else {
        t -= tiles * Hkv;
      }
    }
    s_tile[0] = found;
    s_tile[1] = fk;
    s_tile[2] = fj;
    mbar_init(full, 1);
    mbar_init(s_done, 1);
    mbar_init(o_done, 1);
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

  // ---- TMEM: S in columns [0, 64), O in [64, 64 + D)
  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_addr(s_tmem)),
                 "r"(Sh::kTmemCols));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }

  // ---- this thread's row and half; Q into shared memory (core matrices: 8 rows x 16 bytes)
  const int r = tid & (kRows - 1), half = tid >> 7, row = row_lo + r;
  const bool valid = row < row_hi;
  const int pos = valid ? ctx + row / G : p_max;  // a padding row behaves as the last real one
  {
    const T* q = static_cast<const T*>(p.q) +
                 ((long long)(tok0 + (valid ? row / G : 0)) * p.num_heads + (long long)kvh * G + (valid ? row % G : 0)) * D;
#pragma unroll
    for (int c = half * (D / 16); c < (half + 1) * (D / 16); ++c) {
      const uint4 v = valid ? __ldg(reinterpret_cast<const uint4*>(q) + c) : make_uint4(0, 0, 0, 0);
      *reinterpret_cast<uint4*>(sQ + (r / 8) * (D / 8) * 128 + c * 128 + (r % 8) * 16) = v;
    }
  }

  // ---- producer: blocks of chunk c into the stage (thread 0)
  const int32_t* bt = p.block_tables + (long long)s * p.max_blocks_per_seq;
  // the table entries of the next chunk to issue, loaded one chunk ahead (thread 0)
  int phys[Sh::kBlocks];
  auto load_table = [&](int c) {
#pragma unroll
    for (int b = 0; b < Sh::kBlocks; ++b) {
      const int gb = c * Sh::kBlocks + b;
      phys[b] = gb < nblk ? __ldg(bt + gb) : -1;
    }
  };
  auto issue = [&](int c) {
    unsigned char* st = sStage;
    int nv = 0;
#pragma unroll
    for (int b = 0; b < Sh::kBlocks; ++b)
      if (c * Sh::kBlocks + b < nblk) ++nv;
    mbar_arrive_expect_tx(full, 2 * nv * Sh::kTile);
#pragma unroll
    for (int b = 0; b < Sh::kBlocks; ++b) {
      if (c * Sh::kBlocks + b >= nblk) continue;
      int ph = phys[b];
      if (ph < 0 || ph >= p.num_blocks) {
        set_error(p.err, kErrBlockId);
        ph = 0;
      }
      const long long tl = (long long)ph * p.num_kv_heads + kvh;
      bulk_copy_g2s(st + b * Sh::kTile, static_cast<const unsigned char*>(p.k_cache) + tl * Sh::kTile, Sh::kTile,
                    full);
      bulk_copy_g2s(st + (Sh::kBlocks + b) * Sh::kTile, static_cast<const unsigned char*>(p.v_cache) + tl * Sh::kTile,
                    Sh::kTile, full);
    }
    load_table(c + 1);  // lands while this chunk is processed
  };
  if (tid == 0) {
    load_table(0);
    issue(0);
  }
  // chunk whose copies, S MMAs or P V MMAs are in flight and not yet waited for (-1: none); every
  // thread tracks them alike, so that a CTA that gives up waits for exactly these before it exits
  int pend_full = 0, pend_s = -1, pend_o = -1;
  fence_proxy_async_smem();  // Q's generic stores before the MMAs read it
  fence_before();
  __syncthreads();
  fence_after();
  const uint32_t tmem = *s_tmem;
  const uint32_t t_s = tmem, t_o = tmem + kKeys;
  const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
  constexpr int kHalfKeys = kKeys / 2, kHalfD = D / 2;
  // P's shared-memory piece (16 bytes) of row rr, half hh, key group kg (K-major core matrices)
  auto p_off = [&](int rr, int hh, int kg) {
    return (rr / 8) * (kKeys / 8) * 128 + (hh * (kHalfKeys / 8) + kg) * 128 + (rr % 8) * 16;
  };
  // The two threads of a row exchange their half's maximum (and at the end their
  // sums) through shared memory: each writes into the first P piece its partner
  // will write, and only the partner reads it -- before overwriting it with P.
  float* x_mine = reinterpret_cast<float*>(sP + p_off(r, half ^ 1, 0));
  const float* x_partner = reinterpret_cast<const float*>(sP + p_off(r, half, 0));

  constexpr uint32_t kIdS = idesc<T>(kRows, BS), kIdO = idesc<T>(kRows, D);
  const float sl2 = p.scale_log2;
  float m = -INFINITY, l = 0.f;
  bool ok = true;

  for (int c = 0; c < nchunks && ok; ++c) {
    unsigned char* st = sStage;
    // K and V of this chunk landed
    ok = mbar_wait_bounded(full, c & 1, kWaitNs);
    if (!__syncthreads_and(ok)) {
      ok = false;
      break;
    }
    pend_full = -1;
    // S = Q K^T for the chunk's blocks (thread 0), at once: the S columns of TMEM were read
    // by the previous chunk's softmax, and the MMAs run in issue order after its P V
    if (tid == 0) {
      fence_after();
#pragma unroll
      for (int b = 0; b < Sh::kBlocks; ++b) {
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
          const uint64_t da = sdesc(smem_addr(sQ) + ks * 256, 128, (D / 8) * 128);
          const uint64_t db = sdesc(smem_addr(st) + b * Sh::kTile + ks * 2 * (BS * 16), BS * 16, 128);
          mma(t_s + b * BS, da, db, kIdS, ks > 0);
        }
      }
      commit(s_done);
    }
    pend_s = c;
    // the previous P V is done with V2, P and O before they are touched again
    if (c > 0) ok = mbar_wait_bounded(o_done, (c - 1) & 1, kWaitNs);
    fence_after();
    // V re-layout: piece (key group kg of 8, dim d) -> V2 + kg * (D * 16) + d * 16; keys past the sequence are zero
    for (int i = tid; i < (kKeys / 8) * D; i += kThreads) {
      const int kg = i / D, d = i - kg * D;
      const int key = c * kKeys + kg * 8;  // first key of the piece
      const int b = (kg * 8) / BS, within = (kg * 8) % BS;
      uint4 v = make_uint4(0, 0, 0, 0);
      if (key < L && c * Sh::kBlocks + b < nblk) {
        v = *reinterpret_cast<const uint4*>(st + (Sh::kBlocks + b) * Sh::kTile + d * (BS * 2) + within * 2);
        if (key + 8 > L) {  // a piece straddling the end of the sequence: zero its tail
          T* e = reinterpret_cast<T*>(&v);
#pragma unroll
          for (int j = 0; j < 8; ++j)
            if (key + j >= L) e[j] = DType<T>::from_f32(0.f);
        }
      }
      *reinterpret_cast<uint4*>(sV2 + kg * (D * 16) + d * 16) = v;
    }
    fence_proxy_async_smem();
    if (ok) ok = mbar_wait_bounded(s_done, c & 1, kWaitNs);
    if (!__syncthreads_and(ok)) {
      ok = false;
      break;
    }
    pend_s = pend_o = -1;
    fence_after();
    // the stage is free (K read by the S MMAs, V copied out): prefetch chunk c + 1 into it
    if (c + 1 < nchunks) {
      if (tid == 0) {
        fence_proxy_async_smem();
        issue(c + 1);
      }
      pend_full = c + 1;
    }
    // ---- softmax of this thread's half of the chunk's keys for its row
    float sv[kHalfKeys];
    ld32(t_s + lane_base + half * kHalfKeys, sv);
    const int lim = pos - c * kKeys - half * kHalfKeys;  // keys 0..lim of this half are visible to the row
    float mx = -INFINITY;
    if (lim >= kHalfKeys - 1) {  // all visible (every chunk but the last ones of a row)
#pragma unroll
      for (int j = 0; j < kHalfKeys; ++j) {
        sv[j] *= sl2;
        mx = fmaxf(mx, sv[j]);
      }
    } else {
#pragma unroll
      for (int j = 0; j < kHalfKeys; ++j) {
        sv[j] = j <= lim ? sv[j] * sl2 : -INFINITY;
        mx = fmaxf(mx, sv[j]);
      }
    }
    *x_mine = mx;
    // the two warps of these rows (warp and warp ^ 4) meet; the others go on
    switch (warp & 3) {  // literal barrier ids (1..4; 0 is __syncthreads)
      case 0: asm volatile("bar.sync 1, 64;" ::: "memory"); break;
      case 1: asm volatile("bar.sync 2, 64;" ::: "memory"); break;
      case 2: asm volatile("bar.sync 3, 64;" ::: "memory"); break;
      default: asm volatile("bar.sync 4, 64;" ::: "memory"); break;
    }
    mx = fmaxf(mx, *x_partner);
    // move the running maximum only when it grows by more than 2^8 (P stays <= 256)
    float corr = 1.f;
    const bool move = mx > m + 8.f;
    if (move) {
      corr = m == -INFINITY ? 0.f : exp2f(m - mx);
      m = mx;
      l *= corr;
    }
    float ps = 0.f;
#pragma unroll
    for (int kg = 0; kg < kHalfKeys / 8; ++kg) {
      uint32_t hi[4], lo[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const float x = exp2f(sv[kg * 8 + 2 * j] - m), y = exp2f(sv[kg * 8 + 2 * j + 1] - m);
        ps += x + y;
        hi[j] = pack2<T>(x, y);
        const float2 back = unpack2<T>(hi[j]);
        lo[j] = pack2<T>(x - back.x, y - back.y);
      }
      const int off = p_off(r, half, kg);
      *reinterpret_cast<uint4*>(sP + off) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
      *reinterpret_cast<uint4*>(sP + Sh::kPBytes + off) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
    }
    l += ps;
    // rescale O (idle: the previous P V is done, this one is not issued) where the maximum moved
    if (c > 0 && __any_sync(0xffffffffu, move && corr != 1.f)) {
#pragma unroll
      for (int c0 = half * kHalfD; c0 < (half + 1) * kHalfD; c0 += 32) {
        float o[32];
        ld32(t_o + lane_base + c0, o);
#pragma unroll
        for (int j = 0; j < 32; ++j) o[j] *= corr;
        st32(t_o + lane_base + c0, o);
      }
    }
    fence_proxy_async_smem();
    fence_before();
    __syncthreads();
    // O += P V (thread 0): P's high and low parts against the re-laid-out V
    if (tid == 0) {
      fence_after();
#pragma unroll
      for (int part = 0; part < 2; ++part) {
#pragma unroll
        for (int kk = 0; kk < kKeys / 16; ++kk) {
          const uint64_t da = sdesc(smem_addr(sP) + part * Sh::kPBytes + kk * 256, 128, (kKeys / 8) * 128);
          const uint64_t db = sdesc(smem_addr(sV2) + kk * 2 * (D * 16), D * 16, 128);
          mma(t_o, da, db, kIdO, c > 0 || part > 0 || kk > 0);
        }
      }
      commit(o_done);
    }
    pend_o = c;
  }

  if (ok) {
    ok = mbar_wait_bounded(o_done, (nchunks - 1) & 1, kWaitNs);
    ok = __syncthreads_and(ok);
    if (ok) pend_o = -1;
  }
  if (ok) {
    fence_after();
    // epilogue: out = O / l, rounded to T; l is the sum of the two halves' sums
    *x_mine = l;  // P is no longer read
    __syncthreads();
    const float inv = 1.f / (l + *x_partner);
    T* out = static_cast<T*>(p.out) +
             ((long long)(tok0 + (valid ? row / G : 0)) * p.num_heads + (long long)kvh * G + (valid ? row % G : 0)) * D;
#pragma unroll
    for (int c0 = half * kHalfD; c0 < (half + 1) * kHalfD; c0 += 32) {
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
  } else {
    if (tid == 0) set_error(p.err, kErrTimeout);
    // let copies and MMAs in flight finish (bounded) before the memory they target goes away
    if (pend_full >= 0) mbar_wait_bounded(full, pend_full & 1, kWaitNs / 8);
    if (pend_s >= 0) mbar_wait_bounded(s_done, pend_s & 1, kWaitNs / 8);
    if (pend_o >= 0) mbar_wait_bounded(o_done, pend_o & 1, kWaitNs / 8);
  }
  fence_before();
  __syncthreads();
  if (warp == 0) {
    fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(Sh::kTmemCols));
  }
}

}  // namespace tc
}  // namespace pa
