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
// How it maps to the GB300:
//   * Work unit = (sequence, kv head, tile of 16 query rows), the rows being the
//     chunk's (token, query head) pairs of that kv head, head fastest: a tile of
//     a GQA group holds 16 / G tokens x G heads, so each K/V byte brought in
//     serves every query head that reads it.  One warp runs one unit at a time.
//   * The unit's blocks 0 .. ceil((p_max + 1) / bs) - 1 (p_max: its last row's
//     position) stream through the warp's ring of shared-memory stages by 1-D
//     bulk copies (TMA unit), exactly like decode; the block-table row is read
//     32 entries at a time, one group ahead.
//   * Tensor cores: the 16 rows are the M side of m16n8k16 (S = Q K^T with K as
//     the B operand straight from the stage via ldmatrix; O += P V with V the
//     same way), fp32 accumulation, P split into a rounded 16-bit high part and
//     the rounded remainder.  The causal mask is per row: key t of block j is
//     kept for a row at position p when j * bs + t <= p.  V columns past p_max in
//     the unit's last block are zeroed in shared memory first (0 * NaN).
//   * Units are dealt to warps round-robin over the grid (unit = warp + k * W).
#include <math.h>

#include <type_traits>

#include "pa_device.cuh"
#include "pa_launch.h"
#include "prefill_tc.cuh"

namespace pa {

constexpr uint64_t kPrefillWaitLimitNs = 1000000000ull;
constexpr int kPrefillWarps = 8;
constexpr int kPrefillRows = 16;

template <typename T, int D, int BS>
struct PrefillShape {
  static constexpr int kTile = D * BS * 2;  // bytes of one K (or V) tile, 16-bit caches
  static constexpr int kStages = kInFlightBytes / (kPrefillWarps * 2 * kTile) > 1
                                     ? kInFlightBytes / (kPrefillWarps * 2 * kTile)
                                     : 1;
  static constexpr int kRingBytes = kPrefillWarps * kStages * 2 * kTile;
  static constexpr int kBarBytes = kPrefillWarps * kStages * 8;
  static constexpr int kTableBytes = (kMaxSeqsPerLaunch + 1) * 4 * 3 + 16 * 4;
  static constexpr int kSmem = kRingBytes + kBarBytes + kTableBytes;
};

// The per-warp math over one 16-row tile (rows = (token, head) pairs).
template <typename T, int D, int BS>
struct PrefillMath {
  static constexpr int NT = BS / 8;   // key n-tiles of S
  static constexpr int KS = D / 16;   // k-steps over head dims for S
  static constexpr int DT = D / 8;    // head-dim n-tiles of O
  static constexpr int KK = BS / 16;  // key k-steps for O

  uint32_t qf[KS][4];
  float acc[DT][4];
  float m0, m1, l0, l1;
  uint32_t k_lane_off, v_lane_off;
  int g, t4;

  __device__ __forceinline__ void init(int lane) {
    g = lane >> 2;
    t4 = lane & 3;
    const int mi = lane >> 3, mr = lane & 7;  // ldmatrix: this lane addresses row mr of matrix mi
    // K: matrix mi = (k-step half mi & 1, key n-tile mi >> 1): rows = 8 keys, 16 B = 8 dims
    k_lane_off = ((mi & 1) * BS + (mi >> 1) * 8 + mr) * 16;
    // V: matrix mi = (dims 8 (mi >> 1) .., keys 8 (mi & 1) ..): rows = 8 dims, 16 B = 8 keys
    v_lane_off = ((mi >> 1) * 8 + mr) * (BS * 2) + (mi & 1) * 16;
    for (int i = 0; i < DT; ++i) acc[i][0] = acc[i][1] = acc[i][2] = acc[i][3] = 0.f;
    m0 = m1 = -INFINITY;
    l0 = l1 = 0.f;
  }

  // A fragments of this lane's two rows (q0 / q1 point at the rows' head vectors,
  // nullptr for a padding row, which reads zeros).
  __device__ __forceinline__ void load_q(const T* q0, const T* q1) {
#pragma unroll
    for (int ks = 0; ks < KS; ++ks) {
      const int d = ks * 16 + 2 * t4, d2 = d + 8;
      qf[ks][0] = q0 ? __ldg(reinterpret_cast<const unsigned int*>(q0 + d)) : 0u;
      qf[ks][1] = q1 ? __ldg(reinterpret_cast<const unsigned int*>(q1 + d)) : 0u;
      qf[ks][2] = q0 ? __ldg(reinterpret_cast<const unsigned int*>(q0 + d2)) : 0u;
      qf[ks][3] = q1 ? __ldg(reinterpret_cast<const unsigned int*>(q1 + d2)) : 0u;
    }
  }

  // One block of BS keys; lim0 / lim1: the last key index (within this block) the
  // lane's two rows may see (negative: none).
  __device__ __forceinline__ void block(unsigned char* stage, int tile_bytes, int lim0, int lim1, float scale_log2) {
    const uint32_t kb = smem_addr(stage), vb = kb + tile_bytes;
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
    float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const int key = nt * 8 + 2 * t4 + (c & 1);
        const float v = sc[nt][c] * scale_log2;
        sc[nt][c] = key <= ((c >> 1) ? lim1 : lim0) ? v : -INFINITY;
      }
      mx0 = fmaxf(mx0, fmaxf(sc[nt][0], sc[nt][1]));
      mx1 = fmaxf(mx1, fmaxf(sc[nt][2], sc[nt][3]));
    }
    mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
    mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
    mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
    mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
    // a row with no key in this block keeps its state (its running max is finite:
    // every row sees key 0 in block 0)
    const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
    const float c0 = mn0 == -INFINITY ? 1.f : exp2f(m0 - mn0);
    const float c1 = mn1 == -INFINITY ? 1.f : exp2f(m1 - mn1);
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
        ldsm_x4(vb + v_lane_off + dp * 8 * (BS * 2) + kk * 32, b0, b1, b2, b3);
        mma_16816<T>(acc[dp], ahi, b0, b1);
        mma_16816<T>(acc[dp + 1], ahi, b2, b3);
        mma_16816<T>(acc[dp], alo, b0, b1);
        mma_16816<T>(acc[dp + 1], alo, b2, b3);
      }
    }
  }

  // out rows (o0 / o1, nullptr for padding) = acc / l, rounded to T.
  __device__ __forceinline__ void store(T* o0, T* o1) {
    l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
    l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
    l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
    l1 += __shfl_xor_sync(0xffffffffu, l1, 2);
    const float i0 = 1.f / l0, i1 = 1.f / l1;
#pragma unroll
    for (int dt = 0; dt < DT; ++dt) {
      const int d = dt * 8 + 2 * t4;
      if (o0) *reinterpret_cast<uint32_t*>(o0 + d) = pack2<T>(acc[dt][0] * i0, acc[dt][1] * i0);
      if (o1) *reinterpret_cast<uint32_t*>(o1 + d) = pack2<T>(acc[dt][2] * i1, acc[dt][3] * i1);
    }
  }
};

template <typename T, int D, int BS>
__global__ void __launch_bounds__(kPrefillWarps * 32, 1) prefill_kernel(const PrefillParams p) {
  using Sh = PrefillShape<T, D, BS>;
  constexpr int TILE = Sh::kTile, STAGES = Sh::kStages;
  extern __shared__ __align__(128) unsigned char smem[];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  unsigned char* ring = smem + warp * STAGES * 2 * TILE;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + Sh::kRingBytes) + warp * STAGES;
  int* s_L = reinterpret_cast<int*>(smem + Sh::kRingBytes + Sh::kBarBytes);  // [S] length, 0 when invalid
  int* s_n = s_L + kMaxSeqsPerLaunch + 1;                                      // [S] chunk tokens
  int* s_pre = s_n + kMaxSeqsPerLaunch + 1;                                    // [S + 1] tile prefix

  if (lane == 0) {
    for (int st = 0; st < STAGES; ++st) mbar_init(&bars[st], 1);
    fence_barrier_init();
  }
  __syncwarp();
  griddep_launch_dependents();
  griddep_wait();

  const int S = p.num_seqs, G = p.group, Hkv = p.num_kv_heads;
  // per-sequence tables (one thread; S <= kMaxSeqsPerLaunch)
  if (tid == 0) {
    int acc = 0;
    for (int s = 0; s < S; ++s) {
      int L = p.seq_lens[s];
      const int a = p.query_start_loc[s], b = p.query_start_loc[s + 1];
      int n = b - a;
      if (L < 1 || L > p.max_seq_len || a < 0 || b > p.num_query_tokens || n < 0 || n > L) {
        if (blockIdx.x == 0) set_error(p.err, kErrSeqLen);
        L = 0;
        n = 0;
      }
      s_L[s] = L;
      s_n[s] = n;
      s_pre[s] = acc;
      acc += (n * G + kPrefillRows - 1) / kPrefillRows;
    }
    s_pre[S] = acc;
  }
  __syncthreads();

  const long long units = (long long)s_pre[S] * Hkv;
  const long long W = (long long)gridDim.x * kPrefillWarps;
  PrefillMath<T, D, BS> math;
  unsigned parity = 0;  // bit st: the phase the next wait on stage st expects (the ring outlives units)
  for (long long u = (long long)blockIdx.x * kPrefillWarps + warp; u < units; u += W) {
    // unit -> (sequence, kv head, tile): the sequence with Hkv * pre[s] <= u < Hkv * pre[s + 1]
    int lo = 0, hi = S - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if ((long long)s_pre[mid] * Hkv <= u) lo = mid;
      else hi = mid - 1;
    }
    const int s = lo;
    const int tiles = s_pre[s + 1] - s_pre[s];
    const long long r0 = u - (long long)s_pre[s] * Hkv;
    const int kvh = static_cast<int>(r0 / tiles), tile = static_cast<int>(r0 - (long long)kvh * tiles);
    const int L = s_L[s], n = s_n[s], rows = n * G;
    const int row_lo = tile * kPrefillRows, row_hi = min(rows, row_lo + kPrefillRows);
    const int ctx = L - n;
    const int p_max = ctx + (row_hi - 1) / G;
    const int nblk = p_max / BS + 1;

    math.init(lane);
    // this lane's rows g and g + 8 of the tile
    const int ra = row_lo + math.g, rb = ra + 8;
    const T* q = static_cast<const T*>(p.q);
    T* out = static_cast<T*>(p.out);
    const long long tok0 = p.query_start_loc[s];
    auto row_off = [&](int r) -> long long {  // element offset of row r's head vector in q / out
      const int token = r / G, head = kvh * G + r % G;
      return ((tok0 + token) * p.num_heads + head) * (long long)D;
    };
    const bool va = ra < row_hi, vb = rb < row_hi;
    const int pa = va ? ctx + ra / G : p_max, pb = vb ? ctx + rb / G : p_max;  // padding rows act as the last
    math.load_q(va ? q + row_off(ra) : nullptr, vb ? q + row_off(rb) : nullptr);

    // block-table entries 32 at a time, one group ahead
    const int32_t* bt = p.block_tables + (long long)s * p.max_blocks_per_seq;
    int ent_cur = lane < nblk ? __ldg(bt + lane) : 0;
    int ent_nxt = 32 + lane < nblk ? __ldg(bt + 32 + lane) : 0;
    int group = 0;
    auto issue = [&](int k) {
      if ((k >> 5) != group) {
        ent_cur = ent_nxt;
        ++group;
        ent_nxt = 32 * (group + 1) + lane < nblk ? __ldg(bt + 32 * (group + 1) + lane) : 0;
      }
      int phys = __shfl_sync(0xffffffffu, ent_cur, k & 31);
      if (phys < 0 || phys >= p.num_blocks) {
        if (lane == 0) set_error(p.err, kErrBlockId);
        phys = 0;
      }
      if (lane == 0) {
        const int st = k % STAGES;
        unsigned char* dst = ring + st * 2 * TILE;
        const long long tl = (long long)phys * Hkv + kvh;
        mbar_arrive_expect_tx(&bars[st], 2 * TILE);
        bulk_copy_g2s(dst, static_cast<const unsigned char*>(p.k_cache) + tl * TILE, TILE, &bars[st]);
        bulk_copy_g2s(dst + TILE, static_cast<const unsigned char*>(p.v_cache) + tl * TILE, TILE, &bars[st]);
      }
    };
    for (int k = 0; k < STAGES && k < nblk; ++k) issue(k);
    for (int k = 0; k < nblk; ++k) {
      const int st = k % STAGES;
      const bool ok = __all_sync(0xffffffffu, mbar_wait_bounded(&bars[st], (parity >> st) & 1u, kPrefillWaitLimitNs));
      parity ^= 1u << st;
      if (!ok) {  // record it, let the copies still in flight land (bounded), stop
        if (lane == 0) set_error(p.err, kErrTimeout);
        for (int j = k + 1; j < nblk && j < k + STAGES; ++j) {
          mbar_wait_bounded(&bars[j % STAGES], (parity >> (j % STAGES)) & 1u, kPrefillWaitLimitNs / 8);
          parity ^= 1u << (j % STAGES);
        }
        return;
      }
      unsigned char* stage = ring + st * 2 * TILE;
      const int rem = p_max - k * BS + 1;  // keys of this block some row may see
      if (rem < BS) {                      // the unit's last block: zero the V columns past p_max
        T* v = reinterpret_cast<T*>(stage + TILE);
        for (int idx = lane; idx < D * BS; idx += 32)
          if ((idx % BS) >= rem) v[idx] = DType<T>::from_f32(0.f);
        __syncwarp();
      }
      math.block(stage, TILE, pa - k * BS, pb - k * BS, p.scale_log2);
      __syncwarp();
      if (k + STAGES < nblk) {
        fence_proxy_async_smem();
        issue(k + STAGES);
      }
    }
    __syncwarp();
    fence_proxy_async_smem();  // the next unit's copies land where this one's math read
    math.store(va ? out + row_off(ra) : nullptr, vb ? out + row_off(rb) : nullptr);
  }
}

// ---- host side ------------------------------------------------------------------------------

template <typename T, int D, int BS>
cudaError_t launch_prefill_t(const PrefillParams& p, cudaStream_t stream, int* launches) {
  using Sh = PrefillShape<T, D, BS>;
  *launches = 0;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  static unsigned done = 0;  // devices whose shared-memory attribute is set
  if (dev >= 32 || !(__atomic_load_n(&done, __ATOMIC_ACQUIRE) & (1u << dev))) {
    e = cudaFuncSetAttribute(reinterpret_cast<const void*>(&prefill_kernel<T, D, BS>),
                             cudaFuncAttributeMaxDynamicSharedMemorySize, Sh::kSmem);
    if (e != cudaSuccess) return e;
    if (dev < 32) __atomic_fetch_or(&done, 1u << dev, __ATOMIC_RELEASE);
  }
  int sms = 0, occ = 0;
  e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, &prefill_kernel<T, D, BS>, kPrefillWarps * 32, Sh::kSmem);
  if (e != cudaSuccess) return e;
  if (occ < 1) return cudaErrorInvalidConfiguration;
  // at most Hkv * (T G / 16 + S) units (T query tokens; each sequence adds at most one partial tile)
  const long long units = (long long)p.num_kv_heads *
                          (((long long)p.num_query_tokens * p.group + kPrefillRows - 1) / kPrefillRows + p.num_seqs);
  long long grid = (units + kPrefillWarps - 1) / kPrefillWarps;
  if (grid > (long long)sms * occ) grid = (long long)sms * occ;
  if (grid < 1) grid = 1;
  e = launch_pdl(prefill_kernel<T, D, BS>, dim3(static_cast<unsigned>(grid)), dim3(kPrefillWarps * 32), Sh::kSmem,
                 stream, p);
  if (e == cudaSuccess) *launches = 1;
  return e;
}

// The tcgen05 kernel (prefill_tc.cuh): one CTA per tile of 128 query rows.
template <typename T, int D, int BS>
cudaError_t launch_prefill_tc_t(const PrefillParams& p, cudaStream_t stream, int* launches) {
  using Sh = tc::Shape<T, D, BS>;
  *launches = 0;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  static unsigned done = 0;
  if (dev >= 32 || !(__atomic_load_n(&done, __ATOMIC_ACQUIRE) & (1u << dev))) {
    e = cudaFuncSetAttribute(reinterpret_cast<const void*>(&tc::prefill_tc_kernel<T, D, BS>),
                             cudaFuncAttributeMaxDynamicSharedMemorySize, Sh::kSmem);
    if (e != cudaSuccess) return e;
    if (dev < 32) __atomic_fetch_or(&done, 1u << dev, __ATOMIC_RELEASE);
  }
  // at most Hkv * (T G / 128 + S) tiles; CTAs past the real ones exit at once
  const long long tiles = (long long)p.num_kv_heads *
                          (((long long)p.num_query_tokens * p.group + tc::kRows - 1) / tc::kRows + p.num_seqs);
  if (tiles > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  e = launch_pdl(tc::prefill_tc_kernel<T, D, BS>, dim3(static_cast<unsigned>(tiles)), dim3(tc::kThreads), Sh::kSmem,
                 stream, p);
  if (e == cudaSuccess) *launches = 1;
  return e;
}

// tcgen05 (tensor memory) kernel, or the warp-level one above
constexpr bool kPrefillTensorMemory = true;

template <typename T, int D, int BS>
cudaError_t launch_prefill_pick(const PrefillParams& p, cudaStream_t s, int* n) {
  return kPrefillTensorMemory ? launch_prefill_tc_t<T, D, BS>(p, s, n) : launch_prefill_t<T, D, BS>(p, s, n);
}

template <typename T>
cudaError_t launch_prefill_dispatch(int head_size, int block_size, const PrefillParams& p, cudaStream_t s, int* n) {
  if (head_size == 64 && block_size == 16) return launch_prefill_pick<T, 64, 16>(p, s, n);
  if (head_size == 64 && block_size == 32) return launch_prefill_pick<T, 64, 32>(p, s, n);
  if (head_size == 128 && block_size == 16) return launch_prefill_pick<T, 128, 16>(p, s, n);
  if (head_size == 128 && block_size == 32) return launch_prefill_pick<T, 128, 32>(p, s, n);
  return cudaErrorInvalidValue;
}

cudaError_t launch_prefill(int dtype, int head_size, int block_size, const PrefillParams& p, cudaStream_t stream,
                           int* launches) {
  if (dtype == 1) return launch_prefill_dispatch<__half>(head_size, block_size, p, stream, launches);
  if (dtype == 2) return launch_prefill_dispatch<__nv_bfloat16>(head_size, block_size, p, stream, launches);
  return cudaErrorInvalidValue;
}

}  // namespace pa
