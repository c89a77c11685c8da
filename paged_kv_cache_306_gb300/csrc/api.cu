// api.cu -- the C ABI of libpa (include/pa.h): argument validation, the
// partition planner and launch dispatch.  No call allocates device memory or
// synchronizes, except pa_get_device_error.
#include <atomic>
#include <chrono>
#include <random>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>

#include "pa.h"
#include "pa_launch.h"

namespace {

// The first device-side error of the process on each device (PA_DEVERR_*).
__device__ unsigned g_device_error;

thread_local char t_message[512] = "";
std::atomic<uint64_t> g_launches{0};
std::atomic<uint64_t> g_test_wait_ns{0};  // pa_set_test_wait_limit

constexpr int kMaxDevices = 64;

pa_status fail(pa_status st, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(t_message, sizeof t_message, fmt, ap);
  va_end(ap);
  return st;
}

pa_status cuda_fail(cudaError_t e, const char* what) {
  return fail(PA_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

// Device address of g_device_error on the current device (looked up once per device).
pa_status device_error_ptr(unsigned** out) {
  static std::mutex mu;
  static unsigned* ptrs[kMaxDevices] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev < 0 || dev >= kMaxDevices) return fail(PA_ERR_UNSUPPORTED, "device ordinal %d too large", dev);
  std::lock_guard<std::mutex> lock(mu);
  if (!ptrs[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_device_error);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress");
    ptrs[dev] = static_cast<unsigned*>(p);
  }
  *out = ptrs[dev];
  return PA_OK;
}

int sm_count() {
  static std::atomic<int> cache[kMaxDevices];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 0;
  int n = cache[dev].load(std::memory_order_relaxed);
  if (n > 0) return n;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  cache[dev].store(n, std::memory_order_relaxed);
  return n;
}

int elem_bytes(pa_dtype d) {
  return d == PA_F32 ? 4 : (d == PA_F16 || d == PA_BF16) ? 2 : d == PA_FP8_E4M3 ? 1 : 0;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

int ceil_div(long long a, long long b) { return static_cast<int>((a + b - 1) / b); }

// Shape checks shared by the planner, the workspace query and pa_decode.
pa_status check_decode_shape(int num_seqs, int num_heads, int num_kv_heads, int head_size, int max_seq_len,
                             int block_size, pa_dtype dtype) {
  if (!elem_bytes(dtype)) return fail(PA_ERR_INVALID_ARG, "unknown dtype %d", static_cast<int>(dtype));
  if (num_seqs < 0 || num_seqs > 65535) return fail(PA_ERR_INVALID_ARG, "num_seqs %d outside [0, 65535]", num_seqs);
  if (num_heads < 1 || num_kv_heads < 1 || num_heads % num_kv_heads)
    return fail(PA_ERR_INVALID_ARG, "num_heads %d must be a positive multiple of num_kv_heads %d", num_heads,
                num_kv_heads);
  if (num_heads > 65535) return fail(PA_ERR_UNSUPPORTED, "num_heads %d > 65535", num_heads);
  if (head_size != 64 && head_size != 128) return fail(PA_ERR_UNSUPPORTED, "head_size %d not in {64, 128}", head_size);
  if (block_size != 16 && block_size != 32)
    return fail(PA_ERR_UNSUPPORTED, "block_size %d not in {16, 32}", block_size);
  if (max_seq_len < 1) return fail(PA_ERR_INVALID_ARG, "max_seq_len %d < 1", max_seq_len);
  return PA_OK;
}

// How one pa_decode call is cut into launches and how its workspace is laid out.
struct DecodePlan {
  pa::DecodeKind kind;
  int units;         // head units per sequence
  int rows;          // query rows per partial-result slot
  int part_blocks;   // caller partition in blocks (a huge value when none)
  int chunk;         // sequences per launch
  int grid;          // CTAs of the main kernel (all resident)
  int members;       // sequences per shared-prefix cluster; 0: no shared prefixes
  long long slots;   // partial-result slots
  size_t off_tag, off_ml, off_o, off_first, off_last, off_info, bytes;
};

// Shared prefixes pay off where the tensor-core tile has room for the query heads
// of several sequences.  16-bit caches: clusters fill the 16 columns of two 8-head
// tiles (at most 8 query heads per kv head).  FP8 caches: one 8-head tile, which
// keeps their 16-warp kernel (the widening of the codes needs the warps); at most
// 4 query heads per kv head.  Elsewhere the shared-prefix call runs the plain
// schedule.
int shared_members(pa_dtype dtype, int num_heads, int num_kv_heads) {
  const int group = num_heads / num_kv_heads;
  const int cols = dtype == PA_FP8_E4M3 ? 8 : 16;
  if (dtype == PA_F32 || 2 * group > cols) return 0;
  return cols / group;
}

size_t align256(size_t x) { return (x + 255) / 256 * 256; }

// The schedule: the main kernel runs exactly the CTAs that fit on the GPU at once
// (fewer for small batches, so that every warp gets a few blocks); each warp takes
// an equal share of all blocks of the launch.  A launch covers at most
// kMaxSeqsPerLaunch sequences.  Partial slots: one per warp plus one per segment,
// the most pieces a launch can leave (pieces start at warp or segment boundaries).
pa_status make_plan(int num_seqs, int num_heads, int num_kv_heads, int head_size, int max_seq_len, int block_size,
                    int partition_size, pa_dtype dtype, DecodePlan* pl, bool shared = false) {
  const int group = num_heads / num_kv_heads;
  pl->members = shared ? shared_members(dtype, num_heads, num_kv_heads) : 0;
  if (pl->members && (max_seq_len + block_size - 1) / block_size >= (1 << pa::kInfoOffBits))
    return fail(PA_ERR_UNSUPPORTED, "shared prefixes: at most %d blocks per sequence", (1 << pa::kInfoOffBits) - 1);
  pl->kind = pl->members ? (dtype == PA_FP8_E4M3 ? pa::DecodeKind::kMma8 : pa::DecodeKind::kMma16)
                         : pa::decode_kind(static_cast<int>(dtype), group);
  pl->units = pa::decode_units(pl->kind, num_heads, num_kv_heads);
  pl->rows = pl->members ? (dtype == PA_FP8_E4M3 ? 8 : 16) : pa::decode_rows(pl->kind, num_heads, num_kv_heads);
  const int nblk_max = ceil_div(max_seq_len, block_size);
  pl->part_blocks = partition_size > 0 ? partition_size / block_size : (1 << 30);
  long long chunk = num_seqs < pa::kMaxSeqsPerLaunch ? num_seqs : pa::kMaxSeqsPerLaunch;
  // the schedule's cost prefix per unit stays within int32 (see pa::kSegCost)
  const long long unit_cost = (long long)pa::kSharedCost * nblk_max + 2 * pa::kSegCost;
  if (chunk > 0x7fffffffLL / unit_cost) chunk = 0x7fffffffLL / unit_cost;
  if (chunk < 1) chunk = 1;
  pl->chunk = static_cast<int>(chunk);
  const int ctas = pa::decode_ctas_per_sm(static_cast<int>(dtype), head_size, block_size, pl->kind);
  const int sms = sm_count();
  if (ctas <= 0 || sms <= 0) return fail(PA_ERR_CUDA, "cannot query the device (SM count %d, CTAs per SM %d)", sms, ctas);
  const int warps = pa::decode_warps_for(elem_bytes(dtype), head_size, block_size, pl->kind);
  const long long work = chunk * pl->units * (long long)nblk_max;
  long long grid = (work + 4 * warps - 1) / (4 * warps);
  if (grid > (long long)sms * ctas) grid = (long long)sms * ctas;
  if (grid < 1) grid = 1;
  pl->grid = static_cast<int>(grid);
  // segments: one per (sequence, unit); with shared prefixes two (shared part, own part)
  const long long segs = chunk * pl->units * (pl->members ? 2 : 1);
  pl->slots = grid * warps + segs;
  if (pl->slots > 0x7fffffffLL || segs > 0x7fffffffLL)
    return fail(PA_ERR_UNSUPPORTED, "too many partial results (%lld); use a larger partition_size", pl->slots);
  size_t off = 0;
  pl->off_tag = off;
  off = align256(off + (size_t)pl->slots * 8);
  pl->off_ml = off;
  off = align256(off + (size_t)pl->slots * pl->rows * 2 * sizeof(float));
  pl->off_o = off;
  off = align256(off + (size_t)pl->slots * pl->rows * head_size * sizeof(float));
  pl->off_first = off;
  off = align256(off + (size_t)segs * sizeof(int));
  pl->off_last = off;
  off = align256(off + (size_t)segs * sizeof(int));
  pl->off_info = off;
  if (pl->members) off = align256(off + (size_t)chunk * 2 * sizeof(int));
  pl->bytes = off;
  return PA_OK;
}

// A fresh tag for every launch, so a launch never mistakes a partial slot left by
// an earlier launch for its own.  The sequence starts at a random point, so tags
// left in a reused buffer by another process are as unlikely to match.  Zero is
// never used.
unsigned next_epoch() {
  static std::atomic<unsigned> epoch{static_cast<unsigned>(std::random_device{}()) ^
                                     static_cast<unsigned>(std::chrono::steady_clock::now().time_since_epoch().count())};
  unsigned e = epoch.fetch_add(1, std::memory_order_relaxed) + 1;
  if (e == 0) e = epoch.fetch_add(1, std::memory_order_relaxed) + 1;
  return e;
}

}  // namespace

namespace pa {

// Record a failure with a message for pa_last_error_message (used by other
// translation units of the library).
pa_status record_failure(pa_status st, const char* message) { return fail(st, "%s", message); }

int decode_ctas_per_sm(int dtype, int head_size, int block_size, DecodeKind kind) {
  switch (dtype) {
    case PA_F32: return decode_ctas_per_sm_f32(head_size, block_size, kind);
    case PA_F16: return decode_ctas_per_sm_f16(head_size, block_size, kind);
    case PA_BF16: return decode_ctas_per_sm_bf16(head_size, block_size, kind);
    case PA_FP8_E4M3: return decode_ctas_per_sm_fp8(false, head_size, block_size, kind);
    default: return 0;
  }
}

cudaError_t launch_decode(int dtype, int head_size, int block_size, const DecodeParams& p, DecodeKind kind, int grid,
                          cudaStream_t stream, int* launches) {
  // dtype: the cache dtype for 16-bit and fp32 caches (the query's too); for an
  // FP8 cache, 16 + the query dtype (see decode_impl)
  if (dtype >= 16)
    return launch_decode_fp8(dtype - 16 == PA_BF16, head_size, block_size, p, kind, grid, stream, launches);
  switch (dtype) {
    case PA_F32: return launch_decode_f32(head_size, block_size, p, kind, grid, stream, launches);
    case PA_F16: return launch_decode_f16(head_size, block_size, p, kind, grid, stream, launches);
    case PA_BF16: return launch_decode_bf16(head_size, block_size, p, kind, grid, stream, launches);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace pa

extern "C" {

const char* pa_status_string(pa_status s) {
  switch (s) {
    case PA_OK: return "PA_OK";
    case PA_ERR_INVALID_ARG: return "PA_ERR_INVALID_ARG";
    case PA_ERR_UNSUPPORTED: return "PA_ERR_UNSUPPORTED";
    case PA_ERR_ALIGNMENT: return "PA_ERR_ALIGNMENT";
    case PA_ERR_WORKSPACE: return "PA_ERR_WORKSPACE";
    case PA_ERR_CUDA: return "PA_ERR_CUDA";
    case PA_ERR_OUT_OF_BLOCKS: return "PA_ERR_OUT_OF_BLOCKS";
    default: return "PA_ERR_UNKNOWN";
  }
}

const char* pa_last_error_message(void) { return t_message; }

uint64_t pa_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

void pa_set_test_wait_limit(uint64_t nanoseconds) { g_test_wait_ns.store(nanoseconds, std::memory_order_relaxed); }

pa_status pa_reshape_and_cache(const void* key, const void* value, void* k_cache, void* v_cache,
                               const int64_t* slot_mapping, int64_t num_tokens, int num_kv_heads, int head_size,
                               int block_size, int64_t num_blocks, pa_dtype dtype, void* stream) {
  const int e = elem_bytes(dtype);
  if (!e) return fail(PA_ERR_INVALID_ARG, "unknown dtype %d", static_cast<int>(dtype));
  if (num_tokens < 0 || num_tokens > 0x7fffffffLL) return fail(PA_ERR_INVALID_ARG, "num_tokens %lld", (long long)num_tokens);
  if (num_kv_heads < 1 || head_size < 1 || block_size < 1 || num_blocks < 1)
    return fail(PA_ERR_INVALID_ARG, "num_kv_heads, head_size, block_size and num_blocks must be positive");
  if (num_kv_heads > 65535) return fail(PA_ERR_UNSUPPORTED, "num_kv_heads %d > 65535", num_kv_heads);
  if (head_size % (16 / e)) return fail(PA_ERR_INVALID_ARG, "head_size %d not a multiple of x = %d", head_size, 16 / e);
  if (num_tokens == 0) return PA_OK;
  if (!key || !value || !k_cache || !v_cache || !slot_mapping) return fail(PA_ERR_INVALID_ARG, "null pointer");
  if (!aligned(key, 16) || !aligned(value, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) ||
      !aligned(slot_mapping, 8))
    return fail(PA_ERR_ALIGNMENT, "key/value/caches need 16-byte, slot_mapping 8-byte alignment");
  unsigned* err = nullptr;
  pa_status st = device_error_ptr(&err);
  if (st != PA_OK) return st;
  int n = 0;
  cudaError_t ce = pa::launch_reshape_and_cache(key, value, k_cache, v_cache, slot_mapping, num_tokens, num_kv_heads,
                                                head_size, block_size, num_blocks, e, err,
                                                static_cast<cudaStream_t>(stream), &n);
  g_launches.fetch_add(n, std::memory_order_relaxed);
  return ce == cudaSuccess ? PA_OK : cuda_fail(ce, "reshape_and_cache launch");
}

pa_status pa_reshape_and_cache_scaled(const void* key, const void* value, void* k_cache, void* v_cache,
                                      const int64_t* slot_mapping, int64_t num_tokens, int num_kv_heads, int head_size,
                                      int block_size, int64_t num_blocks, pa_dtype key_dtype, pa_dtype cache_dtype,
                                      float k_scale, float v_scale, void* stream) {
  if (cache_dtype != PA_FP8_E4M3) {
    if (key_dtype != cache_dtype || k_scale != 1.f || v_scale != 1.f)
      return fail(PA_ERR_INVALID_ARG, "a %s cache stores key/value as they are: same dtype, scales 1",
                  cache_dtype == PA_F32 ? "fp32" : "16-bit");
    return pa_reshape_and_cache(key, value, k_cache, v_cache, slot_mapping, num_tokens, num_kv_heads, head_size,
                                block_size, num_blocks, cache_dtype, stream);
  }
  if (key_dtype != PA_F32 && key_dtype != PA_F16 && key_dtype != PA_BF16)
    return fail(PA_ERR_UNSUPPORTED, "an FP8 cache is written from fp32, fp16 or bf16 key/value");
  if (!(k_scale > 0.f) || !(v_scale > 0.f) || !std::isfinite(k_scale) || !std::isfinite(v_scale))
    return fail(PA_ERR_INVALID_ARG, "k_scale and v_scale must be positive and finite");
  if (num_tokens < 0 || num_tokens > 0x7fffffffLL) return fail(PA_ERR_INVALID_ARG, "num_tokens %lld", (long long)num_tokens);
  if (num_kv_heads < 1 || head_size < 1 || block_size < 1 || num_blocks < 1)
    return fail(PA_ERR_INVALID_ARG, "num_kv_heads, head_size, block_size and num_blocks must be positive");
  if (num_kv_heads > 65535) return fail(PA_ERR_UNSUPPORTED, "num_kv_heads %d > 65535", num_kv_heads);
  if (head_size % 16) return fail(PA_ERR_INVALID_ARG, "head_size %d not a multiple of 16", head_size);
  if (num_tokens == 0) return PA_OK;
  if (!key || !value || !k_cache || !v_cache || !slot_mapping) return fail(PA_ERR_INVALID_ARG, "null pointer");
  if (!aligned(key, 16) || !aligned(value, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) ||
      !aligned(slot_mapping, 8))
    return fail(PA_ERR_ALIGNMENT, "key/value/caches need 16-byte, slot_mapping 8-byte alignment");
  unsigned* err = nullptr;
  pa_status st = device_error_ptr(&err);
  if (st != PA_OK) return st;
  int n = 0;
  cudaError_t ce = pa::launch_reshape_and_cache_e4m3(key, value, k_cache, v_cache, slot_mapping, num_tokens,
                                                     num_kv_heads, head_size, block_size, num_blocks,
                                                     static_cast<int>(key_dtype), k_scale, v_scale, err,
                                                     static_cast<cudaStream_t>(stream), &n);
  g_launches.fetch_add(n, std::memory_order_relaxed);
  return ce == cudaSuccess ? PA_OK : cuda_fail(ce, "quantising reshape_and_cache launch");
}

pa_status pa_copy_blocks(void* k_cache, void* v_cache, const int64_t* src_dst, int64_t num_pairs, int num_kv_heads,
                         int head_size, int block_size, int64_t num_blocks, pa_dtype dtype, void* stream) {
  const int e = elem_bytes(dtype);
  if (!e) return fail(PA_ERR_INVALID_ARG, "unknown dtype %d", static_cast<int>(dtype));
  if (num_pairs < 0 || num_pairs > 0x7fffffffLL) return fail(PA_ERR_INVALID_ARG, "num_pairs %lld", (long long)num_pairs);
  if (num_kv_heads < 1 || head_size < 1 || block_size < 1 || num_blocks < 1)
    return fail(PA_ERR_INVALID_ARG, "num_kv_heads, head_size, block_size and num_blocks must be positive");
  if (num_kv_heads > 65535) return fail(PA_ERR_UNSUPPORTED, "num_kv_heads %d > 65535", num_kv_heads);
  const long long block_bytes = (long long)num_kv_heads * head_size * block_size * e;
  if (block_bytes % 16) return fail(PA_ERR_INVALID_ARG, "a block of %lld bytes is not a multiple of 16", block_bytes);
  if (num_pairs == 0) return PA_OK;
  if (!k_cache || !v_cache || !src_dst) return fail(PA_ERR_INVALID_ARG, "null pointer");
  if (!aligned(k_cache, 16) || !aligned(v_cache, 16) || !aligned(src_dst, 8))
    return fail(PA_ERR_ALIGNMENT, "caches need 16-byte, src_dst 8-byte alignment");
  unsigned* err = nullptr;
  pa_status st = device_error_ptr(&err);
  if (st != PA_OK) return st;
  int n = 0;
  cudaError_t ce = pa::launch_copy_blocks(k_cache, v_cache, src_dst, num_pairs, block_bytes, num_blocks, err,
                                          static_cast<cudaStream_t>(stream), &n);
  g_launches.fetch_add(n, std::memory_order_relaxed);
  return ce == cudaSuccess ? PA_OK : cuda_fail(ce, "copy_blocks launch");
}

int pa_decode_plan_partition(int num_seqs, int num_heads, int num_kv_heads, int head_size, int max_seq_len,
                             int block_size, pa_dtype dtype) {
  if (check_decode_shape(num_seqs, num_heads, num_kv_heads, head_size, max_seq_len, block_size, dtype) != PA_OK)
    return -1;
  // The load-balanced schedule needs no caller partitions: every warp already gets
  // an equal share of the blocks, and long sequences are split wherever that falls.
  return PA_PARTITION_NONE;
}

size_t pa_decode_workspace_size(int num_seqs, int num_heads, int num_kv_heads, int head_size, int max_seq_len,
                                int block_size, int partition_size, pa_dtype dtype) {
  if (check_decode_shape(num_seqs, num_heads, num_kv_heads, head_size, max_seq_len, block_size, dtype) != PA_OK)
    return 0;
  if (partition_size == PA_PARTITION_AUTO) partition_size = PA_PARTITION_NONE;
  if (partition_size < 0 || (partition_size > 0 && partition_size % block_size) || num_seqs == 0) return 0;
  DecodePlan pl;
  if (make_plan(num_seqs, num_heads, num_kv_heads, head_size, max_seq_len, block_size, partition_size, dtype, &pl) !=
      PA_OK)
    return 0;
  return pl.bytes;
}

static pa_status decode_impl(void* out, const void* q, const void* k_cache, const void* v_cache,
                             const int32_t* block_tables, int max_blocks_per_seq, const int32_t* seq_lens,
                             int num_seqs, int max_seq_len, int num_heads, int num_kv_heads, int head_size,
                             int block_size, int64_t num_blocks, float scale, int partition_size, void* workspace,
                             size_t workspace_bytes, pa_dtype q_dtype, pa_dtype dtype, float k_scale, float v_scale,
                             void* stream, const void* new_key = nullptr, const void* new_value = nullptr,
                             const int64_t* copy_pairs = nullptr, int64_t num_copies = 0,
                             const int32_t* prefix_group = nullptr, const int32_t* prefix_blocks = nullptr) {
  // new_key != nullptr: the fused step (pa_decode_step), already validated there.
  // `dtype` is the cache dtype from here on; q and out have q_dtype.
  pa_status st = check_decode_shape(num_seqs, num_heads, num_kv_heads, head_size, max_seq_len, block_size, dtype);
  if (st != PA_OK) return st;
  if (dtype == PA_FP8_E4M3) {
    if (q_dtype != PA_F16 && q_dtype != PA_BF16)
      return fail(PA_ERR_UNSUPPORTED, "an FP8 cache is read by fp16 or bf16 queries");
    if (!(k_scale > 0.f) || !(v_scale > 0.f) || !std::isfinite(k_scale) || !std::isfinite(v_scale))
      return fail(PA_ERR_INVALID_ARG, "k_scale and v_scale must be positive and finite");
  } else if (q_dtype != dtype || k_scale != 1.f || v_scale != 1.f) {
    return fail(PA_ERR_INVALID_ARG, "a 16-bit or fp32 cache is read by queries of its own dtype with scales 1");
  }
  if (max_blocks_per_seq < 1 || (long long)max_seq_len > (long long)max_blocks_per_seq * block_size)
    return fail(PA_ERR_INVALID_ARG, "max_seq_len %d exceeds max_blocks_per_seq %d * block_size %d", max_seq_len,
                max_blocks_per_seq, block_size);
  if (num_blocks < 1) return fail(PA_ERR_INVALID_ARG, "num_blocks %lld < 1", (long long)num_blocks);
  if (!std::isfinite(scale)) return fail(PA_ERR_INVALID_ARG, "scale is not finite");
  if (partition_size == PA_PARTITION_AUTO) partition_size = PA_PARTITION_NONE;
  if (partition_size < 0 || (partition_size > 0 && partition_size % block_size))
    return fail(PA_ERR_INVALID_ARG, "partition_size %d must be NONE, AUTO or a positive multiple of block_size %d",
                partition_size, block_size);
  if (num_seqs == 0) return PA_OK;
  if (!out || !q || !k_cache || !v_cache || !block_tables || !seq_lens) return fail(PA_ERR_INVALID_ARG, "null pointer");
  if (!aligned(out, 16) || !aligned(q, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) ||
      !aligned(block_tables, 4) || !aligned(seq_lens, 4))
    return fail(PA_ERR_ALIGNMENT, "q/out/caches need 16-byte, block_tables/seq_lens 4-byte alignment");

  if (prefix_group && (!aligned(prefix_group, 4) || !aligned(prefix_blocks, 4)))
    return fail(PA_ERR_ALIGNMENT, "prefix_group and prefix_blocks need 4-byte alignment");
  DecodePlan pl;
  st = make_plan(num_seqs, num_heads, num_kv_heads, head_size, max_seq_len, block_size, partition_size, dtype, &pl,
                 prefix_group != nullptr);
  if (st != PA_OK) return st;
  if (!workspace || workspace_bytes < pl.bytes)
    return fail(PA_ERR_WORKSPACE, "workspace of %zu bytes needed, %zu given", pl.bytes, workspace ? workspace_bytes : 0);
  if (!aligned(workspace, 16)) return fail(PA_ERR_ALIGNMENT, "workspace needs 16-byte alignment");

  pa::DecodeParams p{};
  char* ws = static_cast<char*>(workspace);
  p.part_tag = reinterpret_cast<int2*>(ws + pl.off_tag);
  p.part_ml = reinterpret_cast<float*>(ws + pl.off_ml);
  p.part_o = reinterpret_cast<float*>(ws + pl.off_o);
  p.seg_first = reinterpret_cast<int*>(ws + pl.off_first);
  p.seg_last = reinterpret_cast<int*>(ws + pl.off_last);
  p.seq_info = reinterpret_cast<int*>(ws + pl.off_info);
  p.shared = pl.members > 0;
  p.members = pl.members;
  p.fused = new_key != nullptr;
  p.write_k_scale = k_scale;
  p.write_v_scale = v_scale;
  st = device_error_ptr(&p.err);
  if (st != PA_OK) return st;
  p.k_cache = k_cache;
  p.v_cache = v_cache;
  p.num_blocks = num_blocks;
  p.max_blocks_per_seq = max_blocks_per_seq;
  p.num_heads = num_heads;
  p.num_kv_heads = num_kv_heads;
  p.group = num_heads / num_kv_heads;
  p.units = pl.units;
  p.rows = pl.rows;
  p.max_seq_len = max_seq_len;
  p.part_blocks = pl.part_blocks;
  p.num_slots = static_cast<int>(pl.slots);
  p.scale_log2 = static_cast<float>(static_cast<double>(scale) * k_scale * 1.4426950408889634);
  p.out_scale = v_scale;
  p.test_wait_ns = g_test_wait_ns.load(std::memory_order_relaxed);

  if (p.fused && num_copies > 0) {  // the copy-on-write copies: their own kernel, before any token lands
    int n = 0;
    const long long block_bytes = (long long)num_kv_heads * head_size * block_size * elem_bytes(dtype);
    const cudaError_t ce = pa::launch_copy_blocks(const_cast<void*>(k_cache), const_cast<void*>(v_cache), copy_pairs,
                                                  num_copies, block_bytes, num_blocks, p.err,
                                                  static_cast<cudaStream_t>(stream), &n);
    g_launches.fetch_add(n, std::memory_order_relaxed);
    if (ce != cudaSuccess) return cuda_fail(ce, "copy_blocks launch");
  }
  const size_t row_bytes = (size_t)num_heads * head_size * elem_bytes(q_dtype);
  const int launch_dtype = dtype == PA_FP8_E4M3 ? 16 + static_cast<int>(q_dtype) : static_cast<int>(dtype);
  for (int c0 = 0; c0 < num_seqs; c0 += pl.chunk) {
    p.num_seqs = num_seqs - c0 < pl.chunk ? num_seqs - c0 : pl.chunk;
    p.q = static_cast<const char*>(q) + (size_t)c0 * row_bytes;
    p.out = static_cast<char*>(out) + (size_t)c0 * row_bytes;
    p.block_tables = block_tables + (size_t)c0 * max_blocks_per_seq;
    p.seq_lens = seq_lens + c0;
    // a chunk's first sequence starts a cluster: its link to the previous chunk is not read
    p.prefix_group = p.shared ? prefix_group + c0 : nullptr;
    p.prefix_blocks = p.shared ? prefix_blocks + c0 : nullptr;
    if (p.fused) {  // the new rows come in the query dtype (an FP8 pool quantises them itself)
      const size_t kv_row_bytes = (size_t)num_kv_heads * head_size * elem_bytes(q_dtype);
      p.new_key = static_cast<const char*>(new_key) + (size_t)c0 * kv_row_bytes;
      p.new_value = static_cast<const char*>(new_value) + (size_t)c0 * kv_row_bytes;
    }
    p.epoch = next_epoch();
    int n = 0;
    const cudaError_t ce = pa::launch_decode(launch_dtype, head_size, block_size, p, pl.kind, pl.grid,
                                             static_cast<cudaStream_t>(stream), &n);
    g_launches.fetch_add(n, std::memory_order_relaxed);
    if (ce != cudaSuccess) return cuda_fail(ce, "decode launch");
  }
  return PA_OK;
}

pa_status pa_decode(void* out, const void* q, const void* k_cache, const void* v_cache, const int32_t* block_tables,
                    int max_blocks_per_seq, const int32_t* seq_lens, int num_seqs, int max_seq_len, int num_heads,
                    int num_kv_heads, int head_size, int block_size, int64_t num_blocks, float scale,
                    int partition_size, void* workspace, size_t workspace_bytes, pa_dtype dtype, void* stream) {
  if (dtype == PA_FP8_E4M3)
    return fail(PA_ERR_UNSUPPORTED, "an FP8 cache needs pa_decode_scaled (query dtype and k/v scales)");
  return decode_impl(out, q, k_cache, v_cache, block_tables, max_blocks_per_seq, seq_lens, num_seqs, max_seq_len,
                     num_heads, num_kv_heads, head_size, block_size, num_blocks, scale, partition_size, workspace,
                     workspace_bytes, dtype, dtype, 1.f, 1.f, stream);
}

pa_status pa_decode_scaled(void* out, const void* q, const void* k_cache, const void* v_cache,
                           const int32_t* block_tables, int max_blocks_per_seq, const int32_t* seq_lens, int num_seqs,
                           int max_seq_len, int num_heads, int num_kv_heads, int head_size, int block_size,
                           int64_t num_blocks, float scale, int partition_size, void* workspace,
                           size_t workspace_bytes, pa_dtype q_dtype, pa_dtype cache_dtype, float k_scale,
                           float v_scale, void* stream) {
  if (!elem_bytes(q_dtype)) return fail(PA_ERR_INVALID_ARG, "unknown query dtype %d", static_cast<int>(q_dtype));
  return decode_impl(out, q, k_cache, v_cache, block_tables, max_blocks_per_seq, seq_lens, num_seqs, max_seq_len,
                     num_heads, num_kv_heads, head_size, block_size, num_blocks, scale, partition_size, workspace,
                     workspace_bytes, q_dtype, cache_dtype, k_scale, v_scale, stream);
}

pa_status pa_decode_step_scaled(void* out, const void* q, const void* key, const void* value, void* k_cache,
                                void* v_cache, const int64_t* src_dst, int64_t num_pairs,
                                const int32_t* block_tables, int max_blocks_per_seq, const int32_t* seq_lens,
                                int num_seqs, int max_seq_len, int num_heads, int num_kv_heads, int head_size,
                                int block_size, int64_t num_blocks, float scale, int partition_size,
                                void* workspace, size_t workspace_bytes, pa_dtype q_dtype, pa_dtype cache_dtype,
                                float k_scale, float v_scale, void* stream) {
  if (cache_dtype != PA_F32 && cache_dtype != PA_F16 && cache_dtype != PA_BF16 && cache_dtype != PA_FP8_E4M3)
    return fail(PA_ERR_UNSUPPORTED, "unknown cache dtype %d", static_cast<int>(cache_dtype));
  if (!elem_bytes(q_dtype)) return fail(PA_ERR_INVALID_ARG, "unknown query dtype %d", static_cast<int>(q_dtype));
  if (num_pairs < 0 || num_pairs > 0x7fffffffLL) return fail(PA_ERR_INVALID_ARG, "num_pairs %lld", (long long)num_pairs);
  if (num_pairs > 0 && (!src_dst || !aligned(src_dst, 8)))
    return fail(num_pairs > 0 && src_dst ? PA_ERR_ALIGNMENT : PA_ERR_INVALID_ARG,
                "src_dst must be a non-null, 8-byte aligned int64 array");
  if (num_seqs > 0 && (!key || !value)) return fail(PA_ERR_INVALID_ARG, "null key or value");
  if (num_seqs > 0 && (!aligned(key, 16) || !aligned(value, 16)))
    return fail(PA_ERR_ALIGNMENT, "key/value need 16-byte alignment");
  if (num_seqs == 0 && num_pairs > 0)  // nothing to decode: the copies alone
    return pa_copy_blocks(k_cache, v_cache, src_dst, num_pairs, num_kv_heads, head_size, block_size, num_blocks,
                          cache_dtype, stream);
  return decode_impl(out, q, k_cache, v_cache, block_tables, max_blocks_per_seq, seq_lens, num_seqs, max_seq_len,
                     num_heads, num_kv_heads, head_size, block_size, num_blocks, scale, partition_size, workspace,
                     workspace_bytes, q_dtype, cache_dtype, k_scale, v_scale, stream, key, value, src_dst, num_pairs);
}

pa_status pa_decode_step(void* out, const void* q, const void* key, const void* value, void* k_cache, void* v_cache,
                         const int64_t* src_dst, int64_t num_pairs, const int32_t* block_tables,
                         int max_blocks_per_seq, const int32_t* seq_lens, int num_seqs, int max_seq_len,
                         int num_heads, int num_kv_heads, int head_size, int block_size, int64_t num_blocks,
                         float scale, int partition_size, void* workspace, size_t workspace_bytes, pa_dtype dtype,
                         void* stream) {
  if (dtype != PA_F32 && dtype != PA_F16 && dtype != PA_BF16)
    return fail(PA_ERR_UNSUPPORTED, "the fused step on an FP8 cache is pa_decode_step_scaled (query dtype, scales)");
  return pa_decode_step_scaled(out, q, key, value, k_cache, v_cache, src_dst, num_pairs, block_tables,
                               max_blocks_per_seq, seq_lens, num_seqs, max_seq_len, num_heads, num_kv_heads, head_size,
                               block_size, num_blocks, scale, partition_size, workspace, workspace_bytes, dtype, dtype,
                               1.f, 1.f, stream);
}

size_t pa_decode_shared_workspace_size(int num_seqs, int num_heads, int num_kv_heads, int head_size, int max_seq_len,
                                       int block_size, int partition_size, pa_dtype cache_dtype) {
  if (check_decode_shape(num_seqs, num_heads, num_kv_heads, head_size, max_seq_len, block_size, cache_dtype) != PA_OK)
    return 0;
  if (partition_size == PA_PARTITION_AUTO) partition_size = PA_PARTITION_NONE;
  if (partition_size < 0 || (partition_size > 0 && partition_size % block_size) || num_seqs == 0) return 0;
  DecodePlan pl;
  if (make_plan(num_seqs, num_heads, num_kv_heads, head_size, max_seq_len, block_size, partition_size, cache_dtype,
                &pl, true) != PA_OK)
    return 0;
  return pl.bytes;
}

pa_status pa_decode_shared(void* out, const void* q, const void* key, const void* value, void* k_cache,
                           void* v_cache, const int64_t* src_dst, int64_t num_pairs, const int32_t* block_tables,
                           int max_blocks_per_seq, const int32_t* seq_lens, const int32_t* prefix_group,
                           const int32_t* prefix_blocks, int num_seqs, int max_seq_len, int num_heads,
                           int num_kv_heads, int head_size, int block_size, int64_t num_blocks, float scale,
                           int partition_size, void* workspace, size_t workspace_bytes, pa_dtype q_dtype,
                           pa_dtype cache_dtype, float k_scale, float v_scale, void* stream) {
  if (cache_dtype != PA_F32 && cache_dtype != PA_F16 && cache_dtype != PA_BF16 && cache_dtype != PA_FP8_E4M3)
    return fail(PA_ERR_UNSUPPORTED, "unknown cache dtype %d", static_cast<int>(cache_dtype));
  if (!elem_bytes(q_dtype)) return fail(PA_ERR_INVALID_ARG, "unknown query dtype %d", static_cast<int>(q_dtype));
  if (num_seqs > 0 && (!prefix_group || !prefix_blocks))
    return fail(PA_ERR_INVALID_ARG, "null prefix_group or prefix_blocks");
  if ((key == nullptr) != (value == nullptr)) return fail(PA_ERR_INVALID_ARG, "key and value: both or neither");
  if (num_pairs < 0 || num_pairs > 0x7fffffffLL) return fail(PA_ERR_INVALID_ARG, "num_pairs %lld", (long long)num_pairs);
  if (num_pairs > 0 && (!src_dst || !aligned(src_dst, 8)))
    return fail(src_dst ? PA_ERR_ALIGNMENT : PA_ERR_INVALID_ARG, "src_dst must be a non-null, 8-byte aligned int64 array");
  if (num_pairs > 0 && !key) return fail(PA_ERR_INVALID_ARG, "block copies come with the step's new tokens");
  if (key && (!aligned(key, 16) || !aligned(value, 16))) return fail(PA_ERR_ALIGNMENT, "key/value need 16-byte alignment");
  if (num_seqs == 0 && num_pairs > 0)  // nothing to decode: the copies alone
    return pa_copy_blocks(k_cache, v_cache, src_dst, num_pairs, num_kv_heads, head_size, block_size, num_blocks,
                          cache_dtype, stream);
  return decode_impl(out, q, k_cache, v_cache, block_tables, max_blocks_per_seq, seq_lens, num_seqs, max_seq_len,
                     num_heads, num_kv_heads, head_size, block_size, num_blocks, scale, partition_size, workspace,
                     workspace_bytes, q_dtype, cache_dtype, k_scale, v_scale, stream, key, value, src_dst, num_pairs,
                     prefix_group, prefix_blocks);
}

pa_status pa_prefill(void* out, const void* q, const void* k_cache, const void* v_cache,
                     const int32_t* block_tables, int max_blocks_per_seq, const int32_t* seq_lens,
                     const int32_t* query_start_loc, int num_seqs, int num_query_tokens, int max_seq_len,
                     int num_heads, int num_kv_heads, int head_size, int block_size, int64_t num_blocks, float scale,
                     pa_dtype dtype, void* stream) {
  pa_status st = check_decode_shape(num_seqs, num_heads, num_kv_heads, head_size, max_seq_len, block_size, dtype);
  if (st != PA_OK) return st;
  if (dtype != PA_F16 && dtype != PA_BF16) return fail(PA_ERR_UNSUPPORTED, "prefill runs on fp16 and bf16 caches");
  if (num_query_tokens < 0) return fail(PA_ERR_INVALID_ARG, "num_query_tokens %d < 0", num_query_tokens);
  if (max_blocks_per_seq < 1 || (long long)max_seq_len > (long long)max_blocks_per_seq * block_size)
    return fail(PA_ERR_INVALID_ARG, "max_seq_len %d exceeds max_blocks_per_seq %d * block_size %d", max_seq_len,
                max_blocks_per_seq, block_size);
  if (num_blocks < 1) return fail(PA_ERR_INVALID_ARG, "num_blocks %lld < 1", (long long)num_blocks);
  // the kernel's tensor maps address the pools in rows with int32 coordinates: the V
  // pool in rows of one dim of one (block, kv head), the most rows of the two maps
  if ((long long)num_blocks * num_kv_heads * head_size > 0x7fffffffLL)
    return fail(PA_ERR_UNSUPPORTED, "prefill addresses at most 2^31 - 1 V rows (num_blocks * num_kv_heads * "
                                    "head_size = %lld)", (long long)num_blocks * num_kv_heads * head_size);
  if (!std::isfinite(scale)) return fail(PA_ERR_INVALID_ARG, "scale is not finite");
  if (num_seqs == 0 || num_query_tokens == 0) return PA_OK;
  if (!out || !q || !k_cache || !v_cache || !block_tables || !seq_lens || !query_start_loc)
    return fail(PA_ERR_INVALID_ARG, "null pointer");
  if (!aligned(out, 16) || !aligned(q, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) ||
      !aligned(block_tables, 4) || !aligned(seq_lens, 4) || !aligned(query_start_loc, 4))
    return fail(PA_ERR_ALIGNMENT, "q/out/caches need 16-byte, tables and lengths 4-byte alignment");
  pa::PrefillParams p{};
  st = device_error_ptr(&p.err);
  if (st != PA_OK) return st;
  p.out = out;
  p.q = q;
  p.k_cache = k_cache;
  p.v_cache = v_cache;
  p.num_blocks = num_blocks;
  p.max_blocks_per_seq = max_blocks_per_seq;
  p.num_query_tokens = num_query_tokens;
  p.num_heads = num_heads;
  p.num_kv_heads = num_kv_heads;
  p.group = num_heads / num_kv_heads;
  p.max_seq_len = max_seq_len;
  p.scale_log2 = static_cast<float>(static_cast<double>(scale) * 1.4426950408889634);
  p.test_wait_ns = g_test_wait_ns.load(std::memory_order_relaxed);
  for (int c0 = 0; c0 < num_seqs; c0 += pa::kMaxSeqsPerLaunch) {
    p.num_seqs = num_seqs - c0 < pa::kMaxSeqsPerLaunch ? num_seqs - c0 : pa::kMaxSeqsPerLaunch;
    p.block_tables = block_tables + (size_t)c0 * max_blocks_per_seq;
    p.seq_lens = seq_lens + c0;
    p.query_start_loc = query_start_loc + c0;  // offsets stay absolute rows of q and out
    int n = 0;
    const cudaError_t ce = pa::launch_prefill(static_cast<int>(dtype), head_size, block_size, p,
                                              static_cast<cudaStream_t>(stream), &n);
    g_launches.fetch_add(n, std::memory_order_relaxed);
    if (ce != cudaSuccess) return cuda_fail(ce, "prefill launch");
  }
  return PA_OK;
}

pa_status pa_get_device_error(int* code, void* stream) {
  if (!code) return fail(PA_ERR_INVALID_ARG, "null code pointer");
  unsigned* err = nullptr;
  pa_status st = device_error_ptr(&err);
  if (st != PA_OK) return st;
  cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
  unsigned v = 0;
  e = cudaMemcpy(&v, err, sizeof v, cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_fail(e, "reading the device error word");
  const unsigned zero = 0;
  e = cudaMemcpy(err, &zero, sizeof zero, cudaMemcpyHostToDevice);
  if (e != cudaSuccess) return cuda_fail(e, "clearing the device error word");
  *code = static_cast<int>(v);
  return PA_OK;
}

}  // extern "C"
