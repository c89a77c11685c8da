// decode_noalloc.cu -- pa_decode_noalloc: decode whose per-partition scratch is
// a fixed array inside the library, so that the call allocates nothing.
//
// For callers that cannot call cudaMalloc when they decode (a process that
// reserved its memory budget up front, or a latency path where an allocation
// may synchronize the device).  The computation is pa_decode's; only where the
// scratch lives differs.
#include <cstdio>
#include <mutex>

#include "pa.h"

namespace pa {
pa_status record_failure(pa_status st, const char* message);
}

namespace {

// The scratch: one per device that loads the library, held until the process
// exits.  Host code must not use its name as an address -- on the host it is a
// stand-in object; the device address comes from cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_decode_scratch[PA_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;

// Device address of g_decode_scratch on the current device, looked up on the
// first call made with that device current and cached afterwards.
pa_status scratch_address(void** out) {
  static std::mutex mu;
  static void* addr[kMaxDevices] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return pa::record_failure(PA_ERR_CUDA, cudaGetErrorString(e));
  if (dev < 0 || dev >= kMaxDevices) return pa::record_failure(PA_ERR_UNSUPPORTED, "device ordinal too large");
  std::lock_guard<std::mutex> lock(mu);
  if (!addr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_decode_scratch);
    if (e != cudaSuccess || !p) {
      char msg[256];
      snprintf(msg, sizeof msg, "cudaGetSymbolAddress of the decode scratch: %s", cudaGetErrorString(e));
      return pa::record_failure(PA_ERR_CUDA, msg);
    }
    addr[dev] = p;
  }
  *out = addr[dev];
  return PA_OK;
}

}  // namespace

extern "C" pa_status pa_decode_noalloc(void* out, const void* q, const void* k_cache, const void* v_cache,
                                       const int32_t* block_tables, int max_blocks_per_seq, const int32_t* seq_lens,
                                       int num_seqs, int max_seq_len, int num_heads, int num_kv_heads, int head_size,
                                       int block_size, int64_t num_blocks, float scale, int partition_size,
                                       pa_dtype dtype, void* stream) {
  // Scratch this call needs (0 for an unsplit call or for arguments pa_decode rejects).
  const size_t need = pa_decode_workspace_size(num_seqs, num_heads, num_kv_heads, head_size, max_seq_len,
                                               block_size, partition_size, dtype);
  if (need > PA_NOALLOC_SCRATCH_BYTES) {
    char msg[256];
    snprintf(msg, sizeof msg,
             "this split needs %zu bytes of scratch but the built-in array holds %zu; use a larger "
             "partition_size or pa_decode with a caller workspace",
             need, (size_t)PA_NOALLOC_SCRATCH_BYTES);
    return pa::record_failure(PA_ERR_WORKSPACE, msg);
  }
  void* scratch = nullptr;
  const pa_status st = scratch_address(&scratch);
  if (st != PA_OK) return st;
  return pa_decode(out, q, k_cache, v_cache, block_tables, max_blocks_per_seq, seq_lens, num_seqs, max_seq_len,
                   num_heads, num_kv_heads, head_size, block_size, num_blocks, scale, partition_size, scratch,
                   PA_NOALLOC_SCRATCH_BYTES, dtype, stream);
}
