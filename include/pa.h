/*
 * pa.h -- C ABI of the GB300 paged-attention decode library (libpa.so).
 *
 * The library implements the two directions of a paged KV cache that the
 * source pages describe:
 *   - the write path, which scatters each new token's K/V rows into a pool of
 *     fixed-size physical blocks through a flat slot number ("Reading vLLM's
 *     PagedAttention kernel", §3.2), plus the whole-block copy that
 *     copy-on-write needs ("vLLM's PagedAttention: why the KV cache is paged",
 *     §4.2);
 *   - the read path, decode attention: every query row walks its sequence's
 *     block-table row, gathers K/V from the scattered blocks and folds them
 *     into an online softmax, optionally split into partitions of
 *     `partition_size` tokens whose partial results a second pass merges
 *     ("Reading vLLM's PagedAttention kernel", §2, §3.3, §3.4).
 *
 * Memory layouts (all C-contiguous, element type `pa_dtype`):
 *   q, out        [num_seqs, num_heads, head_size]
 *   key, value    [num_tokens, num_kv_heads, head_size]
 *   k_cache       [num_blocks, num_kv_heads, head_size / x, block_size, x],
 *                 x = 16 / element_size (fp32: 4, fp16 and bf16: 8)
 *   v_cache       [num_blocks, num_kv_heads, head_size, block_size]
 *   block_tables  int32 [num_seqs, max_blocks_per_seq]; entry i of row s is the
 *                 physical block that holds tokens i*block_size .. of sequence s
 *   seq_lens      int32 [num_seqs], the number of valid tokens per sequence
 *   slot_mapping  int64 [num_tokens], physical_block * block_size + offset
 *   (cache layouts: "Reading vLLM's PagedAttention kernel", §3.1; an FP8 E4M3
 *   cache has x = 16 and one byte per element)
 *
 * Query head h reads kv head h / (num_heads / num_kv_heads).
 *
 * Conventions for every call:
 *   - Every buffer is owned by the caller and lives in device memory of the
 *     current device; the library allocates nothing and keeps no pointer.
 *   - Calls are asynchronous on `stream` (a cudaStream_t; NULL is the legacy
 *     default stream).  A call validates its host-side arguments, enqueues its
 *     kernels and returns; it never synchronizes, except
 *     pa_get_device_error().  A return of PA_OK means the work was enqueued.
 *   - q, out, key, value, k_cache, v_cache and workspace must be 16-byte
 *     aligned; block_tables and seq_lens 4-byte; slot_mapping and the
 *     copy list 8-byte (PA_ERR_ALIGNMENT otherwise).
 *   - Conditions the host cannot see (a block id outside the pool, a seq_len
 *     outside [1, max_seq_len], a slot beyond the pool) are checked on the
 *     device: the offending access is skipped or clamped into the pool, the
 *     affected outputs are unspecified, and the first such error is recorded
 *     for pa_get_device_error().
 *   - Kernels are chained by programmatic dependent launch: a decode kernel may
 *     start while the previous kernel in the stream (another call of this
 *     library) finishes, and reads seq_lens and the prefix groups before it waits
 *     for that kernel; everything else it reads or writes it touches after.  A
 *     caller kernel that writes seq_lens or the prefix groups must not release
 *     its dependents early (griddepcontrol.launch_dependents) before those writes;
 *     an ordinary kernel never does.
 *   - Thread safety: calls may be made from several host threads; the
 *     device-error word and the launch counter are shared per process.
 *   - The library looks up the device addresses of its own device-side objects
 *     (the error word, the scratch of pa_decode_noalloc) once per device, on the
 *     first call that needs them.  A cudaDeviceReset() of a device the library has
 *     used makes those addresses stale: do not call the library on that device
 *     again in the same process.
 */
#ifndef PA_H_
#define PA_H_

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define PA_API __attribute__((visibility("default")))
#else
#define PA_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  PA_OK = 0,
  PA_ERR_INVALID_ARG = 1,  /* a size, pointer or combination is invalid */
  PA_ERR_UNSUPPORTED = 2,  /* valid, but outside what the kernels are built for */
  PA_ERR_ALIGNMENT = 3,    /* a pointer breaks the alignment rule above */
  PA_ERR_WORKSPACE = 4,    /* workspace missing or smaller than required */
  PA_ERR_CUDA = 5,         /* a CUDA runtime call failed (see pa_last_error_message) */
  PA_ERR_OUT_OF_BLOCKS = 6 /* the block manager's pool cannot serve the request (pa_block_manager.h) */
} pa_status;

typedef enum { PA_F32 = 0, PA_F16 = 1, PA_BF16 = 2, PA_FP8_E4M3 = 3 } pa_dtype;

/* partition_size values for pa_decode.  The kernels cut sequences wherever their
 * load-balanced schedule needs to (every warp streams an equal share of all blocks)
 * and merge the pieces, so no caller partition is ever needed for speed: AUTO means
 * "no caller partitions" and is resolved to NONE (see pa_decode_plan_partition). */
#define PA_PARTITION_NONE 0    /* no caller partitions */
#define PA_PARTITION_AUTO (-1) /* the library's choice: currently always PA_PARTITION_NONE */

/* device-side error codes returned by pa_get_device_error */
#define PA_DEVERR_NONE 0
#define PA_DEVERR_BLOCK_ID 1   /* a block-table entry outside [0, num_blocks) */
#define PA_DEVERR_SEQ_LEN 2    /* a seq_lens entry outside [1, max_seq_len] */
#define PA_DEVERR_SLOT 3       /* a slot_mapping entry >= num_blocks * block_size */
#define PA_DEVERR_TIMEOUT 4    /* a pipeline wait in a kernel gave up after ~1 s */
#define PA_DEVERR_COPY_ID 5    /* a copy_blocks id outside [0, num_blocks) */
#define PA_DEVERR_SHARED 6     /* pa_decode_shared: a block declared shared differs between two tables */

/* Human-readable name of a status. Never NULL. */
PA_API const char* pa_status_string(pa_status s);

/* Detail of the last non-OK status returned on the calling host thread. */
PA_API const char* pa_last_error_message(void);

/*
 * Write path ("Reading vLLM's PagedAttention kernel", §3.2): for every token t
 * with slot = slot_mapping[t] >= 0, copy key[t, h, :] into
 * k_cache[slot / block_size, h, :, slot % block_size, :] and value[t, h, :] into
 * v_cache[slot / block_size, h, :, slot % block_size] for all kv heads h.
 * A pure copy: the bytes of the cache equal the bytes of key/value.
 * A negative slot marks a padding token, which is skipped.  Two tokens of one
 * call must not share a slot (the result would be either token's row).
 * head_size must be a multiple of x; block_size >= 1.
 */
PA_API pa_status pa_reshape_and_cache(const void* key, const void* value, void* k_cache, void* v_cache,
                               const int64_t* slot_mapping, int64_t num_tokens, int num_kv_heads,
                               int head_size, int block_size, int64_t num_blocks, pa_dtype dtype,
                               void* stream);

/*
 * Write path into a cache of another dtype ("Reading vLLM's PagedAttention
 * kernel", §3.2: the write also takes kv_cache_dtype, k_scale and v_scale).
 * With cache_dtype PA_FP8_E4M3 every element x of key (value) is stored as the
 * OCP FP8 E4M3 code of x / k_scale (x / v_scale): the division correctly rounded
 * in fp32, the code rounded to nearest with ties to even and clamped to +-448
 * (no infinities; a NaN stays NaN).  A later read of that cache gives
 * code * k_scale (code * v_scale).  key_dtype is PA_F32, PA_F16 or PA_BF16;
 * scales are positive and finite; head_size is a multiple of 16.  For any other
 * cache_dtype the call is pa_reshape_and_cache and requires key_dtype ==
 * cache_dtype and both scales 1.  Layouts, slots and errors as there.
 */
PA_API pa_status pa_reshape_and_cache_scaled(const void* key, const void* value, void* k_cache, void* v_cache,
                                             const int64_t* slot_mapping, int64_t num_tokens, int num_kv_heads,
                                             int head_size, int block_size, int64_t num_blocks,
                                             pa_dtype key_dtype, pa_dtype cache_dtype, float k_scale,
                                             float v_scale, void* stream);

/*
 * Copy-on-write block copy ("vLLM's PagedAttention: why the KV cache is paged",
 * §4.2): for each pair i, physical block src_dst[2i] is copied to block
 * src_dst[2i+1] -- every kv head, K and V.  The pairs run in parallel: no
 * destination may repeat and no destination may be a source of the same call.
 */
PA_API pa_status pa_copy_blocks(void* k_cache, void* v_cache, const int64_t* src_dst, int64_t num_pairs,
                         int num_kv_heads, int head_size, int block_size, int64_t num_blocks,
                         pa_dtype dtype, void* stream);

/*
 * The partition size pa_decode uses for PA_PARTITION_AUTO: PA_PARTITION_NONE for
 * every shape pa_decode accepts (the schedule splits sequences by itself; see
 * PA_PARTITION_AUTO above).  Returns -1 for arguments pa_decode would reject.
 */
PA_API int pa_decode_plan_partition(int num_seqs, int num_heads, int num_kv_heads, int head_size,
                             int max_seq_len, int block_size, pa_dtype dtype);

/*
 * Bytes of workspace pa_decode needs for these arguments (partition_size may be
 * PA_PARTITION_AUTO; it is resolved as pa_decode_plan_partition does).  Zero
 * when no split is made.  The workspace holds per-partition maxima, sums and
 * partial outputs in fp32; its contents need no initialisation and are
 * meaningless between calls.
 */
PA_API size_t pa_decode_workspace_size(int num_seqs, int num_heads, int num_kv_heads, int head_size,
                                int max_seq_len, int block_size, int partition_size,
                                pa_dtype dtype);

/*
 * Decode attention over the paged pool ("Reading vLLM's PagedAttention
 * kernel", §2 flowchart, §3.3, §3.4; "KV Cache and PagedAttention memory
 * management", attention formula): for each sequence s and query head h,
 *     out[s, h, :] = sum_t softmax_t(scale * <q[s, h, :], K_s[t, :]>) V_s[t, :]
 * over the tokens t < seq_lens[s], with K_s and V_s gathered in logical order
 * through block_tables[s] from kv head h / (num_heads / num_kv_heads).
 * Scores, softmax statistics and the weighted sum are kept in fp32; out is
 * rounded once to `dtype` (round to nearest even).
 *
 * max_seq_len is a host-side bound on every seq_lens entry and must not exceed
 * max_blocks_per_seq * block_size.  partition_size is PA_PARTITION_NONE,
 * PA_PARTITION_AUTO or a positive multiple of block_size: a sequence longer
 * than one partition is processed as independent partitions of that many
 * tokens whose (max, sum, partial output) results are merged by a second
 * kernel; the merged result equals the unsplit one up to fp32 rounding, and a
 * sequence that fits in one partition gives bit-identical output to
 * PA_PARTITION_NONE.  workspace must hold pa_decode_workspace_size() bytes
 * (it may be NULL when that is 0).
 *
 * Supported: head_size 64 or 128; block_size 16 or 32; num_heads a multiple
 * of num_kv_heads; num_seqs and num_heads at most 65535.  Output for a given
 * set of arguments is deterministic and does not depend on the physical
 * placement of the blocks.
 */
PA_API pa_status pa_decode(void* out, const void* q, const void* k_cache, const void* v_cache,
                    const int32_t* block_tables, int max_blocks_per_seq, const int32_t* seq_lens,
                    int num_seqs, int max_seq_len, int num_heads, int num_kv_heads, int head_size,
                    int block_size, int64_t num_blocks, float scale, int partition_size,
                    void* workspace, size_t workspace_bytes, pa_dtype dtype, void* stream);

/*
 * pa_decode over a cache whose dtype differs from the query's: with cache_dtype
 * PA_FP8_E4M3 and q_dtype PA_F16 or PA_BF16, K and V read back as
 * code * k_scale and code * v_scale (see pa_reshape_and_cache_scaled); out has
 * q_dtype.  Scores, softmax and the weighted sum are fp32 as in pa_decode.  For
 * any other cache_dtype, q_dtype must equal it and both scales be 1.  The
 * workspace is pa_decode_workspace_size(..., cache_dtype).  pa_decode itself
 * rejects PA_FP8_E4M3 (it has no query dtype or scales).
 */
PA_API pa_status pa_decode_scaled(void* out, const void* q, const void* k_cache, const void* v_cache,
                                  const int32_t* block_tables, int max_blocks_per_seq, const int32_t* seq_lens,
                                  int num_seqs, int max_seq_len, int num_heads, int num_kv_heads, int head_size,
                                  int block_size, int64_t num_blocks, float scale, int partition_size,
                                  void* workspace, size_t workspace_bytes, pa_dtype q_dtype, pa_dtype cache_dtype,
                                  float k_scale, float v_scale, void* stream);

/*
 * One generation step in one call: the copy-on-write copies, then the write of
 * each sequence's new token fused into decode ("vLLM's
 * PagedAttention: why the KV cache is paged", §4.2: a shared block about to be
 * written is copied first, then written; "Reading vLLM's PagedAttention kernel",
 * §3.2 write path and §2 decode).  The result equals, byte for byte in the pools
 * and bit for bit in out, the three calls
 *     pa_copy_blocks(k_cache, v_cache, src_dst, num_pairs, ...);
 *     pa_reshape_and_cache(key, value, k_cache, v_cache, slots, num_seqs, ...);
 *     pa_decode(out, q, k_cache, v_cache, block_tables, ..., seq_lens, ...);
 * where slots[s] is the position seq_lens[s] - 1 of sequence s under its block
 * table: the new token of a sequence is the last one it attends to.
 *
 * key, value  [num_seqs, num_kv_heads, head_size], the cache dtype: one new token
 *             per sequence (a sequence with seq_lens[s] outside [1, max_seq_len]
 *             writes nothing and is reported as in pa_decode)
 * src_dst     int64 [num_pairs, 2] (may be NULL when num_pairs is 0), as in
 *             pa_copy_blocks; the copies complete before any token is written
 * everything else as in pa_decode, with the same workspace size.
 *
 * dtype is PA_F32, PA_F16 or PA_BF16; an FP8 cache takes pa_decode_step_scaled
 * below.  No two sequences of the call may
 * write the same slot, and no sequence may read a slot another one writes
 * (the block manager's copy-on-write guarantees both).
 *
 * Kernels: the decode kernel writes each new token and decodes (the token
 * reaches the stage of its sequence's last block with that block's TMA copy,
 * so decode never waits for the write), then the merge kernel.  With
 * num_pairs > 0 the copy kernel of pa_copy_blocks runs first.  Asynchronous on
 * `stream`.
 */
PA_API pa_status pa_decode_step(void* out, const void* q, const void* key, const void* value, void* k_cache,
                                void* v_cache, const int64_t* src_dst, int64_t num_pairs,
                                const int32_t* block_tables, int max_blocks_per_seq, const int32_t* seq_lens,
                                int num_seqs, int max_seq_len, int num_heads, int num_kv_heads, int head_size,
                                int block_size, int64_t num_blocks, float scale, int partition_size,
                                void* workspace, size_t workspace_bytes, pa_dtype dtype, void* stream);

/*
 * pa_decode_step over a cache whose dtype differs from the query's: with
 * cache_dtype PA_FP8_E4M3 and q_dtype PA_F16 or PA_BF16, key and value come in
 * q_dtype and are stored as pa_reshape_and_cache_scaled stores them (the E4M3
 * code of x / k_scale, x / v_scale), then decode reads the pool as
 * pa_decode_scaled does.  Equal, byte for byte in the pools and bit for bit in
 * out, to pa_copy_blocks + pa_reshape_and_cache_scaled + pa_decode_scaled.  For
 * any other cache_dtype, q_dtype must equal it and both scales be 1 (then it is
 * pa_decode_step).
 */
PA_API pa_status pa_decode_step_scaled(void* out, const void* q, const void* key, const void* value,
                                       void* k_cache, void* v_cache, const int64_t* src_dst, int64_t num_pairs,
                                       const int32_t* block_tables, int max_blocks_per_seq,
                                       const int32_t* seq_lens, int num_seqs, int max_seq_len, int num_heads,
                                       int num_kv_heads, int head_size, int block_size, int64_t num_blocks,
                                       float scale, int partition_size, void* workspace, size_t workspace_bytes,
                                       pa_dtype q_dtype, pa_dtype cache_dtype, float k_scale, float v_scale,
                                       void* stream);

/*
 * Decode (or a whole step) over sequences that share prefix blocks, reading each
 * shared block once for all of its sharers ("vLLM's PagedAttention: why the KV
 * cache is paged", §4.2: the sequences of one request -- parallel samples of a
 * common prompt -- map their first logical blocks to the same physical blocks,
 * with reference counts, until a write forces a copy).  The result is the one the
 * pages define for each sequence on its own: equal, up to fp32 rounding, to
 * pa_decode_step_scaled (key != NULL) or pa_decode_scaled (key == value == NULL)
 * with the same arguments; what changes is that a block held by several sequences
 * of a cluster leaves DRAM once.
 *
 * prefix_group   int32 [num_seqs]: a group is a run of consecutive sequences with
 *                equal values (any ids; a sequence that shares nothing can have a
 *                value of its own).
 * prefix_blocks  int32 [num_seqs]: sequence s holds the first prefix_blocks[s]
 *                blocks of its group's common prefix, so that any two sequences s,
 *                t of a group have equal block-table entries 0 .. min(prefix_blocks[s],
 *                prefix_blocks[t]) - 1.  (Comparing every table of a group with
 *                that of its longest sequence gives such values; so does
 *                pa_bm_prefix_groups.)  Values beyond a sequence's blocks are
 *                clipped.  A declared entry that differs is reported as
 *                PA_DEVERR_SHARED and the affected outputs are unspecified.
 *
 * How it is used: a group is cut into clusters of C / (num_heads / num_kv_heads)
 * consecutive sequences (C = 16 query heads for 16-bit caches, 8 for FP8 caches,
 * whose kernel keeps more warps); the first B blocks of a cluster (B: the second largest
 * prefix_blocks among its members) are attended once, with the query heads of all
 * members in one tensor-core tile (a member's columns take part in the blocks it
 * holds), and merged with each member's own blocks.  The last block of every
 * sequence is always read as its own.  Clusters need a 16-bit cache with at most 8
 * query heads per kv head, or an FP8 cache with at most 4; for other shapes the call runs as
 * pa_decode_step_scaled / pa_decode_scaled.  A launch covers at most 1024
 * sequences; a cluster never spans two launches.
 *
 * key, value may be NULL (both): decode only; then num_pairs must be 0.  Every
 * other argument as in pa_decode_step_scaled, except that the workspace must hold
 * pa_decode_shared_workspace_size() bytes.
 */
PA_API pa_status pa_decode_shared(void* out, const void* q, const void* key, const void* value, void* k_cache,
                                  void* v_cache, const int64_t* src_dst, int64_t num_pairs,
                                  const int32_t* block_tables, int max_blocks_per_seq, const int32_t* seq_lens,
                                  const int32_t* prefix_group, const int32_t* prefix_blocks, int num_seqs,
                                  int max_seq_len, int num_heads, int num_kv_heads, int head_size, int block_size,
                                  int64_t num_blocks, float scale, int partition_size, void* workspace,
                                  size_t workspace_bytes, pa_dtype q_dtype, pa_dtype cache_dtype, float k_scale,
                                  float v_scale, void* stream);

/* Workspace bytes of pa_decode_shared (0 for arguments it would reject). */
PA_API size_t pa_decode_shared_workspace_size(int num_seqs, int num_heads, int num_kv_heads, int head_size,
                                              int max_seq_len, int block_size, int partition_size,
                                              pa_dtype cache_dtype);

/*
 * Read and clear the first device-side error recorded on the current device
 * (PA_DEVERR_*; 0 if none).  Synchronizes `stream` first.
 */
PA_API pa_status pa_get_device_error(int* code, void* stream);

/* Number of kernels this library has launched in this process (all devices). */
PA_API uint64_t pa_launch_count(void);

/*
 * Diagnostics, for testing the timeout path only (no counterpart in the pages).
 * Every pipeline wait in the kernels gives up after about 1 s, records
 * PA_DEVERR_TIMEOUT, waits (bounded) for the copies it has in flight and ends
 * the kernel early, leaving the outputs of the call unspecified; the context
 * stays usable.  While `nanoseconds` > 0, decode, the fused step and prefill
 * launched afterwards make their first pipeline wait (per decode warp, per
 * prefill CTA) on a barrier that nothing completes, for that long, so that this
 * path runs for real.  0 (the default) restores normal operation.  The setting
 * is process-wide and is read when a call enqueues its kernels.
 */
PA_API void pa_set_test_wait_limit(uint64_t nanoseconds);

/*
 * Chunked prefill: causal attention of a chunk of new query tokens per sequence
 * over the paged pool -- the step before decode ("vLLM's PagedAttention: why the
 * KV cache is paged", §2.3: a prompt is processed and its K/V enter the cache,
 * then tokens are generated one at a time).  The chunk's own K/V must already be
 * in the cache (pa_reshape_and_cache with the chunk's slots).  For sequence s,
 * seq_lens[s] = L counts every cached token, the chunk included; the chunk is
 * the n = query_start_loc[s+1] - query_start_loc[s] tokens at positions
 * L - n .. L - 1, its queries are rows query_start_loc[s] .. of q, and query
 * token i (position p = L - n + i) attends to positions 0..p:
 *     out[row, h, :] = softmax(scale * q[row, h, :] . K_s[0..p]^T) V_s[0..p]
 * query head h reading kv head h / (num_heads / num_kv_heads).
 *
 * q, out          [num_query_tokens, num_heads, head_size], the cache dtype
 * query_start_loc int32 [num_seqs + 1], query_start_loc[0] = 0, non-decreasing,
 *                 query_start_loc[num_seqs] = num_query_tokens
 * dtype           PA_F16 or PA_BF16; head_size 64 or 128; block_size 16 or 32
 *
 * No workspace.  A sequence whose length lies outside [1, max_seq_len] or whose
 * chunk is longer than itself is recorded as PA_DEVERR_SEQ_LEN and its rows of
 * out are unspecified.  num_blocks * num_kv_heads * head_size must stay below
 * 2^31 (PA_ERR_UNSUPPORTED otherwise).  The kernel reads the pools through TMA
 * tensor maps encoded on the host at every call (cuTensorMapEncodeTiled, found
 * through the CUDA runtime; PA_ERR_CUDA if the driver does not provide it).
 * Asynchronous on `stream`.
 */
PA_API pa_status pa_prefill(void* out, const void* q, const void* k_cache, const void* v_cache,
                            const int32_t* block_tables, int max_blocks_per_seq, const int32_t* seq_lens,
                            const int32_t* query_start_loc, int num_seqs, int num_query_tokens, int max_seq_len,
                            int num_heads, int num_kv_heads, int head_size, int block_size, int64_t num_blocks,
                            float scale, pa_dtype dtype, void* stream);

/*
 * Decode with no allocation anywhere: the same computation, arguments and
 * results as pa_decode, but the per-partition scratch lives in a fixed array
 * inside the library instead of a caller-provided workspace.  This serves
 * callers that cannot call cudaMalloc at the point where they decode -- for
 * example a process that reserved its whole memory budget up front (weights
 * plus the KV pool) and forbids later allocations, or a caller on a latency
 * path where an allocation may synchronize the device.  (The pages have no
 * counterpart to this call: it is a deployment convenience of this library.)
 *
 *   - The array holds PA_NOALLOC_SCRATCH_BYTES (32 MiB) and every GPU that loads
 *     libpa keeps it until the process exits.  A shape whose split needs more
 *     (see pa_decode_workspace_size) is rejected with PA_ERR_WORKSPACE before
 *     anything is enqueued; pick a larger partition_size or use pa_decode.
 *   - The first call on a device looks up the array's device address (once per
 *     device, with that device current) and keeps it for the life of the process;
 *     make that first call before any stream capture begins.  The address stays
 *     valid until a cudaDeviceReset() of that device, after which this call must
 *     not be used on it again.
 *   - Every call on a device shares the one array and it keeps whatever the last
 *     call left there.  Nothing in it has to start at zero: each call writes
 *     every partial result before its merge reads it.  Calls whose work overlaps
 *     on the GPU (other streams, other host threads) race on the array and give
 *     undefined results: order them on one stream.
 *   - Calls no cudaMalloc, cudaFree or allocating library routine.
 */
#define PA_NOALLOC_SCRATCH_BYTES (32u * 1024u * 1024u)
PA_API pa_status pa_decode_noalloc(void* out, const void* q, const void* k_cache, const void* v_cache,
                                   const int32_t* block_tables, int max_blocks_per_seq,
                                   const int32_t* seq_lens, int num_seqs, int max_seq_len,
                                   int num_heads, int num_kv_heads, int head_size, int block_size,
                                   int64_t num_blocks, float scale, int partition_size,
                                   pa_dtype dtype, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* PA_H_ */
