/*
 * pa_oracle.c -- CPU oracle for paged-attention decode.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the plain, slow, fp64 statement of
 * what the paged decode path computes.  It is used by the tests, by the smoke
 * check and by the benchmark's CPU-baseline leg, and by nothing else.  It shares
 * no code, header, table or helper with the CUDA library, and the library never
 * calls it.
 *
 * Sources (web pages on vLLM's paged KV cache; cited by title and section):
 *   [ILP]   "Reading vLLM's PagedAttention kernel" (inference-learning-path,
 *           part 3): §2 mental model, §3.1 cache layout, §3.2 writing into the
 *           cache, §3.3 kernel structure, §4 runnable CPU reference.
 *   [AIQZ]  "KV Cache and PagedAttention memory management" (aiqz.cc):
 *           the attention formula softmax(Q K^T / sqrt(d_k)) V, paging section.
 *   [BHHXX] "vLLM's PagedAttention: why the KV cache is paged" (bhhxx.wiki):
 *           §4.1 logical/physical block mapping, §4.2 copy-on-write.
 *
 * Readings taken where the pages are silent (each is listed in the design notes):
 *   - x = 16 / element_size for every dtype (the pages state it for fp16 only);
 *   - element (b, h, d, t) of the K pool is k_cache[b][h][d/x][t][d%x] and of
 *     the V pool v_cache[b][h][d][t], all arrays C-contiguous;
 *   - slot s decodes to block s / block_size, offset s % block_size; a negative
 *     slot is a padding token and is skipped;
 *   - query head h reads kv head h / (num_heads / num_kv_heads);
 *   - a quantised (FP8 E4M3) cache stores the code of x / scale per element,
 *     with one k_scale and one v_scale per call, and reads back code * scale.
 *
 * The decode result has a plain definition -- paging changes where K/V live,
 * not what attention computes ([ILP] §4, §6; [BHHXX] §4.3) -- so the oracle is
 * that definition written out: gather K/V in logical order through the block
 * table, then dense softmax(scale * q K^T) V in fp64.  Inputs stored as fp16 or
 * bf16 are widened exactly to fp64.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

enum { OR_F32 = 0, OR_F16 = 1, OR_BF16 = 2, OR_F64 = 3, OR_FP8 = 4 };

enum {
  OR_OK = 0,
  OR_ERR_ARG = 1,        /* bad shape or dtype */
  OR_ERR_SEQ_LEN = 2,    /* seq_len < 1 or beyond the block table */
  OR_ERR_BLOCK_ID = 3,   /* block table entry outside the pool */
  OR_ERR_SLOT = 4,       /* slot beyond the pool */
  OR_ERR_DUP_SLOT = 5,   /* two tokens written to one slot in a call */
  OR_ERR_NOMEM = 6
};

static int elem_bytes(int dtype) {
  switch (dtype) {
    case OR_F32: return 4;
    case OR_F16: return 2;
    case OR_BF16: return 2;
    case OR_F64: return 8;
    case OR_FP8: return 1;
    default: return 0;
  }
}

/* IEEE 754 binary16, from the format: 1 sign bit, 5 exponent bits (bias 15),
 * 10 fraction bits.  Exponent 0 is zero/subnormal (f * 2^-24), 31 is inf/NaN. */
static double half_bits_to_double(uint16_t h) {
  int sign = (h >> 15) & 1;
  int e = (h >> 10) & 0x1f;
  int f = h & 0x3ff;
  double v;
  if (e == 0)
    v = ldexp((double)f, -24);
  else if (e == 31)
    v = f ? NAN : INFINITY;
  else
    v = ldexp((double)(f | 0x400), e - 25);
  return sign ? -v : v;
}

/* bfloat16 is the top half of an IEEE binary32. */
static double bf16_bits_to_double(uint16_t b) {
  uint32_t u = (uint32_t)b << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

/* OCP FP8 E4M3 (the "fn" variant): 1 sign bit, 4 exponent bits (bias 7),
 * 3 fraction bits; exponent 0 is zero/subnormal (f * 2^-9); S.1111.111 is NaN;
 * there are no infinities, so the largest magnitude is 1.75 * 2^8 = 448. */
static double e4m3_bits_to_double(uint8_t b) {
  int sign = (b >> 7) & 1;
  int e = (b >> 3) & 0xf;
  int f = b & 7;
  double v;
  if (e == 15 && f == 7) return NAN;
  if (e == 0)
    v = ldexp((double)f, -9);
  else
    v = ldexp((double)(f | 8), e - 10);
  return sign ? -v : v;
}

/* Nearest E4M3 code to x (ties to the even code), magnitudes beyond 448 clamped
 * to 448: a search over the 127 non-negative finite codes. */
static uint8_t double_to_e4m3_satfinite(double x) {
  if (isnan(x)) return 0x7f;
  const uint8_t sign = signbit(x) ? 0x80 : 0;
  const double a = fabs(x);
  int best = 0;
  double best_d = INFINITY;
  for (int c = 0; c <= 126; ++c) {
    const double d = fabs(e4m3_bits_to_double((uint8_t)c) - a);
    if (d < best_d || (d == best_d && (c & 1) == 0)) {
      best = c;
      best_d = d;
    }
  }
  return (uint8_t)(sign | best);
}

/* Element idx of an array of the given dtype, widened exactly to fp64. */
static double load(const void* base, int64_t idx, int dtype) {
  switch (dtype) {
    case OR_F32: return (double)((const float*)base)[idx];
    case OR_F16: return half_bits_to_double(((const uint16_t*)base)[idx]);
    case OR_BF16: return bf16_bits_to_double(((const uint16_t*)base)[idx]);
    case OR_FP8: return e4m3_bits_to_double(((const uint8_t*)base)[idx]);
    default: return ((const double*)base)[idx];
  }
}

/* [ILP] §3.1: x = 16 / element_size packs head_size into 16-byte groups. */
static int pack_x(int dtype) { return 16 / elem_bytes(dtype); }

/* [ILP] §3.1 K pool [num_blocks, num_kv_heads, head_size/x, block_size, x]. */
static int64_t k_index(int64_t b, int h, int d, int t, int Hkv, int D, int bs, int x) {
  return ((((int64_t)b * Hkv + h) * (D / x) + d / x) * bs + t) * x + d % x;
}

/* [ILP] §3.1 V pool [num_blocks, num_kv_heads, head_size, block_size]. */
static int64_t v_index(int64_t b, int h, int d, int t, int Hkv, int D, int bs) {
  return (((int64_t)b * Hkv + h) * D + d) * bs + t;
}

int oracle_elem_bytes(int dtype) { return elem_bytes(dtype); }
int oracle_pack_x(int dtype) { return elem_bytes(dtype) ? pack_x(dtype) : 0; }

/* Threads the parallel loops use from now on (n >= 1); for timing one core against all. */
void oracle_set_num_threads(int n) {
#ifdef _OPENMP
  if (n >= 1) omp_set_num_threads(n);
#else
  (void)n;
#endif
}

int oracle_num_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

/* E4M3 codes of n fp64 values (ties to even, clamped to +-448). */
int oracle_encode_e4m3(uint8_t* out, const double* in, int64_t n) {
  for (int64_t i = 0; i < n; ++i) out[i] = double_to_e4m3_satfinite(in[i]);
  return OR_OK;
}

/* Widen n elements to fp64 (used by the tests to pin the decoders). */
int oracle_widen(double* out, const void* in, int64_t n, int dtype) {
  if (!elem_bytes(dtype)) return OR_ERR_ARG;
  for (int64_t i = 0; i < n; ++i) out[i] = load(in, i, dtype);
  return OR_OK;
}

/*
 * Write path, [ILP] §3.2: every new token t carries a flat slot
 * (physical block * block_size + offset in block); its K and V rows are copied
 * into that slot of the pools.  key/value are [num_tokens, num_kv_heads,
 * head_size] C-contiguous.  A pure byte copy: nothing is converted.
 */
int oracle_reshape_and_cache(const void* key, const void* value, void* k_cache, void* v_cache,
                             const int64_t* slot_mapping, int64_t num_tokens, int num_kv_heads,
                             int head_size, int block_size, int64_t num_blocks, int dtype) {
  const int e = elem_bytes(dtype);
  if (!e || num_tokens < 0 || num_kv_heads < 1 || block_size < 1 || head_size < 1) return OR_ERR_ARG;
  const int x = pack_x(dtype);
  if (head_size % x) return OR_ERR_ARG;
  const int64_t n_slots = num_blocks * block_size;
  /* Reject a slot outside the pool and a slot written twice in one call. */
  for (int64_t t = 0; t < num_tokens; ++t) {
    const int64_t slot = slot_mapping[t];
    if (slot < 0) continue;
    if (slot >= n_slots) return OR_ERR_SLOT;
    for (int64_t u = 0; u < t; ++u)
      if (slot_mapping[u] == slot) return OR_ERR_DUP_SLOT;
  }
  for (int64_t t = 0; t < num_tokens; ++t) {
    const int64_t slot = slot_mapping[t];
    if (slot < 0) continue;
    const int64_t blk = slot / block_size;
    const int off = (int)(slot % block_size);
    for (int h = 0; h < num_kv_heads; ++h) {
      for (int d = 0; d < head_size; ++d) {
        const int64_t src = ((int64_t)t * num_kv_heads + h) * head_size + d;
        memcpy((char*)k_cache + k_index(blk, h, d, off, num_kv_heads, head_size, block_size, x) * e,
               (const char*)key + src * e, (size_t)e);
        memcpy((char*)v_cache + v_index(blk, h, d, off, num_kv_heads, head_size, block_size) * e,
               (const char*)value + src * e, (size_t)e);
      }
    }
  }
  return OR_OK;
}

/*
 * Write path with a quantised cache ([ILP] §3.2 names the kv_cache_dtype, k_scale
 * and v_scale arguments of the write): each element x of key (value) is stored as
 * the E4M3 code of x / k_scale (x / v_scale), the division done in fp32 as the
 * write kernel does, rounded to nearest (ties to even) and clamped to +-448.
 * Reading it back gives code * scale.  For a 16-bit or fp32 cache of the key's own
 * dtype with both scales 1 this is the plain byte copy above.
 */
int oracle_reshape_and_cache_scaled(const void* key, const void* value, void* k_cache, void* v_cache,
                                    const int64_t* slot_mapping, int64_t num_tokens, int num_kv_heads,
                                    int head_size, int block_size, int64_t num_blocks, int key_dtype,
                                    int cache_dtype, double k_scale, double v_scale) {
  if (cache_dtype != OR_FP8) {
    if (cache_dtype != key_dtype || k_scale != 1.0 || v_scale != 1.0) return OR_ERR_ARG;
    return oracle_reshape_and_cache(key, value, k_cache, v_cache, slot_mapping, num_tokens, num_kv_heads,
                                    head_size, block_size, num_blocks, key_dtype);
  }
  if (key_dtype != OR_F32 && key_dtype != OR_F16 && key_dtype != OR_BF16) return OR_ERR_ARG;
  if (num_tokens < 0 || num_kv_heads < 1 || block_size < 1 || head_size % 16 || !(k_scale > 0) || !(v_scale > 0))
    return OR_ERR_ARG;
  const int64_t n_slots = num_blocks * block_size;
  for (int64_t t = 0; t < num_tokens; ++t) {
    const int64_t slot = slot_mapping[t];
    if (slot < 0) continue;
    if (slot >= n_slots) return OR_ERR_SLOT;
    for (int64_t u = 0; u < t; ++u)
      if (slot_mapping[u] == slot) return OR_ERR_DUP_SLOT;
  }
  const float ks = (float)k_scale, vs = (float)v_scale;
  for (int64_t t = 0; t < num_tokens; ++t) {
    const int64_t slot = slot_mapping[t];
    if (slot < 0) continue;
    const int64_t blk = slot / block_size;
    const int off = (int)(slot % block_size);
    for (int h = 0; h < num_kv_heads; ++h) {
      for (int d = 0; d < head_size; ++d) {
        const int64_t src = ((int64_t)t * num_kv_heads + h) * head_size + d;
        const float kq = (float)load(key, src, key_dtype) / ks;
        const float vq = (float)load(value, src, key_dtype) / vs;
        ((uint8_t*)k_cache)[k_index(blk, h, d, off, num_kv_heads, head_size, block_size, 16)] =
            double_to_e4m3_satfinite((double)kq);
        ((uint8_t*)v_cache)[v_index(blk, h, d, off, num_kv_heads, head_size, block_size)] =
            double_to_e4m3_satfinite((double)vq);
      }
    }
  }
  return OR_OK;
}

/*
 * Copy-on-write block copy, [BHHXX] §4.2: before a shared physical block
 * (refcount > 1) is written, it is first copied to a fresh block.  Pair i of
 * src_dst is (src, dst); the whole block -- every kv head, K and V -- is copied.
 * Pairs are applied in order.
 */
int oracle_copy_blocks(void* k_cache, void* v_cache, const int64_t* src_dst, int64_t n,
                       int num_kv_heads, int head_size, int block_size, int64_t num_blocks,
                       int dtype) {
  const int e = elem_bytes(dtype);
  if (!e || n < 0) return OR_ERR_ARG;
  const size_t blk_bytes = (size_t)num_kv_heads * head_size * block_size * e;
  for (int64_t i = 0; i < n; ++i) {
    const int64_t src = src_dst[2 * i], dst = src_dst[2 * i + 1];
    if (src < 0 || src >= num_blocks || dst < 0 || dst >= num_blocks) return OR_ERR_BLOCK_ID;
    memmove((char*)k_cache + (size_t)dst * blk_bytes, (const char*)k_cache + (size_t)src * blk_bytes, blk_bytes);
    memmove((char*)v_cache + (size_t)dst * blk_bytes, (const char*)v_cache + (size_t)src * blk_bytes, blk_bytes);
  }
  return OR_OK;
}

/*
 * Gather sequence s's first L tokens of kv head kvh, in logical order, through
 * its block-table row ([ILP] §2 and §3.4 steps 1-2; [AIQZ] paging: logical
 * block i maps to physical block p_i for 0 <= i < ceil(L / block_size)).
 * K and V come out as contiguous [L][D] fp64 rows.
 */
static int gather_seq(double* K, double* V, const void* k_cache, const void* v_cache,
                      const int32_t* table_row, int L, int kvh, int Hkv, int D, int bs,
                      int64_t num_blocks, int dtype, double k_scale, double v_scale) {
  const int x = pack_x(dtype);
  for (int t = 0; t < L; ++t) {
    const int64_t phys = table_row[t / bs];
    if (phys < 0 || phys >= num_blocks) return OR_ERR_BLOCK_ID;
    const int off = t % bs;
    for (int d = 0; d < D; ++d) {
      K[(int64_t)t * D + d] = k_scale * load(k_cache, k_index(phys, kvh, d, off, Hkv, D, bs, x), dtype);
      V[(int64_t)t * D + d] = v_scale * load(v_cache, v_index(phys, kvh, d, off, Hkv, D, bs), dtype);
    }
  }
  return OR_OK;
}

/*
 * Decode attention, the definition ([AIQZ] attention formula; [ILP] §4 dense
 * reference): for each sequence s and query head h,
 *     z_t = scale * <q[s,h,:], K_s[t,:]>          t < seq_lens[s]
 *     w   = softmax(z)                             (max-subtracted, fp64)
 *     out[s,h,:] = sum_t w_t V_s[t,:]
 * with K_s, V_s gathered through block_tables[s] from kv head h / G.
 *
 * q is [num_seqs, num_heads, head_size] in `dtype`; out is fp64, same shape.
 * If weights != NULL it receives w for (s, h) at weights[(s*H + h)*w_stride + t].
 * Positions at or beyond seq_lens[s] are never read ([ILP] §4: a partially
 * filled last block is guarded by the true sequence length).
 */
int oracle_decode_scaled(double* out, double* weights, int64_t w_stride, const void* q,
                         const void* k_cache, const void* v_cache, const int32_t* block_tables,
                         int max_blocks_per_seq, const int32_t* seq_lens, int num_seqs, int num_heads,
                         int num_kv_heads, int head_size, int block_size, int64_t num_blocks,
                         double scale, int q_dtype, int cache_dtype, double k_scale, double v_scale) {
  const int dtype = cache_dtype;
  if (!elem_bytes(dtype) || !elem_bytes(q_dtype) || num_seqs < 0 || num_kv_heads < 1 ||
      num_heads % num_kv_heads || block_size < 1 || head_size % pack_x(dtype))
    return OR_ERR_ARG;
  for (int s = 0; s < num_seqs; ++s)
    if (seq_lens[s] < 1 || (int64_t)seq_lens[s] > (int64_t)max_blocks_per_seq * block_size)
      return OR_ERR_SEQ_LEN;
  const int G = num_heads / num_kv_heads;
  const int D = head_size;
  int status = OR_OK;
  const int64_t n_pairs = (int64_t)num_seqs * num_heads;

#pragma omp parallel for schedule(dynamic, 1)
  for (int64_t sh = 0; sh < n_pairs; ++sh) {
    const int s = (int)(sh / num_heads), h = (int)(sh % num_heads);
    const int L = seq_lens[s];
    const int kvh = h / G;
    double* K = (double*)malloc(sizeof(double) * (size_t)L * D);
    double* V = (double*)malloc(sizeof(double) * (size_t)L * D);
    double* z = (double*)malloc(sizeof(double) * (size_t)L);
    if (!K || !V || !z) {
#pragma omp critical
      status = OR_ERR_NOMEM;
      free(K); free(V); free(z);
      continue;
    }
    int st = gather_seq(K, V, k_cache, v_cache, block_tables + (int64_t)s * max_blocks_per_seq, L,
                        kvh, num_kv_heads, D, block_size, num_blocks, dtype, k_scale, v_scale);
    if (st != OR_OK) {
#pragma omp critical
      status = st;
      free(K); free(V); free(z);
      continue;
    }
    const int64_t qo = ((int64_t)s * num_heads + h) * D;
    /* scores */
    for (int t = 0; t < L; ++t) {
      double acc = 0.0;
      for (int d = 0; d < D; ++d) acc += load(q, qo + d, q_dtype) * K[(int64_t)t * D + d];
      z[t] = scale * acc;
    }
    /* softmax with the maximum subtracted */
    double m = z[0];
    for (int t = 1; t < L; ++t) if (z[t] > m) m = z[t];
    double Z = 0.0;
    for (int t = 0; t < L; ++t) { z[t] = exp(z[t] - m); Z += z[t]; }
    for (int t = 0; t < L; ++t) z[t] /= Z;
    if (weights)
      for (int t = 0; t < L; ++t) weights[sh * w_stride + t] = z[t];
    /* weighted sum of the value rows */
    for (int d = 0; d < D; ++d) {
      double acc = 0.0;
      for (int t = 0; t < L; ++t) acc += z[t] * V[(int64_t)t * D + d];
      out[qo + d] = acc;
    }
    free(K); free(V); free(z);
  }
  return status;
}

/*
 * Chunked prefill over the paged pool: the step before decode ([BHHXX] §2.3: a
 * prompt is processed, its K/V enter the cache, then tokens are generated one
 * at a time), read as causal attention of a chunk of new query tokens over the
 * sequence's cached history and the chunk itself.  For sequence s the cache
 * holds L = seq_lens[s] tokens after the chunk's write, the chunk is the
 * n = query_start_loc[s+1] - query_start_loc[s] tokens at positions L-n .. L-1,
 * and query token i (row query_start_loc[s] + i) at position p = L - n + i
 * attends to positions 0..p:
 *     z_t = scale * <q[row,h,:], K_s[t,:]>      t <= p
 *     out[row,h,:] = sum_t softmax(z)_t V_s[t,:]
 * q and out are [num_query_tokens, num_heads, head_size]; K_s, V_s as in decode.
 */
int oracle_prefill(double* out, const void* q, const void* k_cache, const void* v_cache,
                   const int32_t* block_tables, int max_blocks_per_seq, const int32_t* seq_lens,
                   const int32_t* query_start_loc, int num_seqs, int num_heads, int num_kv_heads,
                   int head_size, int block_size, int64_t num_blocks, double scale, int dtype) {
  if (!elem_bytes(dtype) || num_seqs < 0 || num_kv_heads < 1 || num_heads % num_kv_heads || block_size < 1 ||
      head_size % pack_x(dtype) || query_start_loc[0] != 0)
    return OR_ERR_ARG;
  for (int s = 0; s < num_seqs; ++s) {
    const int n = query_start_loc[s + 1] - query_start_loc[s];
    if (n < 0 || n > seq_lens[s] || seq_lens[s] < 1 ||
        (int64_t)seq_lens[s] > (int64_t)max_blocks_per_seq * block_size)
      return OR_ERR_SEQ_LEN;
  }
  const int G = num_heads / num_kv_heads;
  const int D = head_size;
  int status = OR_OK;
  const int64_t n_pairs = (int64_t)num_seqs * num_heads;

#pragma omp parallel for schedule(dynamic, 1)
  for (int64_t sh = 0; sh < n_pairs; ++sh) {
    const int s = (int)(sh / num_heads), h = (int)(sh % num_heads);
    const int L = seq_lens[s], n = query_start_loc[s + 1] - query_start_loc[s];
    if (n == 0) continue;
    double* K = (double*)malloc(sizeof(double) * (size_t)L * D);
    double* V = (double*)malloc(sizeof(double) * (size_t)L * D);
    double* z = (double*)malloc(sizeof(double) * (size_t)L);
    if (!K || !V || !z) {
#pragma omp critical
      status = OR_ERR_NOMEM;
      free(K); free(V); free(z);
      continue;
    }
    int st = gather_seq(K, V, k_cache, v_cache, block_tables + (int64_t)s * max_blocks_per_seq, L, h / G,
                        num_kv_heads, D, block_size, num_blocks, dtype, 1.0, 1.0);
    if (st != OR_OK) {
#pragma omp critical
      status = st;
      free(K); free(V); free(z);
      continue;
    }
    for (int i = 0; i < n; ++i) {
      const int p = L - n + i;  /* position of query token i */
      const int64_t qo = ((int64_t)(query_start_loc[s] + i) * num_heads + h) * D;
      for (int t = 0; t <= p; ++t) {
        double acc = 0.0;
        for (int d = 0; d < D; ++d) acc += load(q, qo + d, dtype) * K[(int64_t)t * D + d];
        z[t] = scale * acc;
      }
      double m = z[0];
      for (int t = 1; t <= p; ++t) if (z[t] > m) m = z[t];
      double Z = 0.0;
      for (int t = 0; t <= p; ++t) { z[t] = exp(z[t] - m); Z += z[t]; }
      for (int d = 0; d < D; ++d) {
        double acc = 0.0;
        for (int t = 0; t <= p; ++t) acc += z[t] * V[(int64_t)t * D + d];
        out[qo + d] = acc / Z;
      }
    }
    free(K); free(V); free(z);
  }
  return status;
}

/*
 * The decode definition above for a cache in the query's own dtype (no scales).
 */
int oracle_decode(double* out, double* weights, int64_t w_stride, const void* q,
                  const void* k_cache, const void* v_cache, const int32_t* block_tables,
                  int max_blocks_per_seq, const int32_t* seq_lens, int num_seqs, int num_heads,
                  int num_kv_heads, int head_size, int block_size, int64_t num_blocks,
                  double scale, int dtype) {
  return oracle_decode_scaled(out, weights, w_stride, q, k_cache, v_cache, block_tables, max_blocks_per_seq,
                              seq_lens, num_seqs, num_heads, num_kv_heads, head_size, block_size, num_blocks,
                              scale, dtype, dtype, 1.0, 1.0);
}
