"""CPU oracle for paged-attention decode -- TEST INFRASTRUCTURE ONLY.

Only the tests, the smoke check and the benchmark's CPU-baseline leg import this
package.  It wraps the fp64 C oracle (``pa_oracle.c``) with numpy arrays and
holds the pure-Python brute force (``brute.py``).  It shares no code with the
CUDA library.

Array conventions (numpy): fp32 caches are ``float32``, fp16 caches ``float16``,
bf16 caches ``uint16`` bit patterns, FP8 E4M3 caches ``uint8`` codes, fp64
caches ``float64``.  Every array must be C-contiguous.
"""
import ctypes
import os

import numpy as np

from . import build as _build

F32, F16, BF16, F64, FP8 = 0, 1, 2, 3, 4
DTYPE_CODES = {"f32": F32, "f16": F16, "bf16": BF16, "f64": F64, "fp8": FP8}

ERRORS = {
    1: "bad argument",
    2: "seq_len out of range",
    3: "block id outside the pool",
    4: "slot outside the pool",
    5: "duplicate slot",
    6: "out of memory",
}

_lib = None


class OracleError(RuntimeError):
    pass


def _load():
    global _lib
    if _lib is None:
        # PA_ORACLE_LIB lets the mutation tests load a deliberately broken copy
        path = os.environ.get("PA_ORACLE_LIB") or _build.build()
        lib = ctypes.CDLL(path)
        P = ctypes.c_void_p
        i64, i32, f64 = ctypes.c_int64, ctypes.c_int, ctypes.c_double
        lib.oracle_decode.argtypes = [P, P, i64, P, P, P, P, i32, P, i32, i32, i32, i32, i32, i64, f64, i32]
        lib.oracle_decode_scaled.argtypes = [P, P, i64, P, P, P, P, i32, P, i32, i32, i32, i32, i32, i64, f64, i32,
                                             i32, f64, f64]
        lib.oracle_reshape_and_cache_scaled.argtypes = [P, P, P, P, P, i64, i32, i32, i32, i64, i32, i32, f64, f64]
        lib.oracle_encode_e4m3.argtypes = [P, P, i64]
        lib.oracle_reshape_and_cache.argtypes = [P, P, P, P, P, i64, i32, i32, i32, i64, i32]
        lib.oracle_copy_blocks.argtypes = [P, P, P, i64, i32, i32, i32, i64, i32]
        lib.oracle_widen.argtypes = [P, P, i64, i32]
        lib.oracle_prefill.argtypes = [P, P, P, P, P, i32, P, P, i32, i32, i32, i32, i32, i64, f64, i32]
        for f in (lib.oracle_decode, lib.oracle_reshape_and_cache, lib.oracle_copy_blocks,
                  lib.oracle_widen, lib.oracle_num_threads, lib.oracle_elem_bytes, lib.oracle_pack_x,
                  lib.oracle_decode_scaled, lib.oracle_reshape_and_cache_scaled, lib.oracle_encode_e4m3,
                  lib.oracle_prefill):
            f.restype = ctypes.c_int
        lib.oracle_set_num_threads.argtypes = [i32]
        lib.oracle_set_num_threads.restype = None
        lib.oracle_elem_bytes.argtypes = [i32]
        lib.oracle_pack_x.argtypes = [i32]
        _lib = lib
    return _lib


def _ptr(a):
    if a is None:
        return None
    if not a.flags["C_CONTIGUOUS"]:
        raise ValueError("oracle arrays must be C-contiguous")
    return a.ctypes.data_as(ctypes.c_void_p)


def _check(status):
    if status != 0:
        raise OracleError(ERRORS.get(status, f"oracle status {status}"))


def _code(dtype):
    return DTYPE_CODES[dtype] if isinstance(dtype, str) else int(dtype)


def num_threads():
    return _load().oracle_num_threads()


def set_num_threads(n):
    """Threads the oracle's parallel loops use from now on."""
    _load().oracle_set_num_threads(int(n))


def pack_x(dtype):
    """x = 16 / element size (Reading vLLM's PagedAttention kernel, section 3.1)."""
    return _load().oracle_pack_x(_code(dtype))


def widen(a, dtype):
    """Widen an array of `dtype` to float64 exactly."""
    out = np.empty(a.size, dtype=np.float64)
    _check(_load().oracle_widen(_ptr(out), _ptr(np.ascontiguousarray(a)), a.size, _code(dtype)))
    return out.reshape(a.shape)


def decode(q, k_cache, v_cache, block_tables, seq_lens, scale, dtype, num_kv_heads=None,
           return_weights=False, q_dtype=None, k_scale=1.0, v_scale=1.0):
    """out[s, h, :] = softmax(scale * q K_s^T) V_s in fp64 (see pa_oracle.c).

    q: [S, H, D]; k_cache: [NB, Hkv, D/x, bs, x]; v_cache: [NB, Hkv, D, bs];
    block_tables: int32 [S, MB]; seq_lens: int32 [S].  `dtype` is the cache dtype;
    q has `q_dtype` (default: the cache dtype).  A quantised cache reads back as
    code * k_scale (K) and code * v_scale (V).
    """
    code = _code(dtype)
    qcode = code if q_dtype is None else _code(q_dtype)
    S, H, D = q.shape
    NB, Hkv = k_cache.shape[0], k_cache.shape[1]
    if num_kv_heads is not None and num_kv_heads != Hkv:
        raise ValueError("num_kv_heads does not match the cache")
    bs = v_cache.shape[3]
    bt = np.ascontiguousarray(block_tables, dtype=np.int32)
    sl = np.ascontiguousarray(seq_lens, dtype=np.int32)
    out = np.zeros((S, H, D), dtype=np.float64)
    w = None
    w_stride = 0
    if return_weights:
        w_stride = int(sl.max()) if S else 0
        w = np.full((S, H, w_stride), np.nan, dtype=np.float64)
    st = _load().oracle_decode_scaled(_ptr(out), _ptr(w), w_stride, _ptr(q), _ptr(k_cache), _ptr(v_cache),
                                      _ptr(bt), bt.shape[1], _ptr(sl), S, H, Hkv, D, bs, NB, float(scale), qcode,
                                      code, float(k_scale), float(v_scale))
    _check(st)
    return (out, w) if return_weights else out


def prefill(q, k_cache, v_cache, block_tables, seq_lens, query_start_loc, scale, dtype):
    """Chunked prefill (see pa_oracle.c): query token i of sequence s, at position
    seq_lens[s] - n_s + i, attends causally to positions 0..itself; fp64 out [T_q, H, D]."""
    code = _code(dtype)
    T, H, D = q.shape
    NB, Hkv = k_cache.shape[0], k_cache.shape[1]
    bs = v_cache.shape[3]
    bt = np.ascontiguousarray(block_tables, dtype=np.int32)
    sl = np.ascontiguousarray(seq_lens, dtype=np.int32)
    qsl = np.ascontiguousarray(query_start_loc, dtype=np.int32)
    if qsl[-1] != T:
        raise ValueError("query_start_loc does not end at the number of query tokens")
    out = np.zeros((T, H, D), dtype=np.float64)
    _check(_load().oracle_prefill(_ptr(out), _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(bt), bt.shape[1], _ptr(sl),
                                  _ptr(qsl), len(sl), H, Hkv, D, bs, NB, float(scale), code))
    return out


def encode_e4m3(x):
    """E4M3 codes (uint8) of float64 values: nearest, ties to even, clamped to +-448."""
    x = np.ascontiguousarray(x, dtype=np.float64)
    out = np.empty(x.shape, dtype=np.uint8)
    _check(_load().oracle_encode_e4m3(_ptr(out), _ptr(x), x.size))
    return out


def reshape_and_cache_scaled(key, value, k_cache, v_cache, slot_mapping, key_dtype, cache_dtype, k_scale,
                             v_scale):
    """Write path into a possibly quantised cache (codes of x / scale for FP8)."""
    sm = np.ascontiguousarray(slot_mapping, dtype=np.int64)
    T, Hkv, D = key.shape
    NB, bs = v_cache.shape[0], v_cache.shape[3]
    _check(_load().oracle_reshape_and_cache_scaled(_ptr(key), _ptr(value), _ptr(k_cache), _ptr(v_cache), _ptr(sm),
                                                   T, Hkv, D, bs, NB, _code(key_dtype), _code(cache_dtype),
                                                   float(k_scale), float(v_scale)))


def reshape_and_cache(key, value, k_cache, v_cache, slot_mapping, dtype):
    """Scatter key/value [T, Hkv, D] into the pools in place (byte copy)."""
    sm = np.ascontiguousarray(slot_mapping, dtype=np.int64)
    T, Hkv, D = key.shape
    NB, bs = v_cache.shape[0], v_cache.shape[3]
    _check(_load().oracle_reshape_and_cache(_ptr(key), _ptr(value), _ptr(k_cache), _ptr(v_cache),
                                            _ptr(sm), T, Hkv, D, bs, NB, _code(dtype)))


def copy_blocks(k_cache, v_cache, src_dst, dtype):
    """Copy whole blocks src -> dst (K and V, every kv head) in place."""
    sd = np.ascontiguousarray(src_dst, dtype=np.int64).reshape(-1, 2)
    NB, Hkv, D, bs = v_cache.shape
    _check(_load().oracle_copy_blocks(_ptr(k_cache), _ptr(v_cache), _ptr(sd), sd.shape[0],
                                      Hkv, D, bs, NB, _code(dtype)))
