"""ctypes binding of libpa.so: argument marshalling only.

Each function takes torch tensors, checks that they match the call's contract
(device, dtype, shape, contiguity), and passes raw pointers, sizes and the
current CUDA stream to the C entry point of the same name (include/pa.h).
Every step of the computation runs in the library's kernels; there is no
fallback path, and a missing library is an error.
"""
import ctypes
import os

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "_build", "libpa.so")

(PA_OK, PA_ERR_INVALID_ARG, PA_ERR_UNSUPPORTED, PA_ERR_ALIGNMENT, PA_ERR_WORKSPACE, PA_ERR_CUDA,
 PA_ERR_OUT_OF_BLOCKS) = range(7)
PA_F32, PA_F16, PA_BF16, PA_FP8_E4M3 = 0, 1, 2, 3
PARTITION_NONE = 0
PARTITION_AUTO = -1
DEVICE_ERRORS = {0: "none", 1: "block id outside the pool", 2: "seq_len outside [1, max_seq_len]",
                 3: "slot outside the pool", 4: "pipeline wait timed out", 5: "copy id outside the pool",
                 6: "a block declared shared differs between two tables"}

_lib = None


class PAError(RuntimeError):
    def __init__(self, status, message):
        super().__init__(message)
        self.status = status


def load():
    """Load libpa.so (built by ``python -m paged_kv_cache_306_gb300.build``)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise PAError(-1, f"{LIB_PATH} is missing: build it with `python -m paged_kv_cache_306_gb300.build`")
    lib = ctypes.CDLL(LIB_PATH)
    P, i32, i64, sz, f32 = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_size_t, ctypes.c_float
    lib.pa_status_string.argtypes = [i32]
    lib.pa_status_string.restype = ctypes.c_char_p
    lib.pa_last_error_message.argtypes = []
    lib.pa_last_error_message.restype = ctypes.c_char_p
    lib.pa_reshape_and_cache.argtypes = [P, P, P, P, P, i64, i32, i32, i32, i64, i32, P]
    lib.pa_copy_blocks.argtypes = [P, P, P, i64, i32, i32, i32, i64, i32, P]
    lib.pa_decode_plan_partition.argtypes = [i32, i32, i32, i32, i32, i32, i32]
    lib.pa_decode_plan_partition.restype = i32
    lib.pa_decode_workspace_size.argtypes = [i32, i32, i32, i32, i32, i32, i32, i32]
    lib.pa_decode_workspace_size.restype = sz
    lib.pa_decode.argtypes = [P, P, P, P, P, i32, P, i32, i32, i32, i32, i32, i32, i64, f32, i32, P, sz, i32, P]
    lib.pa_reshape_and_cache_scaled.argtypes = [P, P, P, P, P, i64, i32, i32, i32, i64, i32, i32, f32, f32, P]
    lib.pa_reshape_and_cache_scaled.restype = i32
    lib.pa_decode_scaled.argtypes = [P, P, P, P, P, i32, P, i32, i32, i32, i32, i32, i32, i64, f32, i32, P, sz, i32,
                                     i32, f32, f32, P]
    lib.pa_decode_scaled.restype = i32
    lib.pa_decode_noalloc.argtypes = [P, P, P, P, P, i32, P, i32, i32, i32, i32, i32, i32, i64, f32, i32, i32, P]
    lib.pa_decode_noalloc.restype = i32
    lib.pa_get_device_error.argtypes = [ctypes.POINTER(i32), P]
    lib.pa_launch_count.argtypes = []
    lib.pa_launch_count.restype = ctypes.c_uint64
    lib.pa_set_test_wait_limit.argtypes = [ctypes.c_uint64]
    lib.pa_set_test_wait_limit.restype = None
    lib.pa_decode_shared.argtypes = [P, P, P, P, P, P, P, i64, P, i32, P, P, P, i32, i32, i32, i32, i32, i32, i64,
                                     f32, i32, P, sz, i32, i32, f32, f32, P]
    lib.pa_decode_shared.restype = i32
    lib.pa_decode_shared_workspace_size.argtypes = [i32, i32, i32, i32, i32, i32, i32, i32]
    lib.pa_decode_shared_workspace_size.restype = sz
    for f in (lib.pa_reshape_and_cache, lib.pa_copy_blocks, lib.pa_decode, lib.pa_get_device_error):
        f.restype = i32
    lib.pa_prefill.argtypes = [P, P, P, P, P, i32, P, P, i32, i32, i32, i32, i32, i32, i32, i64, f32, i32, P]
    lib.pa_prefill.restype = i32
    lib.pa_decode_step.argtypes = [P, P, P, P, P, P, P, i64, P, i32, P, i32, i32, i32, i32, i32, i32, i64, f32, i32,
                                   P, sz, i32, P]
    lib.pa_decode_step.restype = i32
    lib.pa_decode_step_scaled.argtypes = [P, P, P, P, P, P, P, i64, P, i32, P, i32, i32, i32, i32, i32, i32, i64,
                                          f32, i32, P, sz, i32, i32, f32, f32, P]
    lib.pa_decode_step_scaled.restype = i32
    # host-side block manager (include/pa_block_manager.h)
    lib.pa_bm_create.argtypes = [i64, i32, ctypes.POINTER(P)]
    lib.pa_bm_destroy.argtypes = [P]
    lib.pa_bm_destroy.restype = None
    lib.pa_bm_num_free_blocks.argtypes = [P]
    lib.pa_bm_num_free_blocks.restype = i64
    lib.pa_bm_add_sequence.argtypes = [P, i64, i64, P]
    lib.pa_bm_fork.argtypes = [P, i64, i64]
    lib.pa_bm_free_sequence.argtypes = [P, i64]
    lib.pa_bm_append_tokens.argtypes = [P, P, i32, P, P, i64, ctypes.POINTER(i64)]
    lib.pa_bm_seq_len.argtypes = [P, i64, ctypes.POINTER(i64)]
    lib.pa_bm_block_tables.argtypes = [P, P, i32, P, i32, P]
    lib.pa_bm_refcount.argtypes = [P, i64, ctypes.POINTER(i32)]
    lib.pa_bm_prefix_groups.argtypes = [P, P, i32, P, P]
    lib.pa_bm_prefix_groups.restype = i32
    for f in (lib.pa_bm_create, lib.pa_bm_add_sequence, lib.pa_bm_fork, lib.pa_bm_free_sequence,
              lib.pa_bm_append_tokens, lib.pa_bm_seq_len, lib.pa_bm_block_tables, lib.pa_bm_refcount):
        f.restype = i32
    _lib = lib
    return lib


def check(status):
    if status != PA_OK:
        lib = load()
        name = lib.pa_status_string(status).decode()
        msg = lib.pa_last_error_message().decode()
        raise PAError(status, f"{name}: {msg}")


def dtype_code(torch_dtype):
    import torch
    codes = {torch.float32: PA_F32, torch.float16: PA_F16, torch.bfloat16: PA_BF16,
             torch.float8_e4m3fn: PA_FP8_E4M3}
    if torch_dtype not in codes:
        raise PAError(PA_ERR_UNSUPPORTED, f"unsupported dtype {torch_dtype}")
    return codes[torch_dtype]


def _stream(stream):
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None and t.numel() else ctypes.c_void_p(0)


def _need_cuda(name, t, dtype=None, dims=None):
    if not t.is_cuda:
        raise PAError(PA_ERR_INVALID_ARG, f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise PAError(PA_ERR_INVALID_ARG, f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise PAError(PA_ERR_INVALID_ARG, f"{name} has dtype {t.dtype}, expected {dtype}")
    if dims is not None and t.dim() != dims:
        raise PAError(PA_ERR_INVALID_ARG, f"{name} must have {dims} dims")


def _workspace(need, workspace, device, stream):
    """The caller's workspace when it is large enough, else a fresh one from torch's
    allocator.  A fresh one used on a stream other than the current one is recorded
    on that stream, so the allocator does not hand its memory out again before the
    kernels that use it have finished there."""
    import torch
    if not need or (workspace is not None and workspace.numel() * workspace.element_size() >= need):
        return workspace
    ws = torch.empty(need, dtype=torch.uint8, device=device)
    if stream is not None and stream != torch.cuda.current_stream(device):
        ws.record_stream(stream)
    return ws


def pa_reshape_and_cache(key, value, k_cache, v_cache, slot_mapping, stream=None):
    """Scatter key/value [T, Hkv, D] into the paged pools through slot_mapping (int64 [T])."""
    import torch
    for n, t in (("key", key), ("value", value), ("k_cache", k_cache), ("v_cache", v_cache)):
        _need_cuda(n, t, k_cache.dtype)
    _need_cuda("slot_mapping", slot_mapping, torch.int64, 1)
    T, hkv, d = key.shape
    nb, bs = v_cache.shape[0], v_cache.shape[3]
    check(load().pa_reshape_and_cache(_ptr(key), _ptr(value), _ptr(k_cache), _ptr(v_cache), _ptr(slot_mapping),
                                      T, hkv, d, bs, nb, dtype_code(k_cache.dtype), _stream(stream)))


def pa_reshape_and_cache_scaled(key, value, k_cache, v_cache, slot_mapping, k_scale, v_scale, stream=None):
    """Write path into a cache of another dtype: for an FP8 E4M3 cache (torch.float8_e4m3fn)
    each element is stored as the code of x / k_scale (x / v_scale)."""
    import torch
    for n, t in (("key", key), ("value", value)):
        _need_cuda(n, t, key.dtype)
    for n, t in (("k_cache", k_cache), ("v_cache", v_cache)):
        _need_cuda(n, t, k_cache.dtype)
    _need_cuda("slot_mapping", slot_mapping, torch.int64, 1)
    T, hkv, d = key.shape
    nb, bs = v_cache.shape[0], v_cache.shape[3]
    check(load().pa_reshape_and_cache_scaled(_ptr(key), _ptr(value), _ptr(k_cache), _ptr(v_cache),
                                             _ptr(slot_mapping), T, hkv, d, bs, nb, dtype_code(key.dtype),
                                             dtype_code(k_cache.dtype), float(k_scale), float(v_scale),
                                             _stream(stream)))


def pa_copy_blocks(k_cache, v_cache, src_dst, stream=None):
    """Copy whole physical blocks: src_dst is int64 [n, 2] of (src, dst)."""
    import torch
    _need_cuda("k_cache", k_cache)
    _need_cuda("v_cache", v_cache, k_cache.dtype)
    _need_cuda("src_dst", src_dst, torch.int64)
    nb, hkv, d, bs = v_cache.shape
    check(load().pa_copy_blocks(_ptr(k_cache), _ptr(v_cache), _ptr(src_dst), src_dst.numel() // 2, hkv, d, bs, nb,
                                dtype_code(k_cache.dtype), _stream(stream)))


def pa_decode_plan_partition(num_seqs, num_heads, num_kv_heads, head_size, max_seq_len, block_size, dtype):
    return load().pa_decode_plan_partition(num_seqs, num_heads, num_kv_heads, head_size, max_seq_len, block_size,
                                           dtype if isinstance(dtype, int) else dtype_code(dtype))


def pa_decode_workspace_size(num_seqs, num_heads, num_kv_heads, head_size, max_seq_len, block_size, partition_size,
                             dtype):
    return load().pa_decode_workspace_size(num_seqs, num_heads, num_kv_heads, head_size, max_seq_len, block_size,
                                           partition_size, dtype if isinstance(dtype, int) else dtype_code(dtype))


def pa_decode(out, q, k_cache, v_cache, block_tables, seq_lens, scale, max_seq_len,
              partition_size=PARTITION_AUTO, workspace=None, stream=None):
    """Decode attention over the paged pool; writes out [S, H, D].

    max_seq_len is a host-side bound on seq_lens.  When the call needs a
    workspace and none is given, one is taken from torch's allocator.
    Returns the workspace tensor used (or None).
    """
    import torch
    dt = q.dtype
    _need_cuda("q", q, dt, 3)
    _need_cuda("out", out, dt, 3)
    _need_cuda("k_cache", k_cache, dt, 5)
    _need_cuda("v_cache", v_cache, dt, 4)
    _need_cuda("block_tables", block_tables, torch.int32, 2)
    _need_cuda("seq_lens", seq_lens, torch.int32, 1)
    S, H, D = q.shape
    nb, hkv, _, bs = v_cache.shape
    code = dtype_code(dt)
    lib = load()
    need = lib.pa_decode_workspace_size(S, H, hkv, D, max_seq_len, bs, partition_size, code)
    workspace = _workspace(need, workspace, q.device, stream)
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    check(lib.pa_decode(_ptr(out), _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables),
                        block_tables.shape[1], _ptr(seq_lens), S, max_seq_len, H, hkv, D, bs, nb, float(scale),
                        partition_size, _ptr(workspace), ws_bytes, code, _stream(stream)))
    return workspace


def pa_decode_scaled(out, q, k_cache, v_cache, block_tables, seq_lens, scale, max_seq_len, k_scale, v_scale,
                     partition_size=PARTITION_AUTO, workspace=None, stream=None):
    """pa_decode over a cache whose dtype differs from q's (FP8 E4M3 read back as code * scale)."""
    import torch
    dt = q.dtype
    _need_cuda("q", q, dt, 3)
    _need_cuda("out", out, dt, 3)
    _need_cuda("k_cache", k_cache, None, 5)
    _need_cuda("v_cache", v_cache, k_cache.dtype, 4)
    _need_cuda("block_tables", block_tables, torch.int32, 2)
    _need_cuda("seq_lens", seq_lens, torch.int32, 1)
    S, H, D = q.shape
    nb, hkv, _, bs = v_cache.shape
    cc = dtype_code(k_cache.dtype)
    lib = load()
    need = lib.pa_decode_workspace_size(S, H, hkv, D, max_seq_len, bs, partition_size, cc)
    workspace = _workspace(need, workspace, q.device, stream)
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    check(lib.pa_decode_scaled(_ptr(out), _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables),
                               block_tables.shape[1], _ptr(seq_lens), S, max_seq_len, H, hkv, D, bs, nb, float(scale),
                               partition_size, _ptr(workspace), ws_bytes, dtype_code(dt), cc, float(k_scale),
                               float(v_scale), _stream(stream)))
    return workspace


def pa_decode_step(out, q, key, value, k_cache, v_cache, src_dst, block_tables, seq_lens, scale, max_seq_len,
                   partition_size=PARTITION_AUTO, workspace=None, stream=None):
    """One fused generation step: copy the blocks src_dst (int64 [n, 2], or None), write
    each sequence's new token key/value [S, Hkv, D] at position seq_lens[s] - 1, decode.
    Returns the workspace tensor used (or None)."""
    import torch
    dt = q.dtype
    _need_cuda("q", q, dt, 3)
    _need_cuda("out", out, dt, 3)
    _need_cuda("key", key, dt, 3)
    _need_cuda("value", value, dt, 3)
    _need_cuda("k_cache", k_cache, dt, 5)
    _need_cuda("v_cache", v_cache, dt, 4)
    _need_cuda("block_tables", block_tables, torch.int32, 2)
    _need_cuda("seq_lens", seq_lens, torch.int32, 1)
    npairs = 0
    if src_dst is not None:
        _need_cuda("src_dst", src_dst, torch.int64)
        npairs = src_dst.numel() // 2
    S, H, D = q.shape
    nb, hkv, _, bs = v_cache.shape
    if key.shape != (S, hkv, D) or value.shape != (S, hkv, D):
        raise ValueError(f"key/value must be [{S}, {hkv}, {D}]")
    code = dtype_code(dt)
    lib = load()
    need = lib.pa_decode_workspace_size(S, H, hkv, D, max_seq_len, bs, partition_size, code)
    workspace = _workspace(need, workspace, q.device, stream)
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    check(lib.pa_decode_step(_ptr(out), _ptr(q), _ptr(key), _ptr(value), _ptr(k_cache), _ptr(v_cache),
                             _ptr(src_dst) if npairs else None, npairs, _ptr(block_tables), block_tables.shape[1],
                             _ptr(seq_lens), S, max_seq_len, H, hkv, D, bs, nb, float(scale), partition_size,
                             _ptr(workspace), ws_bytes, code, _stream(stream)))
    return workspace


def pa_decode_step_scaled(out, q, key, value, k_cache, v_cache, src_dst, block_tables, seq_lens, scale,
                          max_seq_len, k_scale, v_scale, partition_size=PARTITION_AUTO, workspace=None, stream=None):
    """pa_decode_step over a cache whose dtype differs from q's: an FP8 E4M3 pool takes the
    new key/value rows in q's dtype, stores their codes of x / scale and decodes as
    pa_decode_scaled does."""
    import torch
    dt = q.dtype
    _need_cuda("q", q, dt, 3)
    _need_cuda("out", out, dt, 3)
    _need_cuda("key", key, dt, 3)
    _need_cuda("value", value, dt, 3)
    _need_cuda("k_cache", k_cache, None, 5)
    _need_cuda("v_cache", v_cache, k_cache.dtype, 4)
    _need_cuda("block_tables", block_tables, torch.int32, 2)
    _need_cuda("seq_lens", seq_lens, torch.int32, 1)
    npairs = 0
    if src_dst is not None:
        _need_cuda("src_dst", src_dst, torch.int64)
        npairs = src_dst.numel() // 2
    S, H, D = q.shape
    nb, hkv, _, bs = v_cache.shape
    if key.shape != (S, hkv, D) or value.shape != (S, hkv, D):
        raise ValueError(f"key/value must be [{S}, {hkv}, {D}]")
    cc = dtype_code(k_cache.dtype)
    lib = load()
    need = lib.pa_decode_workspace_size(S, H, hkv, D, max_seq_len, bs, partition_size, cc)
    workspace = _workspace(need, workspace, q.device, stream)
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    check(lib.pa_decode_step_scaled(_ptr(out), _ptr(q), _ptr(key), _ptr(value), _ptr(k_cache), _ptr(v_cache),
                                    _ptr(src_dst) if npairs else None, npairs, _ptr(block_tables),
                                    block_tables.shape[1], _ptr(seq_lens), S, max_seq_len, H, hkv, D, bs, nb,
                                    float(scale), partition_size, _ptr(workspace), ws_bytes, dtype_code(dt), cc,
                                    float(k_scale), float(v_scale), _stream(stream)))
    return workspace


def pa_decode_shared_workspace_size(num_seqs, num_heads, num_kv_heads, head_size, max_seq_len, block_size,
                                    partition_size, cache_dtype):
    return load().pa_decode_shared_workspace_size(num_seqs, num_heads, num_kv_heads, head_size, max_seq_len,
                                                  block_size, partition_size,
                                                  cache_dtype if isinstance(cache_dtype, int) else dtype_code(cache_dtype))


def pa_decode_shared(out, q, key, value, k_cache, v_cache, src_dst, block_tables, seq_lens, prefix_group,
                     prefix_blocks, scale, max_seq_len, k_scale=1.0, v_scale=1.0, partition_size=PARTITION_AUTO,
                     workspace=None, stream=None):
    """Decode (key/value given: the whole fused step) over sequences that share prefix
    blocks: prefix_group (int32 [S], runs of equal values) and prefix_blocks (int32 [S],
    the leading blocks each sequence holds of its group's common prefix) describe the
    sharing; each shared block is read once per cluster of sequences that hold it.
    Returns the workspace tensor used (or None)."""
    import torch
    dt = q.dtype
    _need_cuda("q", q, dt, 3)
    _need_cuda("out", out, dt, 3)
    _need_cuda("k_cache", k_cache, None, 5)
    _need_cuda("v_cache", v_cache, k_cache.dtype, 4)
    _need_cuda("block_tables", block_tables, torch.int32, 2)
    _need_cuda("seq_lens", seq_lens, torch.int32, 1)
    _need_cuda("prefix_group", prefix_group, torch.int32, 1)
    _need_cuda("prefix_blocks", prefix_blocks, torch.int32, 1)
    S, H, D = q.shape
    nb, hkv, _, bs = v_cache.shape
    if prefix_group.numel() != S or prefix_blocks.numel() != S:
        raise PAError(PA_ERR_INVALID_ARG, "prefix_group and prefix_blocks must have num_seqs entries")
    npairs = 0
    if key is not None:
        _need_cuda("key", key, dt, 3)
        _need_cuda("value", value, dt, 3)
        if key.shape != (S, hkv, D) or value.shape != (S, hkv, D):
            raise ValueError(f"key/value must be [{S}, {hkv}, {D}]")
        if src_dst is not None:
            _need_cuda("src_dst", src_dst, torch.int64)
            npairs = src_dst.numel() // 2
    elif src_dst is not None and src_dst.numel():
        raise PAError(PA_ERR_INVALID_ARG, "block copies come with a step's new tokens (key, value)")
    cc = dtype_code(k_cache.dtype)
    lib = load()
    need = lib.pa_decode_shared_workspace_size(S, H, hkv, D, max_seq_len, bs, partition_size, cc)
    workspace = _workspace(need, workspace, q.device, stream)
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    check(lib.pa_decode_shared(_ptr(out), _ptr(q), _ptr(key), _ptr(value), _ptr(k_cache), _ptr(v_cache),
                               _ptr(src_dst) if npairs else None, npairs, _ptr(block_tables), block_tables.shape[1],
                               _ptr(seq_lens), _ptr(prefix_group), _ptr(prefix_blocks), S, max_seq_len, H, hkv, D,
                               bs, nb, float(scale), partition_size, _ptr(workspace), ws_bytes, dtype_code(dt), cc,
                               float(k_scale), float(v_scale), _stream(stream)))
    return workspace


def pa_prefill(out, q, k_cache, v_cache, block_tables, seq_lens, query_start_loc, scale, max_seq_len, stream=None):
    """Chunked prefill: query rows query_start_loc[s] .. query_start_loc[s+1]-1 are the last
    tokens of sequence s (seq_lens[s] tokens in the cache, theirs included) and attend
    causally; writes out [num_query_tokens, H, D]."""
    import torch
    dt = q.dtype
    _need_cuda("q", q, dt, 3)
    _need_cuda("out", out, dt, 3)
    _need_cuda("k_cache", k_cache, dt, 5)
    _need_cuda("v_cache", v_cache, dt, 4)
    _need_cuda("block_tables", block_tables, torch.int32, 2)
    _need_cuda("seq_lens", seq_lens, torch.int32, 1)
    _need_cuda("query_start_loc", query_start_loc, torch.int32, 1)
    T, H, D = q.shape
    nb, hkv, _, bs = v_cache.shape
    S = seq_lens.numel()
    if query_start_loc.numel() != S + 1:
        raise PAError(PA_ERR_INVALID_ARG, "query_start_loc must have num_seqs + 1 entries")
    check(load().pa_prefill(_ptr(out), _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables),
                            block_tables.shape[1], _ptr(seq_lens), _ptr(query_start_loc), S, T, max_seq_len, H, hkv,
                            D, bs, nb, float(scale), dtype_code(dt), _stream(stream)))


def pa_get_device_error(stream=None):
    """Read and clear the first device-side error (0 if none); synchronizes the stream."""
    code = ctypes.c_int(0)
    check(load().pa_get_device_error(ctypes.byref(code), _stream(stream)))
    return code.value


def pa_launch_count():
    return load().pa_launch_count()


def pa_set_test_wait_limit(nanoseconds):
    """Timeout-path test only: while > 0, the kernels' first pipeline wait runs out after
    this many nanoseconds on a barrier nothing completes (0 restores normal operation)."""
    load().pa_set_test_wait_limit(int(nanoseconds))


class BlockManager:
    """The library's host-side block manager (include/pa_block_manager.h): free list,
    reference counts, per-sequence block lists, fork and copy-on-write.  Arrays in
    and out are numpy (host memory); nothing here touches the GPU."""

    def __init__(self, num_blocks, block_size):
        import numpy  # noqa: F401  (arrays below)
        self._lib = load()
        h = ctypes.c_void_p()
        check(self._lib.pa_bm_create(int(num_blocks), int(block_size), ctypes.byref(h)))
        self._h = h
        self.num_blocks, self.block_size = int(num_blocks), int(block_size)

    def close(self):
        if getattr(self, "_h", None) is not None and self._h.value:
            self._lib.pa_bm_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    @property
    def num_free_blocks(self):
        return self._lib.pa_bm_num_free_blocks(self._h)

    def add_sequence(self, seq_id, num_tokens):
        """A new sequence of num_tokens tokens; returns their slots (int64)."""
        import numpy as np
        slots = np.empty(int(num_tokens), np.int64)
        check(self._lib.pa_bm_add_sequence(self._h, int(seq_id), int(num_tokens),
                                           slots.ctypes.data if num_tokens else None))
        return slots

    def fork(self, parent_id, child_id):
        check(self._lib.pa_bm_fork(self._h, int(parent_id), int(child_id)))

    def free_sequence(self, seq_id):
        check(self._lib.pa_bm_free_sequence(self._h, int(seq_id)))

    def append_tokens(self, seq_ids):
        """One new token per listed sequence: returns (slot_mapping int64 [n], copies int64 [k, 2])."""
        import numpy as np
        ids = np.ascontiguousarray(seq_ids, np.int64)
        n = len(ids)
        slots = np.empty(n, np.int64)
        copies = np.empty((max(n, 1), 2), np.int64)
        nc = ctypes.c_int64(0)
        check(self._lib.pa_bm_append_tokens(self._h, ids.ctypes.data if n else None, n,
                                            slots.ctypes.data if n else None, copies.ctypes.data, max(n, 1),
                                            ctypes.byref(nc)))
        return slots, copies[:nc.value].copy()

    def seq_len(self, seq_id):
        n = ctypes.c_int64(0)
        check(self._lib.pa_bm_seq_len(self._h, int(seq_id), ctypes.byref(n)))
        return n.value

    def block_tables(self, seq_ids, max_blocks_per_seq):
        """(block_tables int32 [n, max_blocks_per_seq] with -1 past the end, seq_lens int32 [n])."""
        import numpy as np
        ids = np.ascontiguousarray(seq_ids, np.int64)
        n = len(ids)
        bt = np.empty((max(n, 1), int(max_blocks_per_seq)), np.int32)
        sl = np.empty(max(n, 1), np.int32)
        check(self._lib.pa_bm_block_tables(self._h, ids.ctypes.data if n else None, n, bt.ctypes.data,
                                           int(max_blocks_per_seq), sl.ctypes.data))
        return bt[:n].copy(), sl[:n].copy()

    def prefix_groups(self, seq_ids):
        """(prefix_group, prefix_blocks), int32 [n] each: pa_decode_shared's description of
        which listed sequences share prefix blocks (runs of one fork family)."""
        import numpy as np
        ids = np.ascontiguousarray(seq_ids, np.int64)
        n = len(ids)
        grp = np.empty(max(n, 1), np.int32)
        blk = np.empty(max(n, 1), np.int32)
        check(self._lib.pa_bm_prefix_groups(self._h, ids.ctypes.data if n else None, n, grp.ctypes.data,
                                            blk.ctypes.data))
        return grp[:n].copy(), blk[:n].copy()

    def refcount(self, block):
        r = ctypes.c_int(0)
        check(self._lib.pa_bm_refcount(self._h, int(block), ctypes.byref(r)))
        return r.value
