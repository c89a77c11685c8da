"""pa_decode_noalloc, the decode entry point that allocates nothing.

Some callers cannot call cudaMalloc at the moment they decode: a serving process
that reserved its whole memory budget up front (weights plus the KV pool) and
allows no allocation afterwards, or a caller on a latency path where an
allocation may synchronize the device.  pa_decode_noalloc keeps the split-KV
scratch in a fixed array inside the library instead of a caller workspace.

These tests call it through the C ABI and check it against pa_decode (the entry
point that takes a caller workspace) on the same inputs over two calls in a row
-- the second call finds the first call's leftovers in the shared array.  Both
entry points run the same kernels on the same inputs and the output is
deterministic, so the two results must be equal bit for bit; one of them is
also checked against the CPU oracle within the parity tests' tolerance.  This
file is named so that pytest collects it last.
"""
import ctypes

import numpy as np
import pytest

import workloads as W
from helpers import as_f64, assert_close, oracle_out, oracle_pools, upload

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from paged_kv_cache_306_gb300 import build as pa_build
    pa_build.build()
    import paged_kv_cache_306_gb300 as pa
    return pa.load()


def _args(wl, t, out, partition_size):
    P = ctypes.c_void_p
    code = {"f32": 0, "f16": 1, "bf16": 2}[wl.dtype]
    head = [P(out.data_ptr()), P(t["q"].data_ptr()), P(t["k_cache"].data_ptr()), P(t["v_cache"].data_ptr()),
            P(t["block_tables"].data_ptr()), wl.max_blocks_per_seq, P(t["seq_lens"].data_ptr()), wl.num_seqs,
            wl.max_seq_len, wl.num_heads, wl.num_kv_heads, wl.head_size, wl.block_size, wl.num_blocks,
            ctypes.c_float(wl.scale), partition_size]
    return head, code


def _with_workspace(lib, wl, t, partition_size):
    out = torch.empty_like(t["q"])
    head, code = _args(wl, t, out, partition_size)
    need = lib.pa_decode_workspace_size(wl.num_seqs, wl.num_heads, wl.num_kv_heads, wl.head_size, wl.max_seq_len,
                                        wl.block_size, partition_size, code)
    assert need > 0, "the case must split, so that scratch is used"
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    assert lib.pa_decode(*head, ctypes.c_void_p(ws.data_ptr()), need, code, stream) == 0
    return out


def _no_alloc(lib, wl, t, partition_size):
    out = torch.empty_like(t["q"])
    head, code = _args(wl, t, out, partition_size)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    st = lib.pa_decode_noalloc(*head, code, stream)
    assert st == 0, lib.pa_last_error_message().decode()
    return out


def _device_error(lib):
    code = ctypes.c_int(-1)
    assert lib.pa_get_device_error(ctypes.byref(code), ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)) == 0
    return code.value


def test_no_alloc_matches_the_workspace_entry_point_on_two_calls_in_a_row(lib):
    a = W.make_private("noalloc-a", "f16", [3000, 700, 1, 4096, 1500, 17], 28, 4, 128, 16, seed=501,
                       poison=False, partition_size=256)
    b = W.make_private("noalloc-b", "bf16", [9000, 40, 2600], 32, 8, 128, 16, seed=502, poison=False,
                       partition_size=512)
    ta, tb = upload(a), upload(b)
    ref_a = _with_workspace(lib, a, ta, a.partition_size)
    ref_b = _with_workspace(lib, b, tb, b.partition_size)
    got_a = _no_alloc(lib, a, ta, a.partition_size)      # first call
    got_b = _no_alloc(lib, b, tb, b.partition_size)      # second call, same scratch
    torch.cuda.synchronize()
    assert _device_error(lib) == 0
    for wl, got, ref in ((a, got_a, ref_a), (b, got_b, ref_b)):
        assert torch.isfinite(got.float()).all()
        # same kernels, same inputs, deterministic output: equal bit for bit
        assert torch.equal(got.view(torch.int16), ref.view(torch.int16)), f"{wl.name}: differs from pa_decode"
    # and the result is the attention the oracle computes (the pools as uploaded: no write)
    k, v = oracle_pools(a, write=False)
    assert_close(as_f64(got_a), oracle_out(a, k, v), a.dtype, what="no-alloc decode vs the oracle")


def test_no_alloc_rejects_a_split_larger_than_its_scratch(lib):
    n0 = lib.pa_launch_count()
    # 1024 sequences x 16 kv heads with 16 query heads each: one partial slot per
    # (sequence, kv head) of 16 rows x 128 dims is far beyond 32 MiB
    need = lib.pa_decode_workspace_size(1024, 256, 16, 128, 4096, 16, 0, 1)
    assert need > 32 * 1024 * 1024
    # null pointers: the size check comes first, and without it pa_decode's null check would refuse
    st = lib.pa_decode_noalloc(None, None, None, None, None, 256, None, 1024, 4096, 256, 16, 128, 16,
                               100000, ctypes.c_float(0.1), 0, 1, None)
    assert st == 4                                       # PA_ERR_WORKSPACE, nothing enqueued
    assert b"32 MiB" in lib.pa_last_error_message() or b"holds" in lib.pa_last_error_message()
    assert lib.pa_launch_count() == n0
