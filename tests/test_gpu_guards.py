"""Outputs written into the middle of larger buffers whose ends are filled with
NaN bytes: every call must leave those guard rows byte for byte as they were (no
write past the output it was given), and the rows in between must still match
the oracle."""
import zlib

import numpy as np
import pytest

import workloads as W
from helpers import as_f64, assert_close, oracle_out, oracle_pools, upload

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

GUARD = 2  # rows of guard on each side


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import paged_kv_cache_306_gb300 as pa
    pa.load()


def guarded_like(t):
    """A [GUARD + n + GUARD, ...] buffer of 0xFF bytes and its middle rows, shaped like t."""
    big = torch.empty((t.shape[0] + 2 * GUARD,) + tuple(t.shape[1:]), dtype=t.dtype, device=t.device)
    big.view(torch.uint8).fill_(0xFF)
    return big, big[GUARD:GUARD + t.shape[0]]


def guards_intact(big):
    b = big.view(torch.uint8)
    return bool((b[:GUARD] == 0xFF).all()) and bool((b[-GUARD:] == 0xFF).all())


@pytest.mark.parametrize("dtype,G,bs,part", [("f16", 7, 16, -1), ("bf16", 4, 32, 32), ("f32", 1, 16, 0),
                                             ("f16", 16, 16, 64)])
def test_decode_writes_only_its_output_rows(dtype, G, bs, part):
    import paged_kv_cache_306_gb300 as pa
    rng = np.random.default_rng(zlib.crc32(repr(("guard", dtype, G, bs, part)).encode()))
    wl = W.make_private("guard", dtype, [1, bs + 1, 300, 1200] + list(rng.integers(2, 700, size=4)), 2 * G, 2, 128,
                        bs, seed=int(rng.integers(1 << 30)), partition_size=part)
    t = upload(wl)
    pa.pa_reshape_and_cache(t["key"], t["value"], t["k_cache"], t["v_cache"], t["slot_mapping"])
    big, out = guarded_like(t["q"])
    pa.pa_decode(out, t["q"], t["k_cache"], t["v_cache"], t["block_tables"], t["seq_lens"], wl.scale, wl.max_seq_len,
                 part)
    assert pa.pa_get_device_error() == 0
    assert guards_intact(big)
    k, v = oracle_pools(wl)
    assert_close(as_f64(out), oracle_out(wl, k, v), dtype, with_rounding=True)


def test_fp8_decode_writes_only_its_output_rows():
    import paged_kv_cache_306_gb300 as pa
    wl = W.make_private("guard8", "fp8", [5, 17, 400, 999], 8, 2, 128, 16, seed=7, partition_size=-1, q_dtype="bf16")
    t = upload(wl)
    pa.pa_reshape_and_cache_scaled(t["key"], t["value"], t["k_cache"], t["v_cache"], t["slot_mapping"], wl.k_scale,
                                   wl.v_scale)
    big, out = guarded_like(t["q"])
    pa.pa_decode_scaled(out, t["q"], t["k_cache"], t["v_cache"], t["block_tables"], t["seq_lens"], wl.scale,
                        wl.max_seq_len, wl.k_scale, wl.v_scale)
    assert pa.pa_get_device_error() == 0
    assert guards_intact(big)
    k, v = oracle_pools(wl)
    assert_close(as_f64(out), oracle_out(wl, k, v), "fp8", with_rounding=True, out_dtype="bf16")


def test_fused_step_writes_only_its_output_rows():
    import paged_kv_cache_306_gb300 as pa
    wl = W.make_prefix_shared("guardstep", "f16", 3, 4, 8, 2, 128, 16, seed=8, len_range=(8, 600),
                              prefix_range=(10, 300), partition_size=-1)
    t = upload(wl)
    big, out = guarded_like(t["q"])
    pa.pa_decode_step(out, t["q"], t["key"], t["value"], t["k_cache"], t["v_cache"],
                      t["cow"] if len(wl.cow) else None, t["block_tables"], t["seq_lens"], wl.scale, wl.max_seq_len)
    assert pa.pa_get_device_error() == 0
    assert guards_intact(big)
    k, v = oracle_pools(wl)
    assert_close(as_f64(out), oracle_out(wl, k, v), "f16", with_rounding=True)


@pytest.mark.parametrize("dtype,D,bs", [("f16", 128, 16), ("bf16", 64, 32)])
def test_prefill_writes_only_its_output_rows(dtype, D, bs):
    import oracle
    import paged_kv_cache_306_gb300 as pa
    wl = W.make_prefill("guardpf", dtype, [0, 100, 257], [130, 7, 64], 8, 2, D, bs, seed=9)
    dev = "cuda"
    kc, vc = W.to_torch(wl.k_cache, dtype, dev), W.to_torch(wl.v_cache, dtype, dev)
    q = W.to_torch(wl.q, dtype, dev)
    pa.pa_reshape_and_cache(W.to_torch(wl.key, dtype, dev), W.to_torch(wl.value, dtype, dev), kc, vc,
                            torch.from_numpy(wl.slot_mapping).to(dev))
    big, out = guarded_like(q)
    pa.pa_prefill(out, q, kc, vc, torch.from_numpy(wl.block_tables).to(dev), torch.from_numpy(wl.seq_lens).to(dev),
                  torch.from_numpy(wl.query_start_loc).to(dev), wl.scale, wl.max_seq_len)
    assert pa.pa_get_device_error() == 0
    assert guards_intact(big)
    k, v = wl.clone_pools()
    oracle.reshape_and_cache(wl.key, wl.value, k, v, wl.slot_mapping, dtype)
    ref = oracle.prefill(wl.q, k, v, wl.block_tables, wl.seq_lens, wl.query_start_loc, wl.scale, dtype)
    assert_close(as_f64(out), ref, dtype, with_rounding=True)
