"""The fused generation step (pa_decode_step) on the GPU, through the C ABI.

The decode kernel writes every sequence's new token as part of decode (after
the copy-on-write copies, when there are any).  It must leave the pools byte-identical to, and give outputs
bit-identical with, the three separate calls (pa_copy_blocks,
pa_reshape_and_cache, pa_decode) on the same inputs -- and so match the oracle
within the decode tolerance, which is checked as well.
"""
import zlib

import numpy as np
import pytest

import oracle
import workloads as W
from helpers import as_f64, assert_close, fused_step, gpu_step, oracle_out, oracle_pools, same_bytes, upload

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import paged_kv_cache_306_gb300 as pa
    pa.load()


def check_against_separate_calls(wl, partition_size=None):
    out_f, tf = fused_step(wl, partition_size)
    out_s, ts = gpu_step(wl, partition_size)
    assert same_bytes(tf["k_cache"], ts["k_cache"]), "K pool differs from the separate calls"
    assert same_bytes(tf["v_cache"], ts["v_cache"]), "V pool differs from the separate calls"
    assert same_bytes(out_f, out_s), "output differs from the separate calls"
    return out_f, tf


def small_prefix_shared(dtype, bs, G, seed, num_groups=3, group_size=4, partition_size=-1):
    return W.make_prefix_shared("cow", dtype, num_groups, group_size, 2 * G, 2, 128, bs, seed=seed,
                                len_range=(8, 700), prefix_range=(10, 300), partition_size=partition_size)


@pytest.mark.parametrize("dtype", ["f32", "f16", "bf16"])
@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("bs", [16, 32])
@pytest.mark.parametrize("G", [1, 4, 7, 20])
@pytest.mark.parametrize("part", [0, -1])
def test_fused_step_matches_separate_calls_and_oracle_on_ragged_batches(dtype, D, bs, G, part):
    rng = np.random.default_rng(zlib.crc32(repr(("step", dtype, D, bs, G, part)).encode()))
    L = [1, bs - 1, bs, bs + 1, 2 * bs, 3 * bs + 5] + list(rng.integers(2, 400, size=3))
    wl = W.make_private("ragged", dtype, L, 2 * G, 2, D, bs, seed=int(rng.integers(1 << 30)), partition_size=part)
    out, t = check_against_separate_calls(wl)
    k, v = oracle_pools(wl)
    assert np.array_equal(W.from_torch(t["k_cache"], dtype).view(np.uint8), k.view(np.uint8))
    assert np.array_equal(W.from_torch(t["v_cache"], dtype).view(np.uint8), v.view(np.uint8))
    assert_close(as_f64(out), oracle_out(wl, k, v), dtype, with_rounding=True, what=f"{dtype} D{D} bs{bs} G{G}")


@pytest.mark.parametrize("dtype", ["f32", "f16", "bf16"])
@pytest.mark.parametrize("bs", [16, 32])
@pytest.mark.parametrize("G", [1, 4, 8])
def test_fused_step_with_copy_on_write(dtype, bs, G):
    """Shared partial blocks copied before the new tokens land."""
    wl = small_prefix_shared(dtype, bs, G, seed=zlib.crc32(repr(("cow", dtype, bs, G)).encode()))
    assert len(wl.cow) > 0
    out, t = check_against_separate_calls(wl)
    k, v = oracle_pools(wl)
    assert np.array_equal(W.from_torch(t["k_cache"], dtype).view(np.uint8), k.view(np.uint8))
    assert np.array_equal(W.from_torch(t["v_cache"], dtype).view(np.uint8), v.view(np.uint8))
    assert_close(as_f64(out), oracle_out(wl, k, v), dtype, with_rounding=True)


@pytest.mark.parametrize("i,bs", [(1, None), (2, None), (3, None), (4, None), (5, 16), (5, 32)])
def test_full_size_workloads_match_separate_calls(i, bs):
    """The benchmark's workloads at full size, in the launch configuration the
    benchmark times: bit-identical to the three calls; a sample of sequences
    against the oracle."""
    wl = W.config(i, block_size=bs)
    out, t = check_against_separate_calls(wl)
    seqs = [0, wl.num_seqs - 1] if i == 4 else list(np.random.default_rng(i).choice(wl.num_seqs, 3, replace=False))
    k, v = oracle_pools(wl)
    ref = oracle_out(wl, k, v, seqs)
    assert_close(as_f64(out)[seqs], ref, wl.dtype, with_rounding=True, what=wl.name)


def test_more_sequences_than_one_launch_with_copies():
    """Three decode launches; the copies (made before the first) include blocks of
    sequences that the later launches write into and read."""
    wl = W.make_prefix_shared("many", "f16", 300, 7, 8, 2, 64, 16, seed=91, len_range=(4, 300),
                              prefix_range=(5, 150), partition_size=-1)
    assert wl.num_seqs > 2048 and len(wl.cow) > 0
    late = set(np.nonzero(np.arange(wl.num_seqs) >= 1024)[0].tolist())
    dst_owner = {int(b): s for s in range(wl.num_seqs) for b in wl.block_tables[s] if b >= 0}
    assert any(dst_owner.get(int(d)) in late for d in wl.cow[:, 1])
    out, t = check_against_separate_calls(wl)
    k, v = oracle_pools(wl)
    assert np.array_equal(W.from_torch(t["k_cache"], "f16").view(np.uint8), k.view(np.uint8))
    assert_close(as_f64(out), oracle_out(wl, k, v), "f16", with_rounding=True)


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_repeated_fused_steps_on_one_workspace(dtype):
    """A workspace full of random bytes, reused three times, gives the same bits
    each time."""
    import paged_kv_cache_306_gb300 as pa
    wl = small_prefix_shared(dtype, 16, 4, seed=93, num_groups=6, group_size=6)
    t = upload(wl)
    code = pa.PA_F16 if dtype == "f16" else pa.PA_BF16
    need = pa.pa_decode_workspace_size(wl.num_seqs, wl.num_heads, wl.num_kv_heads, wl.head_size, wl.max_seq_len,
                                       wl.block_size, wl.partition_size, code)
    ws = torch.randint(0, 256, (max(need, 16),), dtype=torch.uint8, device="cuda")
    outs = [fused_step(wl, t=t, workspace=ws)[0] for _ in range(3)]
    assert same_bytes(outs[0], outs[1]) and same_bytes(outs[1], outs[2])
    k, v = oracle_pools(wl)
    assert np.array_equal(W.from_torch(t["k_cache"], dtype).view(np.uint8), k.view(np.uint8))
    assert_close(as_f64(outs[0]), oracle_out(wl, k, v), dtype, with_rounding=True)


def test_launch_count_is_decode_and_merge_plus_copies():
    import paged_kv_cache_306_gb300 as pa
    for wl, n in ((W.make_private("cnt", "f16", [2000, 100], 8, 2, 128, 16, seed=28, partition_size=256), 2),
                  (small_prefix_shared("f16", 16, 4, seed=94), 3)):
        t = upload(wl)
        n0 = pa.pa_launch_count()
        fused_step(wl, t=t)
        assert pa.pa_launch_count() - n0 == n


def test_sequence_outside_the_bound_is_reported_and_writes_nothing():
    import paged_kv_cache_306_gb300 as pa
    wl = W.make_private("bad", "f16", [40, 70, 33, 90], 8, 2, 128, 16, seed=95, partition_size=0)
    t = upload(wl)
    t["seq_lens"][2] = wl.max_seq_len + 7
    out, _ = fused_step(wl, t=t, check_error=False)
    assert pa.pa_get_device_error() == 2
    keep = [0, 1, 3]
    k, v = wl.clone_pools()
    oracle.reshape_and_cache(wl.key[keep], wl.value[keep], k, v, wl.slot_mapping[keep], "f16")
    assert np.array_equal(W.from_torch(t["k_cache"], "f16").view(np.uint8), k.view(np.uint8))
    assert np.array_equal(W.from_torch(t["v_cache"], "f16").view(np.uint8), v.view(np.uint8))
    assert_close(as_f64(out)[keep], oracle_out(wl, k, v, keep), "f16", with_rounding=True)
    assert np.all(as_f64(out)[2] == 0)


def test_copy_id_outside_the_pool_is_reported_and_skipped():
    import paged_kv_cache_306_gb300 as pa
    wl = small_prefix_shared("f16", 16, 4, seed=96)
    t = upload(wl)
    bad = torch.tensor([[wl.num_blocks + 3, 0]], dtype=torch.int64, device="cuda")
    t["cow"] = torch.cat([bad, t["cow"]])
    wl.cow = np.concatenate([np.array([[wl.num_blocks + 3, 0]], np.int64), wl.cow])
    out, _ = fused_step(wl, t=t, check_error=False)
    assert pa.pa_get_device_error() == 5
    wl.cow = wl.cow[1:]
    k, v = oracle_pools(wl)
    assert np.array_equal(W.from_torch(t["k_cache"], "f16").view(np.uint8), k.view(np.uint8))
    assert_close(as_f64(out), oracle_out(wl, k, v), "f16", with_rounding=True)


def test_copies_alone_when_there_is_nothing_to_decode():
    import paged_kv_cache_306_gb300 as pa
    wl = small_prefix_shared("bf16", 16, 1, seed=97)
    t = upload(wl)
    empty_q = t["q"][:0]
    pa.pa_decode_step(empty_q.clone(), empty_q, t["key"][:0], t["value"][:0], t["k_cache"], t["v_cache"], t["cow"],
                      t["block_tables"][:0], t["seq_lens"][:0], wl.scale, 1, 0)
    assert pa.pa_get_device_error() == 0
    k, v = wl.clone_pools()
    oracle.copy_blocks(k, v, wl.cow, "bf16")
    assert np.array_equal(W.from_torch(t["k_cache"], "bf16").view(np.uint8), k.view(np.uint8))
    assert np.array_equal(W.from_torch(t["v_cache"], "bf16").view(np.uint8), v.view(np.uint8))


@pytest.mark.parametrize("dtype,bs", [("f16", 16), ("bf16", 32)])
def test_serving_loop_on_the_fused_step(dtype, bs):
    """The block manager's slots and copy pairs drive the fused step, step after step."""
    import paged_kv_cache_306_gb300 as pa
    rng = np.random.default_rng(98)
    H, Hkv, D, NB = 8, 2, 128, 400
    x = W.pack_x(dtype)
    bm = pa.BlockManager(NB, bs)
    k_host = np.zeros((NB, Hkv, D // x, bs, x), W.NP_STORAGE[dtype])
    v_host = np.zeros((NB, Hkv, D, bs), W.NP_STORAGE[dtype])
    k_dev, v_dev = W.to_torch(k_host, dtype, "cuda"), W.to_torch(v_host, dtype, "cuda")
    ids = []
    for sid, n in enumerate(rng.integers(1, 300, size=6)):
        slots = bm.add_sequence(sid, int(n))
        key, value = W.randn(rng, (int(n), Hkv, D), dtype), W.randn(rng, (int(n), Hkv, D), dtype)
        pa.pa_reshape_and_cache(W.to_torch(key, dtype, "cuda"), W.to_torch(value, dtype, "cuda"), k_dev, v_dev,
                                torch.from_numpy(slots).cuda())
        oracle.reshape_and_cache(key, value, k_host, v_host, slots, dtype)
        ids.append(sid)
    for child, parent in [(10, 0), (11, 0), (12, 3), (13, 12)]:
        bm.fork(parent, child)
        ids.append(child)
    copies_seen = 0
    for step in range(5):
        batch = [int(s) for s in rng.permutation(ids)]
        slots, copies = bm.append_tokens(batch)
        copies_seen += len(copies)
        S = len(batch)
        key, value = W.randn(rng, (S, Hkv, D), dtype), W.randn(rng, (S, Hkv, D), dtype)
        max_len = max(bm.seq_len(s) for s in batch)
        bt, sl = bm.block_tables(batch, -(-max_len // bs))
        q = W.randn(rng, (S, H, D), dtype)
        qd = W.to_torch(q, dtype, "cuda")
        out = torch.empty_like(qd)
        pa.pa_decode_step(out, qd, W.to_torch(key, dtype, "cuda"), W.to_torch(value, dtype, "cuda"), k_dev, v_dev,
                          torch.from_numpy(copies).cuda() if len(copies) else None, torch.from_numpy(bt).cuda(),
                          torch.from_numpy(sl).cuda(), 1 / np.sqrt(D), max_len, pa.PARTITION_AUTO)
        assert pa.pa_get_device_error() == 0
        oracle.copy_blocks(k_host, v_host, copies, dtype)
        oracle.reshape_and_cache(key, value, k_host, v_host, slots, dtype)
        assert np.array_equal(W.from_torch(k_dev, dtype).view(np.uint8), k_host.view(np.uint8)), step
        assert np.array_equal(W.from_torch(v_dev, dtype).view(np.uint8), v_host.view(np.uint8)), step
        ref = oracle.decode(q, k_host, v_host, bt, sl, 1 / np.sqrt(D), dtype)
        assert_close(as_f64(out), ref, dtype, with_rounding=True, what=f"step {step}")
    assert copies_seen > 0
    bm.close()


@pytest.mark.parametrize("q_dtype", ["f16", "bf16"])
@pytest.mark.parametrize("D,bs,G", [(128, 16, 7), (128, 32, 1), (64, 16, 4), (128, 16, 16)])
def test_fused_step_on_an_fp8_pool(q_dtype, D, bs, G):
    """The new token quantised where it is written and where it enters the stage, with
    the write path's conversion: bit-identical with the three separate calls."""
    rng = np.random.default_rng(zlib.crc32(repr(("fp8step", q_dtype, D, bs, G)).encode()))
    L = [1, bs - 1, bs, bs + 1, 3 * bs + 5] + list(rng.integers(2, 500, size=3))
    wl = W.make_private("fp8step", "fp8", L, 2 * G, 2, D, bs, seed=int(rng.integers(1 << 30)), partition_size=-1,
                        q_dtype=q_dtype)
    out, t = check_against_separate_calls(wl)
    k, v = oracle_pools(wl)
    assert np.array_equal(W.from_torch(t["k_cache"], "fp8").view(np.uint8), k.view(np.uint8))
    assert np.array_equal(W.from_torch(t["v_cache"], "fp8").view(np.uint8), v.view(np.uint8))
    assert_close(as_f64(out), oracle_out(wl, k, v), "fp8", with_rounding=True, out_dtype=q_dtype)


def test_fused_step_on_an_fp8_pool_with_copy_on_write():
    wl = W.make_prefix_shared("fp8cow", "fp8", 3, 4, 8, 2, 128, 16, seed=99, len_range=(8, 700),
                              prefix_range=(10, 300), partition_size=-1, q_dtype="f16")
    assert len(wl.cow) > 0
    out, t = check_against_separate_calls(wl)
    k, v = oracle_pools(wl)
    assert np.array_equal(W.from_torch(t["k_cache"], "fp8").view(np.uint8), k.view(np.uint8))
    assert_close(as_f64(out), oracle_out(wl, k, v), "fp8", with_rounding=True, out_dtype="f16")


@pytest.mark.parametrize("cfg", [2, 5])
def test_full_size_fp8_workloads_match_separate_calls(cfg):
    wl = W.config(cfg, kv_dtype="fp8")
    out, t = check_against_separate_calls(wl)
    seqs = list(np.random.default_rng(cfg).choice(wl.num_seqs, 3, replace=False))
    k, v = oracle_pools(wl)
    assert_close(as_f64(out)[seqs], oracle_out(wl, k, v, seqs), "fp8", with_rounding=True, out_dtype=wl.q_dtype)


def test_fp8_fused_step_over_more_sequences_than_one_launch_holds():
    """Later launches start at their sequences' rows of the 16-bit key/value input."""
    rng = np.random.default_rng(101)
    wl = W.make_private("manyfp8", "fp8", rng.integers(1, 60, size=1100), 8, 2, 64, 16, seed=102,
                        partition_size=-1, q_dtype="bf16")
    out, t = check_against_separate_calls(wl)
    k, v = oracle_pools(wl)
    assert np.array_equal(W.from_torch(t["k_cache"], "fp8").view(np.uint8), k.view(np.uint8))
    assert_close(as_f64(out), oracle_out(wl, k, v), "fp8", with_rounding=True, out_dtype="bf16")
