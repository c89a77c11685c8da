"""GPU parity of the decode path against the CPU oracle, through the C ABI.

Outputs must match the fp64 oracle within 2e-3 max-abs for fp16/bf16 caches and
1e-5 for fp32 caches.  Small out-of-workload cases (short sequences, outputs of
order one) also allow half an ulp of the output dtype for the final rounding.
"""
import zlib

import numpy as np
import pytest

import oracle
import workloads as W
from helpers import TOL, as_f64, assert_close, gpu_step, oracle_out, oracle_pools, upload

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import paged_kv_cache_306_gb300 as pa
    pa.load()


def edge_lengths(bs, extra):
    return [1, bs - 1, bs, bs + 1, 2 * bs, 3 * bs + 5] + list(extra)


@pytest.mark.parametrize("dtype", ["f32", "f16", "bf16"])
@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("bs", [16, 32])
@pytest.mark.parametrize("G", [1, 4, 7, 20])
@pytest.mark.parametrize("part", [0, "2bs", -1])
def test_decode_matches_oracle_on_ragged_batches(dtype, D, bs, G, part):
    rng = np.random.default_rng(zlib.crc32(repr((dtype, D, bs, G, part)).encode()))
    L = edge_lengths(bs, rng.integers(2, 400, size=3))
    ps = 2 * bs if part == "2bs" else part
    wl = W.make_private("ragged", dtype, L, 2 * G, 2, D, bs, seed=int(rng.integers(1 << 30)), partition_size=ps)
    out, _ = gpu_step(wl)
    k, v = oracle_pools(wl)
    ref = oracle_out(wl, k, v)
    assert_close(as_f64(out), ref, dtype, with_rounding=True, what=f"{dtype} D{D} bs{bs} G{G} P{ps}")


@pytest.mark.parametrize("dtype", ["f32", "f16", "bf16"])
@pytest.mark.parametrize("G", [1, 4])
def test_partition_boundaries(dtype, G):
    """Lengths on both sides of partition edges, several partitions per sequence."""
    bs, P = 16, 64
    L = [P - 1, P, P + 1, 2 * P - 1, 2 * P, 2 * P + 1, 7 * P + 3]
    wl = W.make_private("pb", dtype, L, 2 * G, 2, 128, bs, seed=41, partition_size=P)
    out, _ = gpu_step(wl)
    k, v = oracle_pools(wl)
    assert_close(as_f64(out), oracle_out(wl, k, v), dtype, with_rounding=True)


@pytest.mark.parametrize("dtype", ["f32", "f16", "bf16"])
@pytest.mark.parametrize("G", [1, 8])
def test_seq_len_one_returns_v0_bit_exactly(dtype, G):
    wl = W.make_private("one", dtype, [1, 1, 1], 2 * G, 2, 128, 16, seed=3, partition_size=0)
    out, t = gpu_step(wl)
    # the only token is the one just written: out[s, h] == value[s, h // G]
    v0 = t["value"].repeat_interleave(G, dim=1)
    assert torch.equal(out.view(torch.int16 if dtype != "f32" else torch.int32),
                       v0.view(torch.int16 if dtype != "f32" else torch.int32))


@pytest.mark.parametrize("dtype", ["f32", "f16", "bf16"])
@pytest.mark.parametrize("G", [1, 4])
@pytest.mark.parametrize("ps", [0, 32, -1])
def test_physical_permutation_is_bit_identical(dtype, G, ps):
    wl = W.make_private("perm", dtype, [700, 33, 256, 1], 2 * G, 2, 128, 16, seed=5, partition_size=ps)
    out1, _ = gpu_step(wl)
    rng = np.random.default_rng(9)
    pi = rng.permutation(wl.num_blocks)
    k2 = np.empty_like(wl.k_cache)
    v2 = np.empty_like(wl.v_cache)
    k2[pi] = wl.k_cache
    v2[pi] = wl.v_cache
    bt2 = np.where(wl.block_tables >= 0, pi[np.maximum(wl.block_tables, 0)], -1).astype(np.int32)
    wl2 = W.Workload(**{**wl.__dict__, "k_cache": k2, "v_cache": v2, "block_tables": bt2,
                        "slot_mapping": pi[wl.slot_mapping // 16] * 16 + wl.slot_mapping % 16})
    out2, _ = gpu_step(wl2)
    assert torch.equal(out1, out2)


@pytest.mark.parametrize("dtype", ["f16", "bf16", "f32"])
@pytest.mark.parametrize("G", [1, 4])
def test_one_partition_covering_the_sequence_equals_no_split_bit_exactly(dtype, G):
    wl = W.make_private("cover", dtype, [300, 17, 512], 2 * G, 2, 128, 16, seed=8, partition_size=0)
    out_none, t = gpu_step(wl)
    out_cover, _ = gpu_step(wl, partition_size=512, t=t, write=False)
    assert torch.equal(out_none, out_cover)


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_split_agrees_with_no_split(dtype):
    wl = W.make_private("split", dtype, [5000, 1200, 77], 16, 4, 128, 16, seed=12, partition_size=0)
    out0, t = gpu_step(wl)
    for ps in (16, 64, 256, 1024, -1):
        out1, _ = gpu_step(wl, partition_size=ps, t=t, write=False)
        d = (out0.double() - out1.double()).abs().max().item()
        assert d <= TOL[dtype], (ps, d)


def test_uniform_values_give_exact_mean_and_softmax_weights_sum_to_one():
    """With V == 1 everywhere the output is sum_t w_t = 1 (softmax weights sum to 1)."""
    wl = W.make_private("ones", "f16", [1000, 31, 4096], 16, 2, 128, 16, seed=13, partition_size=-1)
    wl.v_cache[np.isfinite(wl.v_cache)] = 1.0
    wl.value[...] = 1.0
    out, _ = gpu_step(wl)
    assert (out.double() - 1.0).abs().max().item() <= 1e-3


def test_non_default_stream():
    wl = W.make_private("stream", "bf16", [999, 64], 8, 2, 128, 16, seed=14, partition_size=128)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        out, _ = gpu_step(wl)
    s.synchronize()
    k, v = oracle_pools(wl)
    assert_close(as_f64(out), oracle_out(wl, k, v), "bf16")


# --- the write path ------------------------------------------------------------------------------

@pytest.mark.parametrize("dtype", ["f32", "f16", "bf16"])
@pytest.mark.parametrize("bs", [16, 32])
def test_reshape_and_cache_of_many_tokens_is_bit_exact(dtype, bs):
    """A write of many tokens (the tiled kernel: 32 tokens of one kv head per CTA):
    chunks of consecutive slots at every alignment within a block, crossing blocks,
    scattered slots, padding, and a ragged last tile; bit-identical with the oracle."""
    import paged_kv_cache_306_gb300 as pa
    rng = np.random.default_rng(zlib.crc32(repr(("tiled write", dtype, bs)).encode()))
    Hkv, D, NB = 8, 128, 400
    perm = rng.permutation(NB)
    slots, b = [], 0
    for n in (1, 5, 31, 32, 33, 100, 257, 500):  # runs of consecutive positions through private blocks
        start = int(rng.integers(0, bs))
        nblk = -(-(start + n) // bs)
        table = perm[b:b + nblk]
        b += nblk
        pos = start + np.arange(n)
        slots += list(table[pos // bs] * bs + pos % bs)
    free = np.setdiff1d(np.arange(NB * bs), np.array(slots))
    slots += list(rng.choice(free, size=200, replace=False))  # scattered
    slots = np.array(slots, dtype=np.int64)
    slots[rng.choice(len(slots), size=20, replace=False)] = -1  # padding
    T = len(slots)
    assert (T + 31) // 32 * Hkv >= 256 and T % 32 != 0
    wl = W.make_private("w", dtype, [bs] * 2, Hkv, Hkv, D, bs, seed=23, num_blocks=NB, poison=False)
    key = W.randn(rng, (T, Hkv, D), dtype)
    value = W.randn(rng, (T, Hkv, D), dtype)
    t = upload(wl)
    pa.pa_reshape_and_cache(W.to_torch(key, dtype, "cuda"), W.to_torch(value, dtype, "cuda"), t["k_cache"],
                            t["v_cache"], torch.from_numpy(slots).cuda())
    assert pa.pa_get_device_error() == 0
    k, v = wl.clone_pools()
    oracle.reshape_and_cache(key, value, k, v, slots, dtype)
    assert np.array_equal(W.from_torch(t["k_cache"], dtype).view(np.uint8), k.view(np.uint8))
    assert np.array_equal(W.from_torch(t["v_cache"], dtype).view(np.uint8), v.view(np.uint8))


@pytest.mark.parametrize("dtype", ["f32", "f16", "bf16"])
@pytest.mark.parametrize("bs", [16, 32])
def test_reshape_and_cache_is_bit_exact(dtype, bs):
    import paged_kv_cache_306_gb300 as pa
    rng = np.random.default_rng(21)
    NB, Hkv, D, T = 40, 4, 128, 57
    wl = W.make_private("w", dtype, [bs * 3] * 4, Hkv, Hkv, D, bs, seed=22, num_blocks=NB, poison=False)
    key = W.randn(rng, (T, Hkv, D), dtype)
    value = W.randn(rng, (T, Hkv, D), dtype)
    slots = rng.permutation(NB * bs)[:T].astype(np.int64)
    slots[[3, 10]] = -1
    t = upload(wl)
    pa.pa_reshape_and_cache(W.to_torch(key, dtype, "cuda"), W.to_torch(value, dtype, "cuda"), t["k_cache"],
                            t["v_cache"], torch.from_numpy(slots).cuda())
    assert pa.pa_get_device_error() == 0
    k, v = wl.clone_pools()
    oracle.reshape_and_cache(key, value, k, v, slots, dtype)
    assert np.array_equal(W.from_torch(t["k_cache"], dtype).view(np.uint8), k.view(np.uint8))
    assert np.array_equal(W.from_torch(t["v_cache"], dtype).view(np.uint8), v.view(np.uint8))


@pytest.mark.parametrize("dtype", ["f32", "f16", "bf16"])
def test_copy_blocks_is_bit_exact(dtype):
    import paged_kv_cache_306_gb300 as pa
    wl = W.make_private("c", dtype, [64] * 6, 8, 8, 128, 16, seed=23, num_blocks=40, poison=False)
    used = set(wl.block_tables[wl.block_tables >= 0].tolist())
    free = [b for b in range(wl.num_blocks) if b not in used]
    pairs = np.stack([wl.block_tables[:4, 0], np.array(free[:4])], axis=1).astype(np.int64)
    t = upload(wl)
    pa.pa_copy_blocks(t["k_cache"], t["v_cache"], torch.from_numpy(pairs).cuda())
    assert pa.pa_get_device_error() == 0
    k, v = wl.clone_pools()
    oracle.copy_blocks(k, v, pairs, dtype)
    assert np.array_equal(W.from_torch(t["k_cache"], dtype).view(np.uint8), k.view(np.uint8))
    assert np.array_equal(W.from_torch(t["v_cache"], dtype).view(np.uint8), v.view(np.uint8))


# --- device-side checks ------------------------------------------------------------------------

def test_out_of_pool_block_id_is_reported_not_faulted():
    import paged_kv_cache_306_gb300 as pa
    wl = W.make_private("bad", "f16", [100, 40], 8, 2, 128, 16, seed=24, poison=False, partition_size=0)
    wl.block_tables[1, 1] = wl.num_blocks + 5
    t = upload(wl)
    out = torch.empty_like(t["q"])
    pa.pa_decode(out, t["q"], t["k_cache"], t["v_cache"], t["block_tables"], t["seq_lens"], wl.scale,
                 wl.max_seq_len, 0)
    assert pa.pa_get_device_error() == 1
    assert pa.pa_get_device_error() == 0        # read clears it


def test_seq_len_beyond_the_bound_is_reported_and_zeroed():
    import paged_kv_cache_306_gb300 as pa
    wl = W.make_private("badlen", "bf16", [100, 40], 8, 2, 128, 16, seed=25, poison=False, partition_size=0)
    t = upload(wl)
    t["seq_lens"][1] = 0
    out = torch.full_like(t["q"], 7.0)
    pa.pa_decode(out, t["q"], t["k_cache"], t["v_cache"], t["block_tables"], t["seq_lens"], wl.scale,
                 wl.max_seq_len, 0)
    assert pa.pa_get_device_error() == 2
    assert torch.all(out[1] == 0)
    assert torch.all(torch.isfinite(out[0]))


def test_slot_beyond_the_pool_is_reported():
    import paged_kv_cache_306_gb300 as pa
    wl = W.make_private("badslot", "f16", [32], 2, 2, 64, 16, seed=26, poison=False)
    t = upload(wl)
    slots = torch.tensor([wl.num_blocks * 16], dtype=torch.int64, device="cuda")
    k_before = t["k_cache"].clone()
    pa.pa_reshape_and_cache(t["key"], t["value"], t["k_cache"], t["v_cache"], slots)
    assert pa.pa_get_device_error() == 3
    assert torch.equal(k_before, t["k_cache"])


def test_workspace_too_small_is_rejected():
    import paged_kv_cache_306_gb300 as pa
    wl = W.make_private("ws", "f16", [1000], 8, 2, 128, 16, seed=27, poison=False)
    t = upload(wl)
    out = torch.empty_like(t["q"])
    lib = pa.load()
    st = lib.pa_decode(out.data_ptr(), t["q"].data_ptr(), t["k_cache"].data_ptr(), t["v_cache"].data_ptr(),
                       t["block_tables"].data_ptr(), t["block_tables"].shape[1], t["seq_lens"].data_ptr(), 1,
                       1000, 8, 2, 128, 16, wl.num_blocks, 0.1, 64, None, 0, pa.PA_F16, None)
    assert st == 4


def test_workspace_does_not_depend_on_caller_partitions():
    """Caller partitions are merged inside the warps, so they need no extra partial slots."""
    import paged_kv_cache_306_gb300 as pa
    lib = pa.load()
    none = lib.pa_decode_workspace_size(64, 28, 4, 128, 4096, 16, 0, pa.PA_F16)
    auto = lib.pa_decode_workspace_size(64, 28, 4, 128, 4096, 16, -1, pa.PA_F16)
    p256 = lib.pa_decode_workspace_size(64, 28, 4, 128, 4096, 16, 256, pa.PA_F16)
    assert none > 0 and auto == none and p256 == none
    assert lib.pa_decode_plan_partition(64, 28, 4, 128, 4096, 16, pa.PA_F16) == 0


def test_more_sequences_than_one_launch_holds():
    """Batches beyond one launch's sequence tables are cut into several launches."""
    rng = np.random.default_rng(29)
    L = rng.integers(1, 90, size=2100)
    wl = W.make_private("many", "f16", L, 8, 2, 64, 16, seed=30, partition_size=-1)
    out, _ = gpu_step(wl)
    k, v = oracle_pools(wl)
    assert_close(as_f64(out), oracle_out(wl, k, v), "f16", with_rounding=True)


def test_launch_count_counts_kernels():
    import paged_kv_cache_306_gb300 as pa
    wl = W.make_private("cnt", "f16", [2000, 100], 8, 2, 128, 16, seed=28, partition_size=256)
    t = upload(wl)
    n0 = pa.pa_launch_count()
    gpu_step(wl, t=t)
    assert pa.pa_launch_count() - n0 == 3        # write, decode, merge


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("G", [1, 4, 7])
def test_workspace_full_of_nan_bytes_does_not_leak_into_outputs(dtype, G):
    """A small batch leaves warps with no blocks, so some partial slots inside a
    segment's range are never written; whatever they hold must weigh nothing."""
    import paged_kv_cache_306_gb300 as pa
    wl = W.make_private("nanws", dtype, [1, 15, 17, 53, 200, 333, 90], 2 * G, 2, 128, 16, seed=61,
                        partition_size=32)
    t = upload(wl)
    code = pa.PA_F16 if dtype == "f16" else pa.PA_BF16
    need = pa.pa_decode_workspace_size(wl.num_seqs, wl.num_heads, wl.num_kv_heads, wl.head_size, wl.max_seq_len,
                                       wl.block_size, 32, code)
    ws = torch.full((max(need, 16),), 0xFF, dtype=torch.uint8, device="cuda")   # NaN floats, tags -1
    pa.pa_reshape_and_cache(t["key"], t["value"], t["k_cache"], t["v_cache"], t["slot_mapping"])
    out = torch.empty_like(t["q"])
    pa.pa_decode(out, t["q"], t["k_cache"], t["v_cache"], t["block_tables"], t["seq_lens"], wl.scale,
                 wl.max_seq_len, 32, ws)
    assert pa.pa_get_device_error() == 0
    k, v = oracle_pools(wl)
    assert_close(as_f64(out), oracle_out(wl, k, v), dtype, with_rounding=True)


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_repeated_calls_on_one_workspace_agree_bit_exactly(dtype):
    """The per-segment counters and slot tags of one call must never be taken for
    the next call's: the same workspace, reused, gives the same bits every time,
    also when it starts out full of random bytes."""
    import paged_kv_cache_306_gb300 as pa
    rng = np.random.default_rng(62)
    L = rng.integers(1, 6000, size=40)
    wl = W.make_private("reuse", dtype, L, 28, 4, 128, 16, seed=63, partition_size=-1)
    t = upload(wl)
    code = pa.PA_F16 if dtype == "f16" else pa.PA_BF16
    need = pa.pa_decode_workspace_size(wl.num_seqs, wl.num_heads, wl.num_kv_heads, wl.head_size, wl.max_seq_len,
                                       wl.block_size, 0, code)
    ws = torch.randint(0, 256, (max(need, 16),), dtype=torch.uint8, device="cuda")
    pa.pa_reshape_and_cache(t["key"], t["value"], t["k_cache"], t["v_cache"], t["slot_mapping"])
    outs = []
    for _ in range(3):
        out = torch.empty_like(t["q"])
        pa.pa_decode(out, t["q"], t["k_cache"], t["v_cache"], t["block_tables"], t["seq_lens"], wl.scale,
                     wl.max_seq_len, 0, ws)
        outs.append(out)
    assert pa.pa_get_device_error() == 0
    assert torch.equal(outs[0], outs[1]) and torch.equal(outs[1], outs[2])
    k, v = oracle_pools(wl)
    assert_close(as_f64(outs[0]), oracle_out(wl, k, v), dtype, with_rounding=True)
