"""GPU parity of chunked prefill against the CPU oracle, through the C ABI.

A step writes the chunk's K/V rows through reshape_and_cache, then runs the
prefill: query token i of a chunk of n tokens of a sequence of L cached tokens
(position L - n + i) attends to positions 0..itself.  Outputs must match the
fp64 oracle within 2e-3 max-abs plus half an ulp of the output dtype.
"""
import zlib

import numpy as np
import pytest

import oracle
import workloads as W
from helpers import TOL, as_f64, assert_close

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import paged_kv_cache_306_gb300 as pa
    pa.load()


def run_prefill(wl, t=None):
    import paged_kv_cache_306_gb300 as pa
    if t is None:
        t = {n: W.to_torch(getattr(wl, a), wl.dtype, "cuda") for n, a in
             (("q", "q"), ("key", "key"), ("value", "value"), ("k", "k_cache"), ("v", "v_cache"))}
        t["bt"] = torch.from_numpy(wl.block_tables).cuda()
        t["sl"] = torch.from_numpy(wl.seq_lens).cuda()
        t["qsl"] = torch.from_numpy(wl.query_start_loc).cuda()
        t["slots"] = torch.from_numpy(wl.slot_mapping).cuda()
        pa.pa_reshape_and_cache(t["key"], t["value"], t["k"], t["v"], t["slots"])
    out = torch.empty_like(t["q"])
    pa.pa_prefill(out, t["q"], t["k"], t["v"], t["bt"], t["sl"], t["qsl"], wl.scale, wl.max_seq_len)
    code = pa.pa_get_device_error()
    assert code == 0, f"device error {code}"
    return out, t


def oracle_prefill(wl, seqs=None):
    k, v = wl.clone_pools()
    oracle.reshape_and_cache(wl.key, wl.value, k, v, wl.slot_mapping, wl.dtype)
    return oracle.prefill(wl.q, k, v, wl.block_tables, wl.seq_lens, wl.query_start_loc, wl.scale, wl.dtype)


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("bs", [16, 32])
@pytest.mark.parametrize("G", [1, 4, 7, 20])
def test_prefill_matches_oracle_on_ragged_chunks(dtype, D, bs, G):
    rng = np.random.default_rng(zlib.crc32(repr(("prefill", dtype, D, bs, G)).encode()))
    ctx = [0, 0, 1, bs - 1, bs, bs + 1, 3 * bs + 5] + rng.integers(0, 300, size=2).tolist()
    qn = [1, 37, bs, 1, bs + 1, 2 * bs - 1, 5] + rng.integers(1, 120, size=2).tolist()
    wl = W.make_prefill("ragged", dtype, ctx, qn, 2 * G, 2, D, bs, seed=int(rng.integers(1 << 30)))
    out, _ = run_prefill(wl)
    assert_close(as_f64(out), oracle_prefill(wl), dtype, with_rounding=True,
                 what=f"prefill {dtype} D{D} bs{bs} G{G}")


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_one_token_chunks_agree_with_decode(dtype):
    import paged_kv_cache_306_gb300 as pa
    wl = W.make_prefill("one", dtype, [0, 30, 100, 511], [1, 1, 1, 1], 16, 4, 128, 16, seed=81)
    out, t = run_prefill(wl)
    dec = torch.empty_like(t["q"])
    pa.pa_decode(dec, t["q"], t["k"], t["v"], t["bt"], t["sl"], wl.scale, wl.max_seq_len, 0)
    assert pa.pa_get_device_error() == 0
    assert (out.double() - dec.double()).abs().max().item() <= TOL[dtype]


def test_physical_permutation_is_bit_identical():
    wl = W.make_prefill("perm", "f16", [0, 77, 300], [64, 10, 33], 8, 2, 128, 16, seed=82, poison=False)
    out1, _ = run_prefill(wl)
    pi = np.random.default_rng(83).permutation(wl.num_blocks)
    k2, v2 = np.empty_like(wl.k_cache), np.empty_like(wl.v_cache)
    k2[pi] = wl.k_cache
    v2[pi] = wl.v_cache
    bt2 = np.where(wl.block_tables >= 0, pi[np.maximum(wl.block_tables, 0)], -1).astype(np.int32)
    wl2 = W.Workload(**{**wl.__dict__, "k_cache": k2, "v_cache": v2, "block_tables": bt2,
                        "slot_mapping": pi[wl.slot_mapping // 16] * 16 + wl.slot_mapping % 16})
    out2, _ = run_prefill(wl2)
    assert torch.equal(out1, out2)


def test_a_chunk_longer_than_its_sequence_is_reported():
    import paged_kv_cache_306_gb300 as pa
    wl = W.make_prefill("bad", "f16", [10, 20], [5, 6], 8, 2, 128, 16, seed=84, poison=False)
    _, t = run_prefill(wl)
    t["sl"][0] = 3                                   # 5 queries in a sequence of 3 tokens
    out = torch.zeros_like(t["q"])
    pa.pa_prefill(out, t["q"], t["k"], t["v"], t["bt"], t["sl"], t["qsl"], wl.scale, wl.max_seq_len)
    assert pa.pa_get_device_error() == 2
    assert torch.isfinite(out[5:].float()).all()     # the other sequence is computed


def test_full_size_chunked_prefill_sampled():
    wl = W.prefill_config()
    out, _ = run_prefill(wl)
    # the oracle on four of the sixteen sequences (all their rows)
    keep = [0, 5, 10, 15]
    rows = np.concatenate([np.arange(wl.query_start_loc[s], wl.query_start_loc[s + 1]) for s in keep])
    sub_qsl = np.concatenate([[0], np.cumsum([wl.query_start_loc[s + 1] - wl.query_start_loc[s] for s in keep])])
    k, v = wl.clone_pools()
    oracle.reshape_and_cache(wl.key, wl.value, k, v, wl.slot_mapping, wl.dtype)
    ref = oracle.prefill(np.ascontiguousarray(wl.q[rows]), k, v, wl.block_tables[keep], wl.seq_lens[keep],
                         sub_qsl.astype(np.int32), wl.scale, wl.dtype)
    assert_close(as_f64(out)[rows], ref, "f16", with_rounding=False, what="full-size prefill")


def ramp_scores(wl):
    """Keys t/8 and queries 8 along dim 0 (all else 0), so the score of key t is t:
    every 64-key chunk raises the row maximum by more than 2^8 after scaling, and
    the running maximum moves (O is rescaled in tensor memory) at every chunk."""
    bs, D = wl.block_size, wl.head_size
    k32 = np.zeros(wl.k_cache.shape, np.float32)
    ctx = wl.meta["context_lens"]
    for s, c in enumerate(ctx):
        for t in range(c):
            k32[int(wl.block_tables[s][t // bs]), :, 0, t % bs, 0] = t / 8.0
    keep = wl.k_cache.copy()  # poisoned slots stay poisoned
    kc = W.cast(k32, wl.dtype)
    for s, c in enumerate(ctx):  # only the context slots take the ramp
        for t in range(c):
            blk, off = int(wl.block_tables[s][t // bs]), t % bs
            keep[blk, :, :, off, :] = kc[blk, :, :, off, :]
    wl.k_cache = keep
    q = np.zeros((wl.q.shape[0], wl.num_heads, D), np.float32)
    q[:, :, 0] = 8.0
    wl.q = W.cast(q, wl.dtype)
    key = np.zeros((wl.key.shape[0], wl.num_kv_heads, D), np.float32)
    for s, c in enumerate(ctx):
        for i in range(int(wl.query_start_loc[s + 1] - wl.query_start_loc[s])):
            key[int(wl.query_start_loc[s]) + i, :, 0] = (c + i) / 8.0
    wl.key = W.cast(key, wl.dtype)
    return wl


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("D,G", [(128, 7), (64, 4)])
def test_running_maximum_moving_every_chunk(dtype, D, G):
    wl = W.make_prefill("ramp", dtype, [0, 300, 1000], [200, 70, 129], 2 * G, 2, D, 16, seed=41)
    ramp_scores(wl)
    out, _ = run_prefill(wl)
    assert_close(as_f64(out), oracle_prefill(wl), dtype, with_rounding=True, what=f"{dtype} D{D} G{G}")


def test_more_sequences_than_one_launch_holds():
    rng = np.random.default_rng(43)
    ctx, qn = rng.integers(0, 40, size=1100), rng.integers(1, 6, size=1100)
    wl = W.make_prefill("many", "f16", ctx, qn, 8, 2, 64, 16, seed=44)
    out, _ = run_prefill(wl)
    assert_close(as_f64(out), oracle_prefill(wl), "f16", with_rounding=True)


def test_sequences_with_no_new_tokens_are_skipped():
    """A sequence whose chunk is empty has no query rows and no tiles; the others are
    unaffected (the tile order is computed over all sequences)."""
    wl = W.make_prefill("empty", "bf16", [50, 0, 700, 33, 10], [0, 90, 0, 17, 1], 8, 2, 128, 32, seed=45)
    assert wl.q.shape[0] == 108
    out, _ = run_prefill(wl)
    assert_close(as_f64(out), oracle_prefill(wl), "bf16", with_rounding=True)
