"""Decode steps driven by the library's block manager, on the GPU, against the oracle.

Prompts are written through the slots the manager hands out, some sequences are
forked (sharing their parent's blocks, the partly filled last one included),
and then every step appends one token per sequence: the manager's copy pairs go
to pa_copy_blocks, its slots to pa_reshape_and_cache and its block tables to
pa_decode.  The oracle runs the same three steps on host copies of the pools.
Pools must agree bytewise after every step, outputs within the parity tolerance.
"""
import numpy as np
import pytest

import oracle
import workloads as W
from helpers import as_f64, assert_close

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import paged_kv_cache_306_gb300 as pa
    pa.load()


@pytest.mark.parametrize("dtype,bs", [("f16", 16), ("bf16", 32)])
def test_serving_loop_with_forks_and_copy_on_write(dtype, bs):
    import paged_kv_cache_306_gb300 as pa
    rng = np.random.default_rng(71)
    H, Hkv, D, NB = 8, 2, 128, 400
    x = W.pack_x(dtype)
    bm = pa.BlockManager(NB, bs)
    k_host = np.zeros((NB, Hkv, D // x, bs, x), W.NP_STORAGE[dtype])
    v_host = np.zeros((NB, Hkv, D, bs), W.NP_STORAGE[dtype])
    k_dev, v_dev = W.to_torch(k_host, dtype, "cuda"), W.to_torch(v_host, dtype, "cuda")

    def write(slots, key, value):
        pa.pa_reshape_and_cache(W.to_torch(key, dtype, "cuda"), W.to_torch(value, dtype, "cuda"), k_dev, v_dev,
                                torch.from_numpy(slots).cuda())
        oracle.reshape_and_cache(key, value, k_host, v_host, slots, dtype)

    # prompts
    ids = []
    for sid, n in enumerate(rng.integers(1, 300, size=6)):
        slots = bm.add_sequence(sid, int(n))
        write(slots, W.randn(rng, (int(n), Hkv, D), dtype), W.randn(rng, (int(n), Hkv, D), dtype))
        ids.append(sid)
    # forks share their parent's history (block boundaries and partial blocks alike)
    for child, parent in [(10, 0), (11, 0), (12, 3), (13, 12)]:
        bm.fork(parent, child)
        ids.append(child)

    for step in range(4):
        batch = [int(s) for s in rng.permutation(ids)]
        slots, copies = bm.append_tokens(batch)
        if len(copies):
            pa.pa_copy_blocks(k_dev, v_dev, torch.from_numpy(copies).cuda())
            oracle.copy_blocks(k_host, v_host, copies, dtype)
        S = len(batch)
        write(slots, W.randn(rng, (S, Hkv, D), dtype), W.randn(rng, (S, Hkv, D), dtype))
        max_len = max(bm.seq_len(s) for s in batch)
        bt, sl = bm.block_tables(batch, -(-max_len // bs))
        q = W.randn(rng, (S, H, D), dtype)
        qd = W.to_torch(q, dtype, "cuda")
        out = torch.empty_like(qd)
        pa.pa_decode(out, qd, k_dev, v_dev, torch.from_numpy(bt).cuda(), torch.from_numpy(sl).cuda(),
                     1 / np.sqrt(D), max_len, pa.PARTITION_AUTO)
        assert pa.pa_get_device_error() == 0
        assert np.array_equal(W.from_torch(k_dev, dtype).view(np.uint8), k_host.view(np.uint8)), step
        assert np.array_equal(W.from_torch(v_dev, dtype).view(np.uint8), v_host.view(np.uint8)), step
        ref = oracle.decode(q, k_host, v_host, bt, sl, 1 / np.sqrt(D), dtype)
        assert_close(as_f64(out), ref, dtype, with_rounding=True, what=f"step {step}")
    # every block a sequence references is accounted for
    held = set()
    for s in ids:
        bt, _ = bm.block_tables([s], 64)
        held |= set(int(b) for b in bt[0] if b >= 0)
    assert bm.num_free_blocks == NB - len(held)
    bm.close()
