"""The five decode-layer workloads at full size: one step (copy-on-write block
copies, reshape_and_cache of the new tokens, decode) through the C ABI, checked
against the CPU oracle.

Cache writes must be bit-exact; attention outputs within 2e-3 max-abs (fp16,
bf16) or 1e-5 (fp32).  The oracle checks every sequence where that finishes in
seconds and a spread of sequences otherwise.
"""
import numpy as np
import pytest

import workloads as W
from helpers import TOL, as_f64, gpu_step, max_violation, oracle_out, oracle_pools

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

# (config, block_size, sequences the oracle checks: None = all)
CASES = [(1, None, None), (2, None, None), (3, None, None), (4, None, [0, 3]), (5, 16, None), (5, 32, None)]


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import paged_kv_cache_306_gb300 as pa
    pa.load()


@pytest.mark.parametrize("cfg,bs,seqs", CASES, ids=lambda v: str(v))
def test_layer_workload_step(cfg, bs, seqs):
    wl = W.config(cfg, block_size=bs)
    out, t = gpu_step(wl)
    k, v = oracle_pools(wl)
    # write path: the whole pool, bytewise
    assert np.array_equal(W.from_torch(t["k_cache"], wl.dtype).view(np.uint8), k.view(np.uint8))
    assert np.array_equal(W.from_torch(t["v_cache"], wl.dtype).view(np.uint8), v.view(np.uint8))
    # attention
    idx = np.arange(wl.num_seqs) if seqs is None else np.asarray(seqs)
    ref = oracle_out(wl, k, v, idx)
    got = as_f64(out)[idx]
    err, excess = max_violation(got, ref, wl.dtype, with_rounding=False)
    assert excess <= 0.0, f"config {cfg}: max abs err {err:.3e} > {TOL[wl.dtype]}"


def test_long_context_with_planner_partitioning():
    wl = W.config(4)
    out_auto, t = gpu_step(wl, partition_size=-1)
    out_512, _ = gpu_step(wl, partition_size=512, t=t, write=False)
    k, v = oracle_pools(wl)
    ref = oracle_out(wl, k, v, [0])
    for out in (out_auto, out_512):
        err, excess = max_violation(as_f64(out)[[0]], ref, "bf16", with_rounding=False)
        assert excess <= 0.0, err
