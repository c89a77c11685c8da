"""The timeout path of the kernels' bounded waits, made to run for real.

Every pipeline wait in the decode and prefill kernels gives up after a limit,
records PA_DEVERR_TIMEOUT, waits (bounded, at the normal limit) for the copies it
still has in flight and ends the kernel early, so the context stays usable.
pa_set_test_wait_limit makes the first pipeline wait of each decode warp (each
prefill CTA) wait on an mbarrier that nothing completes, for a short limit: the
wait runs out.  The tests check that the call returns, that the error word holds
PA_DEVERR_TIMEOUT, and that the next call with normal waits is correct again.
No fault, trap or hang is involved: every wait here ends by its own limit.
"""
import numpy as np
import pytest

import workloads as W
from helpers import as_f64, assert_close, fused_step, oracle_out, oracle_pools, upload

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

TIMEOUT = 4          # PA_DEVERR_TIMEOUT
LIMIT_NS = 2_000_000  # 2 ms: short, and long enough that the copies issued have landed


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import paged_kv_cache_306_gb300 as pa
    pa.load()
    yield
    pa.pa_set_test_wait_limit(0)


def _decode(pa, wl, t, part):
    out = torch.empty_like(t["q"])
    pa.pa_decode(out, t["q"], t["k_cache"], t["v_cache"], t["block_tables"], t["seq_lens"], wl.scale, wl.max_seq_len,
                 part)
    return out


@pytest.mark.parametrize("dtype,part", [("f16", -1), ("bf16", 64)])
def test_decode_wait_that_runs_out_reports_a_timeout_and_the_next_call_is_correct(dtype, part):
    import paged_kv_cache_306_gb300 as pa
    wl = W.make_private("timeout-decode", dtype, [1, 17, 300, 2500, 40, 900], 28, 4, 128, 16, seed=91,
                        partition_size=part)
    t = upload(wl)
    pa.pa_reshape_and_cache(t["key"], t["value"], t["k_cache"], t["v_cache"], t["slot_mapping"])
    assert pa.pa_get_device_error() == 0
    try:
        pa.pa_set_test_wait_limit(LIMIT_NS)
        _decode(pa, wl, t, part)
    finally:
        pa.pa_set_test_wait_limit(0)
    assert pa.pa_get_device_error() == TIMEOUT   # the call returned; the wait ran out and said so
    assert pa.pa_get_device_error() == 0         # reading clears the word
    out = _decode(pa, wl, t, part)               # normal waits again: the context is usable
    assert pa.pa_get_device_error() == 0
    k, v = oracle_pools(wl)
    assert_close(as_f64(out), oracle_out(wl, k, v), dtype, what="decode after a timed-out call")


def test_fused_step_wait_that_runs_out_reports_a_timeout():
    import paged_kv_cache_306_gb300 as pa
    wl = W.make_prefix_shared("timeout-step", "f16", 2, 4, 8, 2, 128, 16, seed=92, len_range=(8, 600),
                              prefix_range=(20, 300), partition_size=-1)
    try:
        pa.pa_set_test_wait_limit(LIMIT_NS)
        fused_step(wl, check_error=False)
    finally:
        pa.pa_set_test_wait_limit(0)
    assert pa.pa_get_device_error() == TIMEOUT
    out, _ = fused_step(wl)                      # a fresh upload, normal waits
    k, v = oracle_pools(wl)
    assert_close(as_f64(out), oracle_out(wl, k, v), "f16", what="fused step after a timed-out call")


def test_prefill_wait_that_runs_out_reports_a_timeout_and_the_next_call_is_correct():
    import oracle
    import paged_kv_cache_306_gb300 as pa
    wl = W.make_prefill("timeout-prefill", "bf16", [0, 40, 200, 700], [70, 9, 33, 130], 8, 2, 128, 16, seed=93)
    t = upload(wl)
    qsl = torch.from_numpy(wl.query_start_loc).cuda()
    pa.pa_reshape_and_cache(t["key"], t["value"], t["k_cache"], t["v_cache"], t["slot_mapping"])
    assert pa.pa_get_device_error() == 0

    def prefill():
        out = torch.empty_like(t["q"])
        pa.pa_prefill(out, t["q"], t["k_cache"], t["v_cache"], t["block_tables"], t["seq_lens"], qsl, wl.scale,
                      wl.max_seq_len)
        return out
    try:
        pa.pa_set_test_wait_limit(LIMIT_NS)
        prefill()
    finally:
        pa.pa_set_test_wait_limit(0)
    assert pa.pa_get_device_error() == TIMEOUT
    out = prefill()
    assert pa.pa_get_device_error() == 0
    k, v = wl.clone_pools()
    oracle.reshape_and_cache(wl.key, wl.value, k, v, wl.slot_mapping, wl.dtype)
    ref = oracle.prefill(wl.q, k, v, wl.block_tables, wl.seq_lens, wl.query_start_loc, wl.scale, wl.dtype)
    got = as_f64(out)
    assert np.all(np.isfinite(got))
    assert_close(got, ref, "bf16", what="prefill after a timed-out call")
