"""Host-side pieces of bench.py, on CPU: the multi-rank timing reduction (2 gloo
ranks), the algorithmic byte accounting and the CPU reference arm's JSON line."""
import json
import os
import socket
import subprocess
import sys

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
import workloads as W  # noqa: E402


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank_main(rank, world, port, q):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    bench.barrier(world)
    q.put((rank, bench.max_over_ranks(1.5 + rank, world)))
    dist.destroy_process_group()


def test_timing_is_the_max_over_two_gloo_ranks():
    torch = pytest.importorskip("torch")
    mp = torch.multiprocessing.get_context("spawn")
    q = mp.Queue()
    port = _free_port()
    procs = [mp.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    got = dict(q.get(timeout=120) for _ in range(2))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert got == {0: 2.5, 1: 2.5}


def test_single_rank_needs_no_process_group():
    assert bench.max_over_ranks(3.25, 1) == 3.25


def test_decode_bytes_of_the_llama_layer():
    wl = W.config(3, poison=False)
    # K+V of 16 x 2048 tokens x 32 kv heads x 128 dims x 2 B, q and out, 128 table entries per sequence
    expect = 536_870_912 + 2 * 16 * 32 * 128 * 2 + 16 * 128 * 4 + 16 * 4
    assert bench.decode_bytes(wl) == expect


def test_unique_bytes_count_shared_blocks_once():
    wl = W.make_prefix_shared("t", "f16", 2, 4, 8, 2, 64, 16, seed=3, len_range=(300, 600),
                              prefix_range=(200, 250))
    assert bench.decode_bytes(wl, unique=True) < bench.decode_bytes(wl)


def test_reference_arm_prints_one_json_line():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--workload", "tiny",
                        "--steps", "3", "--warmup", "3"], capture_output=True, text=True, cwd=ROOT, timeout=600)
    assert r.returncode == 0, r.stderr
    line = json.loads(r.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["value"] > 0 and line["unit"] == "GB/s"
    assert line["config"]["workload"] == "tiny-f32" and line["config"]["bytes"]
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] >= 1
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["steps"] == 3


def test_decode_bytes_of_the_llama_layer_with_an_fp8_pool():
    wl = W.config(3, poison=False, kv_dtype="fp8")
    # K+V at one byte per element, q and out still fp16
    expect = 536_870_912 // 2 + 2 * 16 * 32 * 128 * 2 + 16 * 128 * 4 + 16 * 4
    assert bench.decode_bytes(wl) == expect
    # write: fp16 key/value in, one-byte codes out, the slot ids
    assert bench.write_bytes(wl) == 16 * 32 * 128 * (2 + 1) * 2 + 16 * 8


def test_reference_arm_with_an_fp8_pool():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--workload", "llama",
                        "--kv-dtype", "fp8", "--steps", "3", "--warmup", "3"], capture_output=True, text=True,
                       cwd=ROOT, timeout=600)
    assert r.returncode == 0, r.stderr
    line = json.loads(r.stdout.strip().splitlines()[-1])
    assert line["config"]["kv_cache_dtype"] == "fp8_e4m3" and line["value"] > 0
    assert line["dtype"].startswith("fp8_e4m3")


def test_prefill_flops_count_every_key_each_query_row_sees():
    wl = W.make_prefill("f", "f16", [0, 5, 40], [3, 17, 1], 8, 2, 64, 16, seed=1, poison=False)
    keys = sum(c + i + 1 for c, n in zip([0, 5, 40], [3, 17, 1]) for i in range(n))
    assert bench.prefill_flops(wl) == 4 * 64 * 8 * keys


def test_fused_step_is_the_default_for_every_pool():
    import argparse
    fused = argparse.Namespace(step="fused")
    separate = argparse.Namespace(step="separate")
    assert bench.uses_fused_step(fused, W.config(1, poison=False))
    assert not bench.uses_fused_step(separate, W.config(1, poison=False))
    wl8 = W.make_private("fp8", "fp8", [20, 40], 8, 2, 128, 16, seed=1, q_dtype="f16")
    assert bench.uses_fused_step(fused, wl8)


def test_value_counts_shared_blocks_once():
    wl = W.config(5, poison=False, block_size=16)
    assert bench.step_bytes(wl) == bench.decode_bytes(wl, unique=True) + bench.write_bytes(wl)
    assert bench.step_bytes(wl) < bench.decode_bytes(wl) + bench.write_bytes(wl)
    assert bench.call_bytes(wl, True) == bench.step_bytes(wl)
    assert bench.call_bytes(wl, False) == bench.decode_bytes(wl, unique=True)


def test_call_spread_is_median_and_percentiles():
    ms = [0.2] * 80 + [0.1] * 10 + [0.3] * 10 + [5.0]
    s = bench.spread(ms)
    assert s["median"] == 200.0 and s["p10"] <= 200.0 <= s["p90"]
    assert s["p90"] <= 300.0


def test_both_arms_state_the_same_config():
    import argparse
    args = argparse.Namespace(step="fused", partition=None)
    wl = W.config(4, poison=False)
    d = bench.config_dict(args, wl, 4)
    assert d["workload"] == "long-context-bf16" and d["partition_size"] == 512
    assert d == bench.config_dict(args, W.config(4, poison=False), 4)


def test_headline_defaults_to_the_long_context_layer():
    a = bench.parser().parse_args([])
    assert a.workload == "long" and a.gpus == 1 and a.calls >= 200 and a.configs == "all"
    assert bench.WORKLOADS[a.workload] == 4


def test_traffic_record_needs_the_current_kernel_source(tmp_path, monkeypatch):
    wl = W.config(1, poison=False)
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.load_traffic(wl, True) is None


def test_write_bytes_count_tokens_and_copies():
    wl = W.config(5, poison=False, block_size=16)
    e = 2
    tok = wl.num_seqs * wl.num_kv_heads * wl.head_size * (e + e) * 2 + wl.num_seqs * 8
    blk = wl.num_kv_heads * wl.head_size * wl.block_size * e * 2
    assert bench.write_bytes(wl) == tok + len(wl.cow) * (2 * blk + 16)


def test_cpu_baseline_reports_all_threads_and_one():
    wl = W.config(1, poison=False)
    cb = bench.cpu_baseline(wl, seconds=0.5)
    assert cb["kind"] == "oracle" and cb["value"] > 0 and cb["single_core_value"] > 0
    assert cb["cores"] >= 1 and cb["all_vs_single"] > 0


def test_plain_and_shared_calls_keep_separate_traffic_records():
    wl = W.config(5, poison=False, block_size=16)
    assert bench.traffic_key(wl, True) == wl.name
    assert bench.traffic_key(wl, False) == wl.name + "-plain"
    q = W.config(2, poison=False)
    assert bench.traffic_key(q, False) == q.name


def test_prefill_traffic_record_needs_the_current_kernel_source(tmp_path, monkeypatch):
    wl = W.make_prefill("f", "f16", [0, 5], [3, 17], 8, 2, 64, 16, seed=1, poison=False)
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.load_prefill_traffic(wl) is None
