"""Benchmark of one decode step of one attention layer over a paged KV pool.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload long|qwen|llama|mixed|tiny] [--block-size 16|32]
                    [--kv-dtype fp8] [--step fused|separate] [--calls C] [--configs all|none|LIST]

The headline workload is the long-context split-KV layer (4 sequences of 32K to
128K tokens, 32 query / 8 kv heads, head size 128, bf16, PARTITION_SIZE 512).
A step is the whole hot path on one batch: copy-on-write block copies (the
mixed workload only), the write of every sequence's new token, and decode
attention with its partition merge.  By default the step is one pa_decode_step
(pa_decode_step_scaled for an FP8 pool) call, which does all three;
--step separate times pa_copy_blocks + the write + decode instead.

`value` is algorithmic bytes per step / step time over exactly K back-to-back
steps (inputs resident in HBM, pool copies rotated so K/V always come from HBM).
A physical block referenced by several sequences counts once (its bytes leave
DRAM once).  `roofline` times C single calls (default 200, whatever K is), each
between CUDA events on the launching stream, and reports the median, p10 and
p90.  `e2e` is the same step through the Python API with the step's inputs
copied from pinned host memory and the output copied back inside the timed
region.  `configs` repeats the call and step measurements for every other
workload (the other decode layers, both block sizes of the mixed batch, and the
FP8 pools).  Rank 0 prints one JSON line.

--mode prefill times chunked prefill instead (16 sequences of a Qwen2.5-7B-shaped
layer, a chunk of 512 new tokens each after 0..3584 cached ones): a step is the
chunk's reshape_and_cache and the prefill; the metric is attention TFLOP/s
(4 * head_size * keys attended, summed over query rows and heads) against the
measured dense bf16 tensor peak.

--kv-dtype fp8 keeps the workload's shapes and query dtype but stores the pool
as FP8 E4M3 codes (quantising write, dequantising decode); bytes are counted at
one byte per cached element.

--impl reference times the CPU oracle on the host cores instead: each step is a
bounded sample of the same workload (one sequence, a subset of its heads).
"""
import argparse
import json
import math
import os
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads as W  # noqa: E402

METRIC = "paged-decode KV read GB/s (% of GB300 HBM peak) and decode tokens/s per layer"
WORKLOADS = {"tiny": 1, "qwen": 2, "llama": 3, "long": 4, "mixed": 5}
L2_BYTES = 126 * 1024 * 1024
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0
PREFILL_METRIC = "paged chunked-prefill attention TFLOP/s (% of GB300 dense bf16 tensor peak)"
# the workloads measured beside the headline: (key, workload, block size, kv dtype, plain call);
# the prefix-sharing batch once more through the plain call shows what shared reads gain
SUBRECORDS = [
    ("qwen", 2, None, None, False), ("llama", 3, None, None, False), ("mixed-bs16", 5, 16, None, False),
    ("mixed-bs32", 5, 32, None, False), ("mixed-bs16-plain", 5, 16, None, True), ("tiny", 1, None, None, False),
    ("long-fp8", 4, None, "fp8", False), ("qwen-fp8", 2, None, "fp8", False), ("llama-fp8", 3, None, "fp8", False),
    ("mixed-bs16-fp8", 5, 16, "fp8", False),
]


# --- byte accounting ------------------------------------------------------------------------

def decode_bytes(wl, unique=False):
    """Algorithmic bytes of one decode call: K and V of the valid tokens (per kv head),
    q and out, the block-table entries walked and seq_lens.  unique=True counts
    shared physical blocks once (prefix sharing)."""
    e, eq = W.ELEM_BYTES[wl.dtype], W.ELEM_BYTES[wl.q_dtype]
    tokens = wl.unique_tokens if unique else wl.total_tokens
    kv = tokens * wl.num_kv_heads * wl.head_size * e * 2
    qo = 2 * wl.num_seqs * wl.num_heads * wl.head_size * eq
    tables = int(np.sum(-(-wl.seq_lens.astype(np.int64) // wl.block_size))) * 4 + 4 * wl.num_seqs
    return kv + qo + tables


def write_bytes(wl):
    """reshape_and_cache (read key/value, write the slots) and block copies (read + write)."""
    e, eq = W.ELEM_BYTES[wl.dtype], W.ELEM_BYTES[wl.q_dtype]
    tok = wl.num_seqs * wl.num_kv_heads * wl.head_size * (e + eq) * 2 + wl.num_seqs * 8
    blk = wl.num_kv_heads * wl.head_size * wl.block_size * e * 2
    return tok + len(wl.cow) * blk * 2 + len(wl.cow) * 16


def step_bytes(wl):
    """Algorithmic bytes of one whole step (write and copies, then decode), shared
    physical blocks counted once: the numerator of `value`."""
    return decode_bytes(wl, unique=True) + write_bytes(wl)


def call_bytes(wl, fused):
    """Algorithmic bytes of the single timed call: the fused step also writes."""
    return decode_bytes(wl, unique=True) + (write_bytes(wl) if fused else 0)


def measured_peaks(key="hbm_gbs"):
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d[key]), "measured"
    return (FALLBACK_HBM_GBS if key == "hbm_gbs" else FALLBACK_BF16_TFLOPS), "fallback"


def prefill_flops(wl):
    """Useful flops of one prefill: query token i of a chunk of n (sequence of L tokens)
    sees L - n + i + 1 keys; QK^T and PV take 2 * head_size flops per key each."""
    total = 0
    for s in range(wl.num_seqs):
        L = int(wl.seq_lens[s])
        n = int(wl.query_start_loc[s + 1] - wl.query_start_loc[s])
        keys = n * (L - n + 1) + n * (n - 1) // 2
        total += 4 * wl.head_size * wl.num_heads * keys
    return total


def spread(ms):
    """Median, p10 and p90 of per-call times (ms) in microseconds."""
    a = np.asarray(ms, dtype=np.float64) * 1e3
    return {"median": round(float(np.median(a)), 3), "p10": round(float(np.percentile(a, 10)), 3),
            "p90": round(float(np.percentile(a, 90)), 3)}


# --- clocks --------------------------------------------------------------------------------

class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons while the GPU work runs;
    summaries are taken afterwards over the time window of each timed region."""
    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    NAMES = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.path = None
        self.rows = []

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100", "-f", self.path], stdout=subprocess.DEVNULL, stderr=subprocess.DEVNULL)
        except (OSError, ValueError):
            self.proc = None
        time.sleep(0.3)

    def stop(self):
        if self.proc is None:
            return
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        with open(self.path) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) < 10:
                    continue
                try:
                    ts = time.mktime(time.strptime(parts[0].split(".")[0], "%Y/%m/%d %H:%M:%S"))
                    ts += float("0." + parts[0].split(".")[1]) if "." in parts[0] else 0.0
                    self.rows.append((ts, float(parts[2]), float(parts[3]), parts[6:10]))
                except (ValueError, IndexError):
                    continue
        os.unlink(self.path)

    def window(self, t0, t1):
        """Median SM clock, its maximum and the throttle reasons seen within [t0, t1]
        (the nearest samples when the window is shorter than the sampling period)."""
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        inside = [r for r in self.rows if t0 - 0.15 <= r[0] <= t1 + 0.15]
        if not inside and self.rows:
            mid = 0.5 * (t0 + t1)
            inside = [min(self.rows, key=lambda r: abs(r[0] - mid))]
        if not inside:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        reasons = sorted({self.NAMES[i] for r in inside for i, v in enumerate(r[3]) if v.lower() == "active"})
        return {"sm_mhz": float(np.median([r[1] for r in inside])), "sm_max_mhz": max(r[2] for r in inside),
                "reasons": reasons, "samples": len(inside)}


# --- distributed plumbing (one process per GPU; replicas, no data-path collective) ---------

def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def max_over_ranks(value, world_size, device=None):
    """MAX of a per-rank scalar (the timed duration) over all ranks."""
    if world_size <= 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world_size, device=None):
    if world_size > 1:
        import torch.distributed as dist
        if device is not None:
            dist.barrier(device_ids=[device.index])
        else:
            dist.barrier()


# --- the workload description (identical in both arms) ---------------------------------------

def pool_bytes(wl):
    return wl.num_blocks * wl.num_kv_heads * wl.head_size * wl.block_size * W.ELEM_BYTES[wl.dtype] * 2


def pool_copies(wl):
    """Copies of the pool rotated between steps so that >= 4x L2 of K/V lies between
    two uses of one copy."""
    return max(2, math.ceil(4 * L2_BYTES / pool_bytes(wl)))


def describe(wl, cfg):
    L = wl.seq_lens
    d = {"workload": wl.name, "num_seqs": wl.num_seqs, "num_heads": wl.num_heads,
         "num_kv_heads": wl.num_kv_heads, "head_size": wl.head_size, "block_size": wl.block_size,
         "seq_lens": {"min": int(L.min()), "max": int(L.max()), "total": int(L.sum())},
         "num_blocks": wl.num_blocks, "cow_copies": int(len(wl.cow)), "seed": 306 + cfg}
    if wl.dtype == "fp8":
        d.update({"kv_cache_dtype": "fp8_e4m3", "q_dtype": wl.q_dtype, "k_scale": wl.k_scale,
                  "v_scale": wl.v_scale})
    return d


def config_dict(args, wl, cfg):
    """The workload as both arms state it: shapes, seed, split, step and the L2 rule."""
    ps = wl.partition_size if args.partition is None else args.partition
    d = describe(wl, cfg)
    call = "pa_decode_shared" if uses_shared(args, wl) else "pa_decode_step"
    d.update({"partition_size": "auto" if ps == -1 else int(ps),
              "step": (f"fused: one {call} call (block copies, new tokens and decode) + merge"
                       if uses_fused_step(args, wl) else
                       "separate: pa_copy_blocks + reshape_and_cache + " +
                       ("pa_decode_shared" if uses_shared(args, wl) else "decode")),
              "l2": f"inputs larger than L2: {pool_copies(wl)} pool copies of {pool_bytes(wl) / 1e6:.0f} MB "
                    f"rotated between steps",
              "bytes": "shared physical blocks counted once"})
    return d


def dtype_label(wl):
    """The arithmetic type of the path: an FP8 pool is widened to the query dtype."""
    return wl.dtype if wl.dtype != "fp8" else f"fp8_e4m3 cache, {wl.q_dtype} compute"


def uses_fused_step(args, wl):
    """One pa_decode_step(_scaled) call per step unless --step separate."""
    return args.step == "fused"


def uses_shared(args, wl):
    """Batches of forked sequences (the mixed workload) go through pa_decode_shared,
    which reads each shared block once per cluster, unless --plain."""
    return "group_size" in wl.meta and not getattr(args, "plain", False)


def pa_dtype(wl):
    import torch
    return {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}[wl.q_dtype]


# --- our arm ---------------------------------------------------------------------------------

def api_calls(wl):
    """(write, decode, step) through the public API for the workload's cache dtype."""
    import paged_kv_cache_306_gb300 as pa
    if wl.dtype != "fp8":
        def fused(out, q, key, value, k, v, cow, bt, sl, scale, msl, ps, ws, stream=None):
            return pa.pa_decode_step(out, q, key, value, k, v, cow, bt, sl, scale, msl, ps, ws, stream=stream)
        return pa.pa_reshape_and_cache, pa.pa_decode, fused

    def write(key, value, k, v, slots, stream=None):
        pa.pa_reshape_and_cache_scaled(key, value, k, v, slots, wl.k_scale, wl.v_scale, stream=stream)

    def decode(out, q, k, v, bt, sl, scale, max_seq_len, partition_size, ws, stream=None):
        return pa.pa_decode_scaled(out, q, k, v, bt, sl, scale, max_seq_len, wl.k_scale, wl.v_scale,
                                   partition_size, ws, stream=stream)

    def fused(out, q, key, value, k, v, cow, bt, sl, scale, msl, ps, ws, stream=None):
        return pa.pa_decode_step_scaled(out, q, key, value, k, v, cow, bt, sl, scale, msl, wl.k_scale, wl.v_scale,
                                        ps, ws, stream=stream)
    return write, decode, fused


def oracle_pools_after_write(wl):
    """The pool as the step leaves it (block copies, then the new tokens), by the oracle."""
    import oracle
    k, v = wl.clone_pools()
    oracle.copy_blocks(k, v, wl.cow, wl.dtype)
    if wl.dtype == "fp8":
        oracle.reshape_and_cache_scaled(wl.key, wl.value, k, v, wl.slot_mapping, wl.q_dtype, wl.dtype, wl.k_scale,
                                        wl.v_scale)
    else:
        oracle.reshape_and_cache(wl.key, wl.value, k, v, wl.slot_mapping, wl.dtype)
    return k, v


def oracle_decode(wl, q, k, v, sub):
    import oracle
    return oracle.decode(q, k, v, sub.block_tables, sub.seq_lens, wl.scale, wl.dtype, q_dtype=wl.q_dtype,
                         k_scale=wl.k_scale, v_scale=wl.v_scale)


class Runner:
    """A workload resident on the GPU (rotated pool copies, tables, workspace) and its step."""

    def __init__(self, args, wl, dev, stream):
        import torch
        import paged_kv_cache_306_gb300 as pa
        self.wl, self.dev, self.stream = wl, dev, stream
        self.copies = pool_copies(wl)
        free = torch.cuda.mem_get_info(dev)[0]
        self.copies = max(1, min(self.copies, int(0.6 * free // pool_bytes(wl))))
        self.sets = []
        for _ in range(self.copies):
            self.sets.append({
                "q": W.to_torch(wl.q, wl.q_dtype, dev), "key": W.to_torch(wl.key, wl.q_dtype, dev),
                "value": W.to_torch(wl.value, wl.q_dtype, dev), "k": W.to_torch(wl.k_cache, wl.dtype, dev),
                "v": W.to_torch(wl.v_cache, wl.dtype, dev),
                "out": torch.empty(wl.q.shape, dtype=pa_dtype(wl), device=dev)})
        self.bt = torch.from_numpy(wl.block_tables).to(dev)
        self.sl = torch.from_numpy(wl.seq_lens).to(dev)
        self.slots = torch.from_numpy(wl.slot_mapping).to(dev)
        self.cow = torch.from_numpy(np.ascontiguousarray(wl.cow)).to(dev)
        self.ps = wl.partition_size if args.partition is None else args.partition
        code = {"f32": pa.PA_F32, "f16": pa.PA_F16, "bf16": pa.PA_BF16, "fp8": pa.PA_FP8_E4M3}[wl.dtype]
        self.resolved = pa.pa_decode_plan_partition(wl.num_seqs, wl.num_heads, wl.num_kv_heads, wl.head_size,
                                                    wl.max_seq_len, wl.block_size, code) if self.ps == -1 else self.ps
        need = pa.pa_decode_workspace_size(wl.num_seqs, wl.num_heads, wl.num_kv_heads, wl.head_size,
                                           wl.max_seq_len, wl.block_size, self.resolved, code)
        self.ws = torch.empty(max(need, 16), dtype=torch.uint8, device=dev)
        self.write, self.decode, self.fused_call = api_calls(wl)
        self.fused = uses_fused_step(args, wl)
        self.shared = uses_shared(args, wl)
        if self.shared:  # the forked sequences' prefix groups, and the larger workspace of the shared call
            grp, blk = W.prefix_groups(wl.block_tables, wl.seq_lens, wl.block_size)
            self.grp, self.blk = torch.from_numpy(grp).to(dev), torch.from_numpy(blk).to(dev)
            need = pa.pa_decode_shared_workspace_size(wl.num_seqs, wl.num_heads, wl.num_kv_heads, wl.head_size,
                                                      wl.max_seq_len, wl.block_size, self.resolved, code)
            self.ws = torch.empty(max(need, 16), dtype=torch.uint8, device=dev)
            self.fused_call, self.decode = self._shared_calls()

    def _shared_calls(self):
        import paged_kv_cache_306_gb300 as pa
        wl = self.wl

        def fused(out, q, key, value, k, v, cow, bt, sl, scale, msl, ps, ws, stream=None, grp=None, blk=None):
            return pa.pa_decode_shared(out, q, key, value, k, v, cow, bt, sl, self.grp if grp is None else grp,
                                       self.blk if blk is None else blk, scale, msl, wl.k_scale, wl.v_scale, ps, ws,
                                       stream=stream)

        def decode(out, q, k, v, bt, sl, scale, msl, ps, ws, stream=None, grp=None, blk=None):
            return pa.pa_decode_shared(out, q, None, None, k, v, None, bt, sl, self.grp if grp is None else grp,
                                       self.blk if blk is None else blk, scale, msl, wl.k_scale, wl.v_scale, ps, ws,
                                       stream=stream)
        return fused, decode

    def step(self, i, ev=None):
        """Step i on pool copy i mod copies; with `ev`, events around the timed call."""
        wl, s, st = self.wl, self.sets[i % self.copies], self.stream
        cow = self.cow if len(wl.cow) else None
        if self.fused:
            if ev is not None:
                ev[0].record(st)
            self.fused_call(s["out"], s["q"], s["key"], s["value"], s["k"], s["v"], cow, self.bt, self.sl, wl.scale,
                            wl.max_seq_len, self.resolved, self.ws, stream=st)
            if ev is not None:
                ev[1].record(st)
            return
        import paged_kv_cache_306_gb300 as pa
        if cow is not None:
            pa.pa_copy_blocks(s["k"], s["v"], cow, stream=st)
        self.write(s["key"], s["value"], s["k"], s["v"], self.slots, stream=st)
        if ev is not None:
            ev[0].record(st)
        self.decode(s["out"], s["q"], s["k"], s["v"], self.bt, self.sl, wl.scale, wl.max_seq_len, self.resolved,
                    self.ws, stream=st)
        if ev is not None:
            ev[1].record(st)

    def timed_steps(self, steps, world_size=1):
        """Exactly `steps` steps back to back between events; returns (ms, launches, t0, t1)."""
        import torch
        import paged_kv_cache_306_gb300 as pa
        start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        barrier(world_size, self.dev)
        torch.cuda.synchronize(self.dev)
        launches0 = pa.pa_launch_count()
        t0 = time.time()
        start.record(self.stream)
        for i in range(steps):
            self.step(i)
        stop.record(self.stream)
        torch.cuda.synchronize(self.dev)
        t1 = time.time()
        launches = pa.pa_launch_count() - launches0
        barrier(world_size, self.dev)
        return start.elapsed_time(stop), launches, t0, t1

    def timed_calls(self, calls):
        """`calls` single calls, each between events on the launching stream; per-call ms."""
        import torch
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(calls)]
        torch.cuda.synchronize(self.dev)
        t0 = time.time()
        for i in range(calls):
            self.step(i, evs[i])
        torch.cuda.synchronize(self.dev)
        t1 = time.time()
        return [a.elapsed_time(b) for a, b in evs], t0, t1


def device_error_check(where):
    import paged_kv_cache_306_gb300 as pa
    code = pa.pa_get_device_error()
    if code != 0:
        raise RuntimeError(f"device error {code} ({pa.DEVICE_ERRORS.get(code)}) {where}")


def traffic_key(wl, shared):
    """The name a call's DRAM record is kept under: a batch of forked sequences taken
    through the plain call (--plain) is a different call from the shared one."""
    return wl.name + ("-plain" if "group_size" in wl.meta and not shared else "")


def roofline_of(wl, fused, call_ms, peak, peak_kind, shared=False):
    nbytes = call_bytes(wl, fused)
    med = float(np.median(call_ms))
    achieved = nbytes / (med * 1e-3) / 1e9
    if shared:
        kernel = ("shared-prefix call: copy_blocks_kernel (when the step has copies) + decode_kernel (new tokens, "
                  "decode) + decode_merge_kernel")
    elif fused:
        kernel = ("fused step call: copy_blocks_kernel (when the step has copies) + decode_kernel (new tokens, "
                  "decode) + decode_merge_kernel")
    else:
        kernel = "decode call: decode_kernel + decode_merge_kernel"
    return {"bound": "hbm", "achieved": round(achieved, 2), "peak": peak, "unit": "GB/s",
            "frac": round(achieved / peak, 4), "traffic": load_traffic(wl, fused, shared),
            "kernel": kernel,
            "bytes_per_launch": int(nbytes), "launch_us": spread(call_ms), "calls": len(call_ms),
            "peak_source": f"{peak_kind} hbm_gbs (of {peak_kind})"}


def run_ours(args, wl, cfg, world_size, rank, local_rank):
    import torch
    import paged_kv_cache_306_gb300 as pa

    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream(dev)
    r = Runner(args, wl, dev, stream)
    for i in range(args.warmup):
        r.step(i)
    torch.cuda.synchronize(dev)
    device_error_check("during warm-up")

    sampler = ClockSampler(local_rank) if rank == 0 else None
    if sampler:
        sampler.start()
    ms_total, launches, t0, t1 = r.timed_steps(args.steps, world_size)
    device_error_check("in the timed region")
    ms_total = max_over_ranks(ms_total, world_size, dev)
    ms_step = ms_total / args.steps

    # single calls between events on the launching stream: a fixed count, whatever --steps is
    call_ms, c0, c1 = r.timed_calls(args.calls)
    device_error_check("in the per-call pass")
    e2e = run_e2e(args, r)
    peak, peak_kind = measured_peaks()
    sbytes = step_bytes(wl)
    line = {
        "metric": METRIC, "value": round(world_size * sbytes / (ms_step * 1e-3) / 1e9, 2), "unit": "GB/s",
        "n_gpus": world_size, "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_step, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": dtype_label(wl),
        "data": "synthetic (seeded N(0,1) K/V/q, shuffled physical blocks)", "config": config_dict(args, wl, cfg),
        "roofline": roofline_of(wl, r.fused, call_ms, peak, peak_kind, r.shared),
        "tokens_per_s_per_layer": round(world_size * wl.num_seqs / (ms_step * 1e-3), 1),
        "detail": {"decode_bytes": int(decode_bytes(wl)), "decode_unique_bytes": int(decode_bytes(wl, unique=True)),
                   "write_bytes": int(write_bytes(wl)), "step_bytes": int(sbytes),
                   "pct_of_hbm_peak_step": round(100 * sbytes / (ms_step * 1e-3) / 1e9 / peak, 2),
                   "partition_size_resolved": int(r.resolved), "pool_copies_rotated": r.copies,
                   "parallelism": f"replicas x{world_size}", "peak_gbs": peak, "peak_kind": peak_kind},
        "e2e": e2e, "gpu_launches": int(launches),
    }
    del r
    torch.cuda.empty_cache()
    subs = []
    windows = []
    if args.configs != "none" and world_size == 1:
        keys = [k for k, *_ in SUBRECORDS] if args.configs == "all" else args.configs.split(",")
        for key in keys:
            rec, win = run_subrecord(args, key, dev, stream, peak, peak_kind)
            subs.append(rec)
            windows.append(win)
    if sampler:
        sampler.stop()
        line["clocks"] = sampler.window(t0, t1)
        line["clocks_calls"] = sampler.window(c0, c1)
        for rec, win in zip(subs, windows):
            rec["clocks"] = sampler.window(*win)
    if subs:
        line["configs"] = subs
    return line


def run_subrecord(args, key, dev, stream, peak, peak_kind):
    """Call and step measurements of one other workload, as for the headline."""
    import torch
    spec = {k: (c, bs, kd, plain) for k, c, bs, kd, plain in SUBRECORDS}
    if key not in spec:
        raise SystemExit(f"unknown --configs entry {key!r}")
    cfg, bs, kd, plain = spec[key]
    wl = W.config(cfg, poison=False, block_size=bs, kv_dtype=kd)
    sub_args = argparse.Namespace(**{**vars(args), "partition": None, "plain": plain})
    r = Runner(sub_args, wl, dev, stream)
    for i in range(max(3, args.warmup)):
        r.step(i)
    torch.cuda.synchronize(dev)
    steps = max(args.steps, 20)
    ms, _, t0, _ = r.timed_steps(steps)
    call_ms, _, t1 = r.timed_calls(args.calls)
    device_error_check(f"in sub-record {key}")
    ms_step = ms / steps
    sbytes = step_bytes(wl)
    roof = roofline_of(wl, r.fused, call_ms, peak, peak_kind, r.shared)
    rec = {"workload": wl.name, "dtype": dtype_label(wl), "partition_size": "auto" if r.ps == -1 else int(r.ps),
           "call_us": roof["launch_us"], "calls": len(call_ms), "bytes_per_call": roof["bytes_per_launch"],
           "call_gbs": roof["achieved"], "frac": roof["frac"], "traffic": roof["traffic"],
           "step_us": round(ms_step * 1e3, 3), "steps": steps,
           "value_gbs": round(sbytes / (ms_step * 1e-3) / 1e9, 2),
           "pct_of_hbm_peak_step": round(100 * sbytes / (ms_step * 1e-3) / 1e9 / peak, 2),
           "tokens_per_s_per_layer": round(wl.num_seqs / (ms_step * 1e-3), 1),
           "decode_bytes": int(decode_bytes(wl)), "decode_unique_bytes": int(decode_bytes(wl, unique=True)),
           "step": "fused" if r.fused else "separate", "pool_copies_rotated": r.copies,
           "call": "pa_decode_shared" if r.shared else (("pa_decode_step_scaled" if wl.dtype == "fp8" else "pa_decode_step")
                                                   if r.fused else "pa_decode")}
    if cfg == 1:
        rec["note"] = "latency-bound batch (4 short sequences): no roofline claim"
    del r
    torch.cuda.empty_cache()
    return rec, (t0, t1)


def run_e2e(args, r):
    """Same step through the Python API, with the step's inputs copied from pinned
    host memory and the output copied back, every step.  The inputs are packed in
    one pinned staging buffer (one host-to-device copy per step)."""
    import torch
    wl, dev, stream, s = r.wl, r.dev, r.stream, r.sets[0]
    parts = {
        "q": W.to_torch(wl.q, wl.q_dtype, "cpu"),
        "key": W.to_torch(wl.key, wl.q_dtype, "cpu"),
        "value": W.to_torch(wl.value, wl.q_dtype, "cpu"),
        "bt": torch.from_numpy(wl.block_tables),
        "sl": torch.from_numpy(wl.seq_lens),
        "slots": torch.from_numpy(wl.slot_mapping),
        "cow": torch.from_numpy(np.ascontiguousarray(wl.cow)),
    }
    if r.fused:  # the fused step finds each new token's slot through the block table
        del parts["slots"]
    if r.shared:  # the prefix groups travel with the step's tables
        parts["grp"], parts["blk"] = r.grp.cpu(), r.blk.cpu()
    offs, off = {}, 0
    for k, t in parts.items():
        offs[k] = off
        off += (t.numel() * t.element_size() + 255) // 256 * 256
    h_stage = torch.empty(off, dtype=torch.uint8).pin_memory()
    d_stage = torch.empty(off, dtype=torch.uint8, device=dev)
    devt = {}
    for k, t in parts.items():
        nb = t.numel() * t.element_size()
        h_stage[offs[k]:offs[k] + nb].copy_(t.contiguous().view(-1).view(torch.uint8))
        devt[k] = d_stage[offs[k]:offs[k] + nb].view(t.dtype).view(t.shape)
    out_host = torch.empty(wl.q.shape, dtype=pa_dtype(wl)).pin_memory()
    h2d = off
    d2h = out_host.numel() * out_host.element_size()
    steps = min(args.steps, 2000)
    cow = devt["cow"] if len(wl.cow) else None
    import paged_kv_cache_306_gb300 as pa

    kw = {"grp": devt["grp"], "blk": devt["blk"]} if r.shared else {}

    def step():
        d_stage.copy_(h_stage, non_blocking=True)
        if r.fused:
            r.fused_call(s["out"], devt["q"], devt["key"], devt["value"], s["k"], s["v"], cow, devt["bt"],
                         devt["sl"], wl.scale, wl.max_seq_len, r.resolved, r.ws, stream=stream, **kw)
        else:
            if cow is not None:
                pa.pa_copy_blocks(s["k"], s["v"], cow, stream=stream)
            r.write(devt["key"], devt["value"], s["k"], s["v"], devt["slots"], stream=stream)
            r.decode(s["out"], devt["q"], s["k"], s["v"], devt["bt"], devt["sl"], wl.scale, wl.max_seq_len,
                     r.resolved, r.ws, stream=stream, **kw)
        out_host.copy_(s["out"], non_blocking=True)

    for _ in range(3):
        step()
    torch.cuda.synchronize(dev)
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for _ in range(steps):
        step()
    b.record(stream)
    torch.cuda.synchronize(dev)
    ms = a.elapsed_time(b) / steps
    return {"value": round(step_bytes(wl) / (ms * 1e-3) / 1e9, 2), "unit": "GB/s",
            "ms_per_step": round(ms, 5), "steps": steps, "h2d_bytes_per_step": int(h2d),
            "d2h_bytes_per_step": int(d2h), "copies_per_step": 2}


def load_traffic(wl, fused, shared=False):
    """DRAM bytes per timed call from the committed ncu summary, if it was taken on the
    current kernel source and on the same kind of call; otherwise null."""
    p = os.path.join(ROOT, "profiles", "decode_traffic.json")
    if not os.path.exists(p):
        return None
    try:
        import hashlib
        d = json.load(open(p))
        src = open(os.path.join(ROOT, "paged_kv_cache_306_gb300", "csrc", "decode_kernels.cuh"), "rb").read()
        if d.get("kernel_sha256") != hashlib.sha256(src).hexdigest():
            return None
        ent = d.get("workloads", {}).get(traffic_key(wl, shared))
        if not ent or ent.get("fused", True) != fused:
            return None
        return ent.get("dram_bytes_per_launch")
    except (OSError, ValueError, KeyError):
        return None


def load_prefill_traffic(wl):
    """DRAM bytes per prefill launch from the committed ncu summary, if it was taken on
    the current prefill kernel source; otherwise null."""
    p = os.path.join(ROOT, "profiles", "prefill_traffic.json")
    if not os.path.exists(p):
        return None
    try:
        import hashlib
        d = json.load(open(p))
        src = open(os.path.join(ROOT, "paged_kv_cache_306_gb300", "csrc", "prefill_ws.cuh"), "rb").read()
        if d.get("kernel_sha256") != hashlib.sha256(src).hexdigest():
            return None
        return d.get("workloads", {}).get(wl.name, {}).get("dram_bytes_per_launch")
    except (OSError, ValueError, KeyError):
        return None


# --- the CPU oracle (reference arm and cpu_baseline) ------------------------------------------

def cpu_baseline(wl, seconds=12.0):
    """The oracle on the host cores over a bounded sample: whole sequences, all heads.
    Also a shorter single-thread pass over the same sequences, for the ratio."""
    import oracle
    # the oracle sees the pool after the step's write (as the GPU does)
    k, v = oracle_pools_after_write(wl)
    order = np.argsort(wl.seq_lens)             # shortest first keeps the sample bounded
    e = W.ELEM_BYTES[wl.dtype]

    def run(budget):
        done, nbytes, t0 = 0, 0, time.perf_counter()
        while time.perf_counter() - t0 < budget and done < wl.num_seqs:
            s = int(order[done])
            sub = W.subset(wl, [s])
            oracle_decode(wl, sub.q, k, v, sub)
            nbytes += int(wl.seq_lens[s]) * wl.num_kv_heads * wl.head_size * e * 2
            done += 1
        return done, nbytes, time.perf_counter() - t0

    cores = oracle.num_threads()
    done, nbytes, dt = run(seconds)
    oracle.set_num_threads(1)
    done1, nbytes1, dt1 = run(seconds / 4)
    oracle.set_num_threads(cores)
    all_core, one_core = nbytes / dt / 1e9, nbytes1 / dt1 / 1e9
    return {"value": round(all_core, 4), "unit": "GB/s", "cores": cores, "kind": "oracle",
            "single_core_value": round(one_core, 4), "all_vs_single": round(all_core / one_core, 2),
            "sample": f"{done} of {wl.num_seqs} sequences (shortest first), all heads, {dt:.1f} s on {cores} "
                      f"threads; single thread: {done1} sequences, {dt1:.1f} s; fp64 C oracle"}


def run_reference(args, wl, cfg, world_size, rank):
    """The CPU oracle as the reference arm: each step is one sequence of the workload."""
    import oracle
    k, v = oracle_pools_after_write(wl)
    e = W.ELEM_BYTES[wl.dtype]
    G = wl.num_heads // wl.num_kv_heads

    def one(i, kvh):
        s = i % wl.num_seqs
        sub = W.subset(wl, [s])
        q = np.ascontiguousarray(sub.q[:, :kvh * G])
        kk = np.ascontiguousarray(k[:, :kvh]) if kvh < wl.num_kv_heads else k
        vv = np.ascontiguousarray(v[:, :kvh]) if kvh < wl.num_kv_heads else v
        oracle_decode(wl, q, kk, vv, sub)
        return int(wl.seq_lens[s]) * kvh * wl.head_size * e * 2

    # size the per-step sample (kv heads of one sequence) so the run stays within ~2 minutes
    budget = 120.0 / max(1, args.steps + args.warmup)
    t = time.perf_counter()
    one(0, 1)
    per_head = time.perf_counter() - t
    kv_sub = int(max(1, min(wl.num_kv_heads, budget // max(per_head, 1e-6))))
    if kv_sub < wl.num_kv_heads:
        k = np.ascontiguousarray(k[:, :kv_sub])
        v = np.ascontiguousarray(v[:, :kv_sub])
    for i in range(args.warmup):
        one(i, kv_sub)
    nbytes, t0 = 0, time.perf_counter()
    for i in range(args.steps):
        nbytes += one(i, kv_sub)
    dt = time.perf_counter() - t0
    value = nbytes / dt / 1e9
    sample = (f"per step one sequence of the workload (rotating), {kv_sub} of {wl.num_kv_heads} kv heads "
              f"with their {G} query heads each; fp64 C oracle")
    return {"metric": METRIC, "value": round(value, 4), "unit": "GB/s", "n_gpus": world_size, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(dt / args.steps * 1e3, 4), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": dtype_label(wl), "data": "synthetic", "impl": "reference",
            "config": config_dict(args, wl, cfg),
            "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": oracle.num_threads(),
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def run_prefill(args, world_size, rank, local_rank):
    """Chunked prefill of the Qwen2.5-7B-shaped layer: write the chunk, then prefill."""
    import torch
    import paged_kv_cache_306_gb300 as pa

    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream(dev)
    wl = W.prefill_config(poison=False)
    pbytes = wl.num_blocks * wl.num_kv_heads * wl.head_size * wl.block_size * 2 * 2
    copies = max(2, math.ceil(4 * L2_BYTES / pbytes))
    sets = [{"q": W.to_torch(wl.q, wl.dtype, dev), "key": W.to_torch(wl.key, wl.dtype, dev),
             "value": W.to_torch(wl.value, wl.dtype, dev), "k": W.to_torch(wl.k_cache, wl.dtype, dev),
             "v": W.to_torch(wl.v_cache, wl.dtype, dev), "out": torch.empty(wl.q.shape, dtype=torch.float16, device=dev)}
            for _ in range(copies)]
    bt = torch.from_numpy(wl.block_tables).to(dev)
    sl = torch.from_numpy(wl.seq_lens).to(dev)
    qsl = torch.from_numpy(wl.query_start_loc).to(dev)
    slots = torch.from_numpy(wl.slot_mapping).to(dev)

    def step(i, ev=None):
        s = sets[i % copies]
        pa.pa_reshape_and_cache(s["key"], s["value"], s["k"], s["v"], slots, stream=stream)
        if ev is not None:
            ev[0].record(stream)
        pa.pa_prefill(s["out"], s["q"], s["k"], s["v"], bt, sl, qsl, wl.scale, wl.max_seq_len, stream=stream)
        if ev is not None:
            ev[1].record(stream)

    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize(dev)
    device_error_check("during warm-up")
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    sampler = ClockSampler(local_rank) if rank == 0 else None
    if sampler:
        sampler.start()
    barrier(world_size, dev)
    torch.cuda.synchronize(dev)
    launches0 = pa.pa_launch_count()
    t0 = time.time()
    start.record(stream)
    for i in range(args.steps):
        step(i)
    stop.record(stream)
    torch.cuda.synchronize(dev)
    t1 = time.time()
    launches = pa.pa_launch_count() - launches0
    barrier(world_size, dev)
    device_error_check("in the timed region")
    ms_step = max_over_ranks(start.elapsed_time(stop), world_size, dev) / args.steps
    kn = args.calls
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(kn)]
    c0 = time.time()
    for i in range(kn):
        step(i, evs[i])
    torch.cuda.synchronize(dev)
    c1 = time.time()
    pre_ms = [a.elapsed_time(b) for a, b in evs]

    # end to end: q, key, value, tables, lengths and slots from pinned host memory, out back
    s0 = sets[0]
    parts = {"q": W.to_torch(wl.q, wl.dtype, "cpu"), "key": W.to_torch(wl.key, wl.dtype, "cpu"),
             "value": W.to_torch(wl.value, wl.dtype, "cpu"), "bt": torch.from_numpy(wl.block_tables),
             "sl": torch.from_numpy(wl.seq_lens), "qsl": torch.from_numpy(wl.query_start_loc),
             "slots": torch.from_numpy(wl.slot_mapping)}
    offs, off = {}, 0
    for k_, t_ in parts.items():
        offs[k_] = off
        off += (t_.numel() * t_.element_size() + 255) // 256 * 256
    h_stage = torch.empty(off, dtype=torch.uint8).pin_memory()
    d_stage = torch.empty(off, dtype=torch.uint8, device=dev)
    devt = {}
    for k_, t_ in parts.items():
        nb_ = t_.numel() * t_.element_size()
        h_stage[offs[k_]:offs[k_] + nb_].copy_(t_.contiguous().view(-1).view(torch.uint8))
        devt[k_] = d_stage[offs[k_]:offs[k_] + nb_].view(t_.dtype).view(t_.shape)
    out_host = torch.empty(wl.q.shape, dtype=torch.float16).pin_memory()

    def e2e_step():
        d_stage.copy_(h_stage, non_blocking=True)
        pa.pa_reshape_and_cache(devt["key"], devt["value"], s0["k"], s0["v"], devt["slots"], stream=stream)
        pa.pa_prefill(s0["out"], devt["q"], s0["k"], s0["v"], devt["bt"], devt["sl"], devt["qsl"], wl.scale,
                      wl.max_seq_len, stream=stream)
        out_host.copy_(s0["out"], non_blocking=True)

    for _ in range(3):
        e2e_step()
    torch.cuda.synchronize(dev)
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ne = min(args.steps, 500)
    a.record(stream)
    for _ in range(ne):
        e2e_step()
    b.record(stream)
    torch.cuda.synchronize(dev)
    e2e_ms = a.elapsed_time(b) / ne
    if sampler:
        sampler.stop()

    flops = prefill_flops(wl)
    peak, kind = measured_peaks("bf16_tflops")
    med = float(np.median(pre_ms))
    achieved = flops / (med * 1e-3) / 1e12
    L = wl.seq_lens
    cfg = {"workload": wl.name, "num_seqs": wl.num_seqs, "num_heads": wl.num_heads, "num_kv_heads": wl.num_kv_heads,
           "head_size": wl.head_size, "block_size": wl.block_size, "query_tokens": int(wl.query_start_loc[-1]),
           "chunk": 512, "seq_lens": {"min": int(L.min()), "max": int(L.max()), "total": int(L.sum())},
           "num_blocks": wl.num_blocks, "seed": 406,
           "l2": f"inputs larger than L2: {copies} pool copies of {pbytes / 1e6:.0f} MB rotated"}
    line = {"metric": PREFILL_METRIC, "value": round(world_size * flops / (ms_step * 1e-3) / 1e12, 2),
            "unit": "TFLOP/s", "n_gpus": world_size, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(ms_step, 5), "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "f16", "data": "synthetic (seeded N(0,1) K/V/q, shuffled physical blocks)", "config": cfg,
            "roofline": {"bound": "tensor", "achieved": round(achieved, 2), "peak": peak, "unit": "TFLOP/s",
                         "frac": round(achieved / peak, 4), "traffic": load_prefill_traffic(wl), "kernel": "prefill_ws_kernel",
                         "flops_per_launch": int(flops), "launch_us": spread(pre_ms), "calls": kn,
                         "peak_source": f"{kind} bf16_tflops (of {kind}; fp16 runs at the bf16 rate)"},
            "detail": {"flops_per_step": int(flops), "parallelism": f"replicas x{world_size}"},
            "e2e": {"value": round(flops / (e2e_ms * 1e-3) / 1e12, 2), "unit": "TFLOP/s",
                    "ms_per_step": round(e2e_ms, 5), "steps": ne, "h2d_bytes_per_step": int(off),
                    "d2h_bytes_per_step": int(out_host.numel() * 2), "copies_per_step": 2},
            "gpu_launches": int(launches)}
    if sampler:
        line["clocks"] = sampler.window(t0, t1)
        line["clocks_calls"] = sampler.window(c0, c1)
    return line, wl


def prefill_cpu_baseline(wl, seconds=12.0):
    """The oracle on the host cores over a bounded sample: the first rows of one sequence."""
    import oracle
    k, v = wl.clone_pools()
    oracle.reshape_and_cache(wl.key, wl.value, k, v, wl.slot_mapping, wl.dtype)
    s = int(np.argmin(wl.seq_lens))
    n = int(wl.query_start_loc[s + 1] - wl.query_start_loc[s])
    rows, done_flops, t0 = 8, 0, time.perf_counter()
    while True:
        r = min(rows, n)
        # the sample: the chunk's last r tokens as a chunk of their own (positions L - r ..)
        q = np.ascontiguousarray(wl.q[wl.query_start_loc[s + 1] - r:wl.query_start_loc[s + 1]])
        oracle.prefill(q, k, v, wl.block_tables[[s]], wl.seq_lens[[s]], np.array([0, r], np.int32), wl.scale,
                       wl.dtype)
        L = int(wl.seq_lens[s])
        done_flops += 4 * wl.head_size * wl.num_heads * (r * (L - r + 1) + r * (r - 1) // 2)
        dt = time.perf_counter() - t0
        if dt > seconds / 4 or r == n:
            break
        rows *= 2
    return {"value": round(done_flops / dt / 1e12, 6), "unit": "TFLOP/s", "cores": oracle.num_threads(),
            "kind": "oracle", "sample": f"the last {r} query tokens of sequence {s} ({L} tokens), all heads, "
                                        f"{dt:.1f} s, fp64 C oracle"}


def parser():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--calls", type=int, default=200, help="single calls timed between events (median, p10, p90)")
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=sorted(WORKLOADS), default="long")
    ap.add_argument("--block-size", type=int, default=None, help="mixed workload only: 16 or 32")
    ap.add_argument("--partition", type=int, default=None, help="override the workload's partition size")
    ap.add_argument("--mode", choices=["decode", "prefill"], default="decode")
    ap.add_argument("--kv-dtype", choices=["fp8"], default=None,
                    help="store the pool as FP8 E4M3 codes (not for the fp32 tiny workload)")
    ap.add_argument("--step", choices=["fused", "separate"], default="fused",
                    help="one pa_decode_step call, or copy_blocks + reshape_and_cache + decode")
    ap.add_argument("--plain", action="store_true",
                    help="run the prefix-sharing workload through pa_decode_step / decode, not pa_decode_shared")
    ap.add_argument("--configs", default="all",
                    help="other workloads measured beside the headline: all, none, or a comma list of "
                         + ",".join(k for k, *_ in SUBRECORDS))
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    return ap


def main(argv=None):
    ap = parser()
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    if args.calls < 50:
        ap.error("--calls must be at least 50")

    world_size, rank, local_rank = dist_env()
    cfg = WORKLOADS[args.workload]

    if args.mode == "prefill":
        if args.impl == "reference":
            if rank != 0:
                return 0
            wl = W.prefill_config(poison=False)
            cb = prefill_cpu_baseline(wl, seconds=min(120.0, 4.0 * (args.steps + args.warmup)))
            print(json.dumps({"metric": PREFILL_METRIC, "value": cb["value"], "unit": "TFLOP/s", "n_gpus": world_size,
                              "steps": args.steps, "warmup": args.warmup, "higher_is_better": True,
                              "scaling": "weak", "vs_baseline": None, "dtype": "f16", "data": "synthetic",
                              "impl": "reference", "config": {"workload": wl.name}, "cpu_baseline": cb,
                              "e2e": {"value": cb["value"], "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                                      "d2h_bytes_per_step": 0}}), flush=True)
            return 0
        if world_size > 1:
            import torch
            import torch.distributed as dist
            torch.cuda.set_device(local_rank)
            dist.init_process_group("nccl")
        line, wl = run_prefill(args, world_size, rank, local_rank)
        if rank == 0:
            if not args.no_cpu_baseline:
                line["cpu_baseline"] = prefill_cpu_baseline(wl, args.cpu_seconds)
            print(json.dumps(line), flush=True)
        if world_size > 1:
            import torch.distributed as dist
            dist.destroy_process_group()
        return 0

    if args.impl == "reference":
        if rank != 0:
            return 0
        wl = W.config(cfg, poison=False, block_size=args.block_size, kv_dtype=args.kv_dtype)
        print(json.dumps(run_reference(args, wl, cfg, world_size, rank)), flush=True)
        return 0

    if world_size > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl")
    # every rank holds its own replica of the workload (weak scaling)
    wl = W.config(cfg, poison=False, block_size=args.block_size, kv_dtype=args.kv_dtype)
    line = run_ours(args, wl, cfg, world_size, rank, local_rank)
    if rank == 0:
        if not args.no_cpu_baseline:
            line["cpu_baseline"] = cpu_baseline(wl, args.cpu_seconds)
        print(json.dumps(line), flush=True)
    if world_size > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
