"""Shared helpers for the GPU parity tests: run a decode step through the C ABI
and through the CPU oracle on the same seeded inputs, and compare."""
import numpy as np

import oracle
import workloads as W

# Max-abs tolerance on attention outputs: 2e-3 for 16-bit caches with fp32
# accumulation, 1e-5 for fp32 caches.  An FP8 cache is compared with the oracle
# reading the same codes, so only the arithmetic differs: the 16-bit bar holds.
TOL = {"f32": 1e-5, "f16": 2e-3, "bf16": 2e-3, "fp8": 2e-3}


def half_ulp(ref, dtype):
    """Half the spacing of `dtype` at |ref|: the error of the final rounding alone."""
    ax = np.abs(ref)
    if dtype == "f16":
        return 0.5 * np.spacing(ax.astype(np.float16)).astype(np.float64)
    if dtype == "bf16":
        e = np.floor(np.log2(np.maximum(ax, 2.0 ** -126)))
        return 0.5 * 2.0 ** (e - 7)
    return 0.5 * np.spacing(ax.astype(np.float32)).astype(np.float64)


def torch_dtype(dtype):
    import torch
    return {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}[dtype]


def upload(wl, device="cuda"):
    import torch
    t = {
        "q": W.to_torch(wl.q, wl.q_dtype, device),
        "key": W.to_torch(wl.key, wl.q_dtype, device),
        "value": W.to_torch(wl.value, wl.q_dtype, device),
        "k_cache": W.to_torch(wl.k_cache, wl.dtype, device),
        "v_cache": W.to_torch(wl.v_cache, wl.dtype, device),
        "block_tables": torch.from_numpy(wl.block_tables).to(device),
        "seq_lens": torch.from_numpy(wl.seq_lens).to(device),
        "slot_mapping": torch.from_numpy(wl.slot_mapping).to(device),
        "cow": torch.from_numpy(np.ascontiguousarray(wl.cow)).to(device),
    }
    return t


def gpu_step(wl, partition_size=None, t=None, write=True):
    """copy_blocks -> reshape_and_cache -> decode through the library; returns (out, tensors)."""
    import torch
    import paged_kv_cache_306_gb300 as pa
    t = upload(wl) if t is None else t
    if write:
        if len(wl.cow):
            pa.pa_copy_blocks(t["k_cache"], t["v_cache"], t["cow"])
        if wl.dtype == "fp8":
            pa.pa_reshape_and_cache_scaled(t["key"], t["value"], t["k_cache"], t["v_cache"], t["slot_mapping"],
                                           wl.k_scale, wl.v_scale)
        else:
            pa.pa_reshape_and_cache(t["key"], t["value"], t["k_cache"], t["v_cache"], t["slot_mapping"])
    out = torch.empty_like(t["q"])
    ps = wl.partition_size if partition_size is None else partition_size
    if wl.dtype == "fp8":
        pa.pa_decode_scaled(out, t["q"], t["k_cache"], t["v_cache"], t["block_tables"], t["seq_lens"], wl.scale,
                            wl.max_seq_len, wl.k_scale, wl.v_scale, ps)
    else:
        pa.pa_decode(out, t["q"], t["k_cache"], t["v_cache"], t["block_tables"], t["seq_lens"], wl.scale,
                     wl.max_seq_len, ps)
    code = pa.pa_get_device_error()
    assert code == 0, f"device error {code}: {pa.DEVICE_ERRORS.get(code)}"
    return out, t


def oracle_pools(wl, write=True):
    k, v = wl.clone_pools()
    if write:
        oracle.copy_blocks(k, v, wl.cow, wl.dtype)
        if wl.dtype == "fp8":
            oracle.reshape_and_cache_scaled(wl.key, wl.value, k, v, wl.slot_mapping, wl.q_dtype, wl.dtype,
                                            wl.k_scale, wl.v_scale)
        else:
            oracle.reshape_and_cache(wl.key, wl.value, k, v, wl.slot_mapping, wl.dtype)
    return k, v


def oracle_out(wl, k, v, seqs=None):
    sub = wl if seqs is None else W.subset(wl, seqs)
    return oracle.decode(sub.q, k, v, sub.block_tables, sub.seq_lens, wl.scale, wl.dtype, q_dtype=wl.q_dtype,
                         k_scale=wl.k_scale, v_scale=wl.v_scale)


def as_f64(out):
    import torch
    return out.detach().to(torch.float64).cpu().numpy()


def max_violation(got, ref, dtype, with_rounding, out_dtype=None):
    err = np.abs(got - ref)
    tol = TOL[dtype] + (half_ulp(ref, out_dtype or dtype) if with_rounding else 0.0)
    assert np.all(np.isfinite(got)), "non-finite output"
    return float(err.max()), float((err - tol).max())


def assert_close(got, ref, dtype, with_rounding=True, what="", out_dtype=None):
    err, worst = max_violation(got, ref, dtype, with_rounding, out_dtype)
    assert worst <= 0.0, f"{what}: max abs err {err:.3e} exceeds tolerance (excess {worst:.3e})"
    return err


def fused_step(wl, partition_size=None, t=None, workspace=None, check_error=True):
    """The same step as gpu_step in one call (pa_decode_step); returns (out, tensors)."""
    import torch
    import paged_kv_cache_306_gb300 as pa
    t = upload(wl) if t is None else t
    out = torch.empty_like(t["q"])
    ps = wl.partition_size if partition_size is None else partition_size
    if wl.dtype == "fp8":
        pa.pa_decode_step_scaled(out, t["q"], t["key"], t["value"], t["k_cache"], t["v_cache"],
                                 t["cow"] if len(wl.cow) else None, t["block_tables"], t["seq_lens"], wl.scale,
                                 wl.max_seq_len, wl.k_scale, wl.v_scale, ps, workspace)
    else:
        pa.pa_decode_step(out, t["q"], t["key"], t["value"], t["k_cache"], t["v_cache"],
                          t["cow"] if len(wl.cow) else None, t["block_tables"], t["seq_lens"], wl.scale,
                          wl.max_seq_len, ps, workspace)
    if check_error:
        code = pa.pa_get_device_error()
        assert code == 0, f"device error {code}: {pa.DEVICE_ERRORS.get(code)}"
    return out, t


def same_bytes(a, b):
    """Bitwise equality of two CUDA tensors of one dtype and shape."""
    import torch
    return a.shape == b.shape and torch.equal(a.contiguous().view(torch.uint8), b.contiguous().view(torch.uint8))
