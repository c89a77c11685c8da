"""GPU parity of the FP8 E4M3 KV cache against the CPU oracle, through the C ABI.

An FP8 pool stores the E4M3 code of x / scale (round to nearest even, finite
values beyond 448 saturate) and reads back code * scale; queries, new-token rows
and outputs stay fp16 or bf16.  The quantising write must be bit-exact against
the oracle's encoder; the attention output is compared with the fp64 oracle
reading the same codes, within 2e-3 max-abs (the bar of the 16-bit caches, as
only the arithmetic differs), plus half an output ulp on the small cases.
"""
import zlib

import numpy as np
import pytest

import oracle
import workloads as W
from helpers import TOL, as_f64, assert_close, gpu_step, max_violation, oracle_out, oracle_pools, upload

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


# --- the quantising write --------------------------------------------------------------------------

@pytest.mark.parametrize("key_dtype", ["f32", "f16", "bf16"])
@pytest.mark.parametrize("bs", [16, 32])
@pytest.mark.parametrize("scales", [(1.0 / 64, 1.0 / 32), (0.0173, 0.021)])
def test_scaled_write_is_bit_exact(key_dtype, bs, scales):
    """Codes of x / scale for ordinary values, values past 448 * scale (saturate),
    subnormal codes, exact zeros and both signs."""
    import paged_kv_cache_306_gb300 as pa
    ks, vs = scales
    rng = np.random.default_rng(zlib.crc32(repr((key_dtype, bs, scales)).encode()))
    NB, Hkv, D, T = 40, 4, 128, 57
    wl = W.make_private("w8", "fp8", [bs * 3] * 4, Hkv, Hkv, D, bs, seed=31, num_blocks=NB, poison=False,
                        q_dtype="f16", kv_scale=ks)
    x = rng.standard_normal((2, T, Hkv, D)).astype(np.float32)
    x[:, :8] *= 600.0 * ks            # beyond the largest code after division
    x[:, 8:16] *= 2.0 ** -8 * ks      # subnormal codes
    x[:, 16, :, :5] = 0.0
    x[:, 17, :, :5] = -0.0
    key, value = W.cast(x[0], key_dtype), W.cast(x[1], key_dtype)
    slots = rng.permutation(NB * bs)[:T].astype(np.int64)
    slots[[3, 10]] = -1
    t = upload(wl)
    pa.pa_reshape_and_cache_scaled(W.to_torch(key, key_dtype, "cuda"), W.to_torch(value, key_dtype, "cuda"),
                                   t["k_cache"], t["v_cache"], torch.from_numpy(slots).cuda(), ks, vs)
    assert pa.pa_get_device_error() == 0
    k, v = wl.clone_pools()
    oracle.reshape_and_cache_scaled(key, value, k, v, slots, key_dtype, "fp8", ks, vs)
    assert np.array_equal(W.from_torch(t["k_cache"], "fp8"), k)
    assert np.array_equal(W.from_torch(t["v_cache"], "fp8"), v)


def test_scaled_write_to_a_16_bit_cache_is_the_plain_write():
    import paged_kv_cache_306_gb300 as pa
    wl = W.make_private("w16", "bf16", [40, 17], 4, 2, 128, 16, seed=32, poison=False)
    t1, t2 = upload(wl), upload(wl)
    pa.pa_reshape_and_cache(t1["key"], t1["value"], t1["k_cache"], t1["v_cache"], t1["slot_mapping"])
    pa.pa_reshape_and_cache_scaled(t2["key"], t2["value"], t2["k_cache"], t2["v_cache"], t2["slot_mapping"], 1.0, 1.0)
    assert torch.equal(t1["k_cache"], t2["k_cache"]) and torch.equal(t1["v_cache"], t2["v_cache"])
    with pytest.raises(pa.PAError):
        pa.pa_reshape_and_cache_scaled(t2["key"], t2["value"], t2["k_cache"], t2["v_cache"], t2["slot_mapping"],
                                       0.5, 1.0)


def test_copy_blocks_moves_fp8_codes_bit_exactly():
    import paged_kv_cache_306_gb300 as pa
    wl = W.make_private("c8", "fp8", [64] * 6, 8, 8, 128, 16, seed=33, num_blocks=40, poison=False, q_dtype="bf16")
    used = set(wl.block_tables[wl.block_tables >= 0].tolist())
    free = [b for b in range(wl.num_blocks) if b not in used]
    pairs = np.stack([wl.block_tables[:4, 0], np.array(free[:4])], axis=1).astype(np.int64)
    t = upload(wl)
    pa.pa_copy_blocks(t["k_cache"], t["v_cache"], torch.from_numpy(pairs).cuda())
    assert pa.pa_get_device_error() == 0
    k, v = wl.clone_pools()
    oracle.copy_blocks(k, v, pairs, "fp8")
    assert np.array_equal(W.from_torch(t["k_cache"], "fp8"), k)
    assert np.array_equal(W.from_torch(t["v_cache"], "fp8"), v)


# --- decode ----------------------------------------------------------------------------------------

@pytest.mark.parametrize("q_dtype", ["f16", "bf16"])
@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("bs", [16, 32])
@pytest.mark.parametrize("G", [1, 4, 7, 20])
@pytest.mark.parametrize("part", [0, "2bs", -1])
def test_fp8_decode_matches_oracle_on_ragged_batches(q_dtype, D, bs, G, part):
    rng = np.random.default_rng(zlib.crc32(repr(("fp8", q_dtype, D, bs, G, part)).encode()))
    L = edge_lengths(bs, rng.integers(2, 400, size=3))
    ps = 2 * bs if part == "2bs" else part
    wl = W.make_private("ragged8", "fp8", L, 2 * G, 2, D, bs, seed=int(rng.integers(1 << 30)), partition_size=ps,
                        q_dtype=q_dtype)
    out, _ = gpu_step(wl)
    k, v = oracle_pools(wl)
    ref = oracle_out(wl, k, v)
    assert_close(as_f64(out), ref, "fp8", with_rounding=True, out_dtype=q_dtype,
                 what=f"fp8/{q_dtype} D{D} bs{bs} G{G} P{ps}")


@pytest.mark.parametrize("q_dtype", ["f16", "bf16"])
@pytest.mark.parametrize("G", [1, 8])
def test_fp8_decode_with_scales_that_are_not_powers_of_two(q_dtype, G):
    wl = W.make_private("odd8", "fp8", [1, 300, 1029, 64], 2 * G, 2, 128, 16, seed=34, partition_size=-1,
                        q_dtype=q_dtype, kv_scale=0.0173)
    wl.v_scale = 0.0291
    out, _ = gpu_step(wl)
    k, v = oracle_pools(wl)
    assert_close(as_f64(out), oracle_out(wl, k, v), "fp8", with_rounding=True, out_dtype=q_dtype)


@pytest.mark.parametrize("q_dtype", ["f16", "bf16"])
@pytest.mark.parametrize("G", [1, 8])
def test_fp8_seq_len_one_returns_the_dequantised_v0_bit_exactly(q_dtype, G):
    """The only token is the one just written, so out[s, h] is code(value / v_scale) * v_scale
    rounded to the query dtype; with v_scale a power of two that product is exact."""
    wl = W.make_private("one8", "fp8", [1, 1, 1], 2 * G, 2, 128, 16, seed=35, partition_size=0, q_dtype=q_dtype)
    out, t = gpu_step(wl)
    vals = t["v_cache"].float()[:, :, :, 0]            # slot 0 of each block: [NB, Hkv, D]
    blocks = torch.from_numpy(wl.block_tables[:, 0].astype(np.int64)).cuda()
    v0 = (vals[blocks] * wl.v_scale).to(out.dtype).repeat_interleave(G, dim=1)
    assert torch.equal(out.view(torch.int16), v0.view(torch.int16))


@pytest.mark.parametrize("q_dtype", ["f16", "bf16"])
@pytest.mark.parametrize("G", [1, 4])
def test_fp8_decode_widens_every_finite_code_exactly(q_dtype, G):
    """Every finite E4M3 code goes through the decode kernel's widening: one-token
    sequences whose cached V rows hold all 254 finite codes (each twice; the two NaN
    codes replaced by 0), their K rows code 0, read by a decode-only call (G = 4 takes
    the tensor-core path, G = 1 the CUDA-core one).  With one token P = 1, so each output
    element is its code's value times v_scale (a power of two), exact in fp16 and in
    bf16 (E4M3 values have at most 4 significant bits): it must equal the oracle's
    decoding of the same code exactly."""
    D, bs = 128, 16
    wl = W.make_private("codes8", "fp8", [1, 1, 1, 1], 2 * G, 2, D, bs, seed=61, partition_size=0, q_dtype=q_dtype)
    assert np.log2(wl.v_scale) == np.round(np.log2(wl.v_scale))
    k, v = wl.k_cache.view(np.uint8), wl.v_cache.view(np.uint8)  # [NB, Hkv, D/16, bs, 16], [NB, Hkv, D, bs]
    expect = np.zeros((4, 2 * G, D))
    for s in range(4):
        blk = int(wl.block_tables[s][0])
        for h in range(2):
            codes = ((np.arange(D) + (2 * s + h) * D) % 256).astype(np.uint8)
            codes[(codes == 0x7F) | (codes == 0xFF)] = 0
            v[blk, h, :, 0] = codes
            k[blk, h, :, 0, :] = 0
            expect[s, h * G:(h + 1) * G, :] = oracle.widen(codes, "fp8") * wl.v_scale
    covered = {int(c) for s in range(4) for h in range(2) for c in v[int(wl.block_tables[s][0]), h, :, 0]}
    assert covered == set(range(256)) - {0x7F, 0xFF}
    out, _ = gpu_step(wl, write=False)
    want = torch.from_numpy(expect).to(out.dtype).cuda()
    # equal values (the code of -0 comes out as +0: the attention sum starts from +0)
    assert torch.equal(out.float(), want.float())


@pytest.mark.parametrize("q_dtype", ["f16", "bf16"])
@pytest.mark.parametrize("G", [1, 4])
def test_fp8_physical_permutation_is_bit_identical(q_dtype, G):
    wl = W.make_private("perm8", "fp8", [700, 33, 256, 1], 2 * G, 2, 128, 16, seed=36, partition_size=-1,
                        q_dtype=q_dtype)
    out1, _ = gpu_step(wl)
    pi = np.random.default_rng(10).permutation(wl.num_blocks)
    k2 = np.empty_like(wl.k_cache)
    v2 = np.empty_like(wl.v_cache)
    k2[pi] = wl.k_cache
    v2[pi] = wl.v_cache
    bt2 = np.where(wl.block_tables >= 0, pi[np.maximum(wl.block_tables, 0)], -1).astype(np.int32)
    wl2 = W.Workload(**{**wl.__dict__, "k_cache": k2, "v_cache": v2, "block_tables": bt2,
                        "slot_mapping": pi[wl.slot_mapping // 16] * 16 + wl.slot_mapping % 16})
    out2, _ = gpu_step(wl2)
    assert torch.equal(out1, out2)


def test_fp8_split_agrees_with_no_split():
    wl = W.make_private("split8", "fp8", [5000, 1200, 77], 16, 4, 128, 16, seed=37, partition_size=0,
                        q_dtype="bf16")
    out0, t = gpu_step(wl)
    for ps in (16, 256, -1):
        out1, _ = gpu_step(wl, partition_size=ps, t=t, write=False)
        d = (out0.double() - out1.double()).abs().max().item()
        assert d <= TOL["fp8"], (ps, d)


def test_pa_decode_refuses_an_fp8_cache():
    import paged_kv_cache_306_gb300 as pa
    wl = W.make_private("ref8", "fp8", [40], 8, 2, 128, 16, seed=38, q_dtype="f16")
    t = upload(wl)
    lib = pa.load()
    out = torch.empty_like(t["q"])
    st = lib.pa_decode(out.data_ptr(), t["q"].data_ptr(), t["k_cache"].data_ptr(), t["v_cache"].data_ptr(),
                       t["block_tables"].data_ptr(), t["block_tables"].shape[1], t["seq_lens"].data_ptr(), 1,
                       40, 8, 2, 128, 16, wl.num_blocks, 0.1, 0, None, 0, pa.PA_FP8_E4M3, None)
    assert st == pa.PA_ERR_UNSUPPORTED


# --- the layer workloads with an FP8 pool, at full size --------------------------------------------

@pytest.mark.parametrize("cfg,seqs", [(2, None), (3, None), (4, [0, 3]), (5, None)], ids=str)
def test_fp8_layer_workload_step(cfg, seqs):
    wl = W.config(cfg, kv_dtype="fp8")
    out, t = gpu_step(wl)
    k, v = oracle_pools(wl)
    assert np.array_equal(W.from_torch(t["k_cache"], "fp8"), k)
    assert np.array_equal(W.from_torch(t["v_cache"], "fp8"), v)
    idx = np.arange(wl.num_seqs) if seqs is None else np.asarray(seqs)
    ref = oracle_out(wl, k, v, idx)
    err, excess = max_violation(as_f64(out)[idx], ref, "fp8", with_rounding=False)
    assert excess <= 0.0, f"config {cfg} fp8: max abs err {err:.3e} > {TOL['fp8']}"


@pytest.mark.parametrize("G", [1, 4, 16])
def test_fp8_bf16_queries_far_from_unit_scale(G):
    """bf16 queries whose heads span many orders of magnitude (the FP8 path widens
    the cache to fp16 operands and rescales each query head by a power of two)."""
    wl = W.make_private("bigq8", "fp8", [1, 40, 300, 1029], 2 * G, 2, 128, 16, seed=39, partition_size=-1,
                        q_dtype="bf16")
    rng = np.random.default_rng(40)
    q = rng.standard_normal((wl.num_seqs, wl.num_heads, wl.head_size)).astype(np.float32)
    factors = np.float32(2.0) ** rng.choice([-20, -5, 0, 6, 12, 30], size=(wl.num_seqs, wl.num_heads, 1))
    q *= factors
    q[0, 0, :] = 0.0                                  # an all-zero head: uniform attention
    wl.q = W.cast(q, "bf16")
    out, _ = gpu_step(wl)
    k, v = oracle_pools(wl)
    assert_close(as_f64(out), oracle_out(wl, k, v), "fp8", with_rounding=True, out_dtype="bf16")
