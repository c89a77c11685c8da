"""Pins of the CPU oracle to facts outside itself (no GPU needed).

Each test ties the oracle to something the pages or the mathematics fix:
the pages' worked example, a brute-force restatement of the pages' online-softmax
walk, library routines (numpy/torch dtype conversion, numpy transposes for the
cache layout), closed forms and invariants the pages state.
"""
import json
import math
import os

import numpy as np
import pytest

import oracle
from oracle import brute

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def pools_from_logical(Kl, Vl, x):
    """Lay logical per-block rows [NB, Hkv, bs, D] out as the paged pools.

    Written with numpy reshapes from the layout statement ("Reading vLLM's
    PagedAttention kernel" §3.1: the key cache is viewed as
    [num_blocks, num_kv_heads, head_size // x, block_size, x], the value cache is
    [num_blocks, num_kv_heads, head_size, block_size]); independent of the
    oracle's own index arithmetic.
    """
    NB, Hkv, bs, D = Kl.shape
    k = np.ascontiguousarray(Kl.reshape(NB, Hkv, bs, D // x, x).transpose(0, 1, 3, 2, 4))
    v = np.ascontiguousarray(Vl.transpose(0, 1, 3, 2))
    return k, v


def logical_from_pools(k, v):
    NB, Hkv, Dx, bs, x = k.shape
    Kl = np.ascontiguousarray(k.transpose(0, 1, 3, 2, 4).reshape(NB, Hkv, bs, Dx * x))
    Vl = np.ascontiguousarray(v.transpose(0, 1, 3, 2))
    return Kl, Vl


def tiny_case(rng, S, H, Hkv, D, bs, NB, max_len):
    """Random fp64 logical pool, distinct random block ids per sequence."""
    Kl = rng.standard_normal((NB, Hkv, bs, D))
    Vl = rng.standard_normal((NB, Hkv, bs, D))
    L = rng.integers(1, max_len + 1, size=S).astype(np.int32)
    nblk = -(-L // bs)
    MB = int(nblk.max())
    perm = rng.permutation(NB)
    assert nblk.sum() <= NB
    bt = np.full((S, MB), -1, np.int32)
    c = 0
    for s in range(S):
        bt[s, :nblk[s]] = perm[c:c + nblk[s]]
        c += nblk[s]
    q = rng.standard_normal((S, H, D))
    return q, Kl, Vl, bt, L


def brute_force(q, Kl, Vl, bt, L, scale, G):
    S, H, D = q.shape
    bs = Kl.shape[2]
    out = np.zeros((S, H, D))
    for s in range(S):
        for h in range(H):
            kvh = h // G
            kb = {int(p): Kl[p, kvh].tolist() for p in bt[s] if p >= 0}
            vb = {int(p): Vl[p, kvh].tolist() for p in bt[s] if p >= 0}
            out[s, h] = brute.paged_decode_one(q[s, h].tolist(), [int(p) for p in bt[s] if p >= 0],
                                               kb, vb, int(L[s]), bs, scale)
    return out


# --- the pages' worked example ---------------------------------------------------------

def test_worked_example_matches_printed_output():
    ex = json.load(open(os.path.join(GOLDEN, "worked_example.json")))
    d, bs, L = ex["head_size"], ex["block_size"], ex["seq_len"]
    table = ex["block_table"]
    NB = max(table) + 1
    Kl = np.zeros((NB, 1, bs, d))
    Vl = np.zeros((NB, 1, bs, d))
    for i in range(L):
        Kl[table[i // bs], 0, i % bs] = ex["K"][i]
        Vl[table[i // bs], 0, i % bs] = ex["V"][i]
    k, v = pools_from_logical(Kl, Vl, oracle.pack_x("f64"))
    q = np.array([[ex["q"]]])
    out = oracle.decode(q, k, v, np.array([table], np.int32), np.array([L], np.int32),
                        1 / math.sqrt(d), "f64")
    assert np.round(out[0, 0], 6).tolist() == ex["expected_out_6dp"]
    # paged equals dense to the printed machine-epsilon level
    dense = brute.dense_decode_one(ex["q"], ex["K"], ex["V"], 1 / math.sqrt(d))
    assert np.max(np.abs(out[0, 0] - dense)) <= 4 * ex["expected_paged_vs_dense_max_abs_diff"]


# --- widening of stored values -------------------------------------------------------------

def test_fp16_widening_matches_numpy_on_every_bit_pattern():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ours = oracle.widen(bits.view(np.float16), "f16")
    ref = bits.view(np.float16).astype(np.float64)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan], ref[~nan])


def test_bf16_widening_matches_torch_on_every_bit_pattern():
    torch = pytest.importorskip("torch")
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ours = oracle.widen(bits, "bf16")
    ref = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan], ref[~nan])


def test_pack_x_is_16_bytes_over_element_size():
    # "x = 16 // element_size; FP16 -> x = 8" (Reading vLLM's PagedAttention kernel §3.1)
    assert oracle.pack_x("f16") == 8
    assert oracle.pack_x("bf16") == 8
    assert oracle.pack_x("f32") == 4
    assert oracle.pack_x("f64") == 2


# --- the oracle against an independent brute force ---------------------------------------

@pytest.mark.parametrize("D,bs,G", [(2, 1, 1), (4, 2, 2), (4, 4, 1), (8, 16, 3), (8, 4, 2)])
def test_oracle_matches_brute_force_online_softmax(D, bs, G):
    rng = np.random.default_rng(1000 + D * 31 + bs * 7 + G)
    Hkv = 2
    H = Hkv * G
    q, Kl, Vl, bt, L = tiny_case(rng, S=3, H=H, Hkv=Hkv, D=D, bs=bs, NB=64, max_len=min(40, 64 * bs // 3))
    scale = 1 / math.sqrt(D)
    k, v = pools_from_logical(Kl, Vl, oracle.pack_x("f64"))
    out = oracle.decode(q, k, v, bt, L, scale, "f64")
    ref = brute_force(q, Kl, Vl, bt, L, scale, G)
    assert np.max(np.abs(out - ref)) < 1e-12


def test_oracle_matches_brute_force_on_fp32_pool():
    rng = np.random.default_rng(7)
    q, Kl, Vl, bt, L = tiny_case(rng, S=2, H=4, Hkv=2, D=8, bs=4, NB=32, max_len=30)
    Kl, Vl, q = Kl.astype(np.float32), Vl.astype(np.float32), q.astype(np.float32)
    k, v = pools_from_logical(Kl, Vl, oracle.pack_x("f32"))
    out = oracle.decode(q, k, v, bt, L, 0.3, "f32")
    ref = brute_force(q.astype(np.float64), Kl.astype(np.float64), Vl.astype(np.float64), bt, L, 0.3, 2)
    assert np.max(np.abs(out - ref)) < 1e-12


# --- invariants the pages state -------------------------------------------------------------

def test_paged_equals_dense_on_the_original_arrays():
    """Paging is storage only: gather through the table == attention on contiguous rows."""
    rng = np.random.default_rng(11)
    D, bs, Lmax = 8, 4, 37
    Kd = rng.standard_normal((Lmax, D))
    Vd = rng.standard_normal((Lmax, D))
    q = rng.standard_normal(D)
    nblk = -(-Lmax // bs)
    table = rng.permutation(3 * nblk)[:nblk]
    NB = 3 * nblk
    Kl = np.full((NB, 1, bs, D), np.nan)
    Vl = np.full((NB, 1, bs, D), np.nan)
    for t in range(Lmax):
        Kl[table[t // bs], 0, t % bs] = Kd[t]
        Vl[table[t // bs], 0, t % bs] = Vd[t]
    k, v = pools_from_logical(Kl, Vl, 2)
    for L in (1, 2, bs - 1, bs, bs + 1, Lmax):
        out = oracle.decode(q[None, None], k, v, table[None].astype(np.int32), np.array([L], np.int32),
                            0.25, "f64")
        s = 0.25 * Kd[:L] @ q
        w = np.exp(s - s.max())
        ref = (w / w.sum()) @ Vd[:L]
        assert np.max(np.abs(out[0, 0] - ref)) < 1e-13


def test_physical_permutation_leaves_output_bit_identical():
    rng = np.random.default_rng(12)
    q, Kl, Vl, bt, L = tiny_case(rng, S=4, H=4, Hkv=2, D=8, bs=4, NB=80, max_len=60)
    k, v = pools_from_logical(Kl, Vl, 2)
    out = oracle.decode(q, k, v, bt, L, 0.35, "f64")
    pi = rng.permutation(80)                      # new id of old block b is pi[b]
    k2 = np.empty_like(k)
    v2 = np.empty_like(v)
    k2[pi] = k
    v2[pi] = v
    bt2 = np.where(bt >= 0, pi[np.maximum(bt, 0)], -1).astype(np.int32)
    out2 = oracle.decode(q, k2, v2, bt2, L, 0.35, "f64")
    assert np.array_equal(out, out2)


def test_softmax_weights_sum_to_one():
    rng = np.random.default_rng(13)
    q, Kl, Vl, bt, L = tiny_case(rng, S=3, H=2, Hkv=1, D=4, bs=4, NB=64, max_len=80)
    k, v = pools_from_logical(Kl, Vl, 2)
    _, w = oracle.decode(3 * q, k, v, bt, L, 0.5, "f64", return_weights=True)
    for s in range(3):
        for h in range(2):
            ws = w[s, h, :L[s]]
            assert np.all(ws > 0)
            assert abs(ws.sum() - 1.0) < 1e-14
            assert np.all(np.isnan(w[s, h, L[s]:]))


@pytest.mark.parametrize("dtype", ["f64", "f32", "f16", "bf16"])
def test_seq_len_one_returns_v0_exactly(dtype):
    rng = np.random.default_rng(14)
    D, bs, NB = 16, 4, 8
    st = {"f64": np.float64, "f32": np.float32, "f16": np.float16}
    x = oracle.pack_x(dtype)
    if dtype == "bf16":
        raw = (rng.standard_normal((NB, 1, bs, D)).astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
        Kl, Vl = raw, raw[::-1].copy()
        q = (rng.standard_normal((1, 1, D)).astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
    else:
        Kl = rng.standard_normal((NB, 1, bs, D)).astype(st[dtype])
        Vl = rng.standard_normal((NB, 1, bs, D)).astype(st[dtype])
        q = rng.standard_normal((1, 1, D)).astype(st[dtype])
    k, v = pools_from_logical(Kl, Vl, x)
    out = oracle.decode(q, k, v, np.array([[5]], np.int32), np.array([1], np.int32), 0.3, dtype)
    v0 = oracle.widen(np.ascontiguousarray(Vl[5, 0, 0]), dtype)
    assert np.array_equal(out[0, 0], v0)


def test_identical_keys_give_the_mean_of_values():
    rng = np.random.default_rng(15)
    D, bs, L = 8, 4, 23
    nblk = -(-L // bs)
    Kl = np.broadcast_to(rng.standard_normal(D), (nblk, 1, bs, D)).copy()
    Vl = rng.standard_normal((nblk, 1, bs, D))
    k, v = pools_from_logical(Kl, Vl, 2)
    table = np.arange(nblk, dtype=np.int32)[::-1].copy()
    out = oracle.decode(rng.standard_normal((1, 1, D)), k, v, table[None], np.array([L], np.int32),
                        0.7, "f64")
    rows = np.concatenate([Vl[table[j], 0] for j in range(nblk)])[:L]
    assert np.max(np.abs(out[0, 0] - rows.mean(axis=0))) < 1e-14


def test_partial_last_block_ignores_poisoned_slots():
    rng = np.random.default_rng(16)
    D, bs, NB = 8, 4, 16
    Kl = rng.standard_normal((NB, 2, bs, D))
    Vl = rng.standard_normal((NB, 2, bs, D))
    table = np.array([[9, 2, 7]], np.int32)
    for L in (9, 11):
        Kp, Vp = Kl.copy(), Vl.copy()
        Kp[7, :, L - 8:] = np.nan
        Vp[7, :, L - 8:] = np.nan
        q = rng.standard_normal((1, 4, D))
        a = oracle.decode(q, *pools_from_logical(Kl, Vl, 2), table, np.array([L], np.int32), 0.4, "f64")
        b = oracle.decode(q, *pools_from_logical(Kp, Vp, 2), table, np.array([L], np.int32), 0.4, "f64")
        assert np.all(np.isfinite(b))
        assert np.array_equal(a, b)


def test_scale_multiplies_the_scores():
    rng = np.random.default_rng(17)
    q, Kl, Vl, bt, L = tiny_case(rng, S=2, H=2, Hkv=2, D=4, bs=2, NB=40, max_len=30)
    k, v = pools_from_logical(Kl, Vl, 2)
    a = oracle.decode(q, k, v, bt, L, 0.5, "f64")
    b = oracle.decode(0.5 * q, k, v, bt, L, 1.0, "f64")
    c = oracle.decode(q, k, v, bt, L, 1.0, "f64")
    assert np.max(np.abs(a - b)) < 1e-14
    assert np.max(np.abs(a - c)) > 1e-3


def test_gqa_query_heads_share_consecutive_kv_heads():
    """Reading adopted for the unstated GQA mapping: query head h reads kv head h // G."""
    rng = np.random.default_rng(18)
    q, Kl, Vl, bt, L = tiny_case(rng, S=2, H=6, Hkv=2, D=4, bs=4, NB=40, max_len=30)
    k, v = pools_from_logical(Kl, Vl, 2)
    out = oracle.decode(q, k, v, bt, L, 0.5, "f64")
    for h in range(6):
        kv = h // 3
        single = oracle.decode(np.ascontiguousarray(q[:, h:h + 1]), np.ascontiguousarray(k[:, kv:kv + 1]),
                               np.ascontiguousarray(v[:, kv:kv + 1]), bt, L, 0.5, "f64")
        assert np.array_equal(out[:, h], single[:, 0])


def test_decode_rejects_out_of_pool_block_ids_and_bad_lengths():
    rng = np.random.default_rng(19)
    q, Kl, Vl, bt, L = tiny_case(rng, S=1, H=1, Hkv=1, D=4, bs=4, NB=8, max_len=8)
    k, v = pools_from_logical(Kl, Vl, 2)
    bad = bt.copy()
    bad[0, 0] = 8
    with pytest.raises(oracle.OracleError):
        oracle.decode(q, k, v, bad, L, 1.0, "f64")
    with pytest.raises(oracle.OracleError):
        oracle.decode(q, k, v, bt, np.array([0], np.int32), 1.0, "f64")
    with pytest.raises(oracle.OracleError):
        oracle.decode(q, k, v, bt, np.array([bt.shape[1] * 4 + 1], np.int32), 1.0, "f64")


# --- write path -------------------------------------------------------------------------------

@pytest.mark.parametrize("dtype", ["f32", "f16", "f64"])
def test_slot_mapping_round_trip(dtype):
    """Writes scatter through slot = block*block_size + offset; reading back through the
    same placement returns the rows bit for bit, and no other slot changes."""
    rng = np.random.default_rng(20)
    st = {"f64": np.float64, "f32": np.float32, "f16": np.float16}[dtype]
    NB, Hkv, D, bs, T = 12, 3, 16, 4, 17
    x = oracle.pack_x(dtype)
    k = rng.standard_normal((NB, Hkv, D // x, bs, x)).astype(st)
    v = rng.standard_normal((NB, Hkv, D, bs)).astype(st)
    k0, v0 = k.copy(), v.copy()
    key = rng.standard_normal((T, Hkv, D)).astype(st)
    val = rng.standard_normal((T, Hkv, D)).astype(st)
    slots = rng.permutation(NB * bs)[:T].astype(np.int64)
    slots[3] = slots[T - 1] = -1                        # padding tokens are skipped (one after every real one)
    oracle.reshape_and_cache(key, val, k, v, slots, dtype)
    Kl, Vl = logical_from_pools(k, v)
    K0, V0 = logical_from_pools(k0, v0)
    touched = np.zeros((NB, bs), bool)
    for t in range(T):
        if slots[t] < 0:
            continue
        b, o = divmod(int(slots[t]), bs)
        touched[b, o] = True
        assert np.array_equal(Kl[b, :, o].view(np.uint8), key[t].view(np.uint8))
        assert np.array_equal(Vl[b, :, o].view(np.uint8), val[t].view(np.uint8))
    for b in range(NB):
        for o in range(bs):
            if not touched[b, o]:
                assert np.array_equal(Kl[b, :, o].view(np.uint8), K0[b, :, o].view(np.uint8))
                assert np.array_equal(Vl[b, :, o].view(np.uint8), V0[b, :, o].view(np.uint8))


def test_reshape_rejects_duplicate_and_out_of_pool_slots():
    k = np.zeros((2, 1, 1, 4, 4), np.float32)
    v = np.zeros((2, 1, 4, 4), np.float32)
    key = np.ones((2, 1, 4), np.float32)
    with pytest.raises(oracle.OracleError):
        oracle.reshape_and_cache(key, key, k, v, np.array([3, 3]), "f32")
    with pytest.raises(oracle.OracleError):
        oracle.reshape_and_cache(key, key, k, v, np.array([1, 8]), "f32")


def test_copy_on_write_block_copy():
    """A shared block is copied before it is written; the source is untouched and a
    later write into the copy leaves the source's readers unchanged."""
    rng = np.random.default_rng(21)
    NB, Hkv, D, bs = 6, 2, 8, 4
    k = rng.standard_normal((NB, Hkv, D // 4, bs, 4)).astype(np.float32)
    v = rng.standard_normal((NB, Hkv, D, bs)).astype(np.float32)
    k0, v0 = k.copy(), v.copy()
    oracle.copy_blocks(k, v, np.array([[1, 4], [2, 0]]), "f32")
    assert np.array_equal(k[4], k0[1]) and np.array_equal(v[4], v0[1])
    assert np.array_equal(k[0], k0[2]) and np.array_equal(v[0], v0[2])
    for b in (1, 2, 3, 5):
        assert np.array_equal(k[b], k0[b]) and np.array_equal(v[b], v0[b])
    key = np.full((1, Hkv, D), 7.0, np.float32)
    oracle.reshape_and_cache(key, key, k, v, np.array([4 * bs + 2]), "f32")
    assert np.array_equal(k[1], k0[1]) and np.array_equal(v[1], v0[1])
    assert not np.array_equal(k[4], k0[1])


def test_kv_bytes_of_llama7b_layer_times_layers_matches_memory_formula():
    """M = 2 * L * d_model * S * B * 2 bytes for fp16 (KV Cache and PagedAttention memory
    management, memory model): LLaMA-7B, L=32, d=4096, S=2048, B=16 -> 17,179,869,184 B.
    One layer of it is the 16-sequence, 32-head, head-size-128, 2048-token fp16 workload."""
    seqs, heads, D, L, e = 16, 32, 128, 2048, 2
    per_layer = 2 * seqs * L * heads * D * e
    assert per_layer * 32 == 4 * 32 * 4096 * 2048 * 16 == 17_179_869_184


# --- FP8 E4M3 cache (kv_cache_dtype, k_scale, v_scale of the write path) ----------------------

def test_e4m3_decoding_matches_torch_on_every_code():
    torch = pytest.importorskip("torch")
    codes = np.arange(256, dtype=np.uint8)
    ours = oracle.widen(codes, "fp8")
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    nan = np.isnan(ref)
    assert nan.sum() == 2 and np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan], ref[~nan])


def test_e4m3_encoding_matches_torch_within_range():
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(30)
    x = np.concatenate([rng.uniform(-464, 464, 20000), rng.standard_normal(20000) * 3,
                        rng.standard_normal(20000) * 2.0 ** -7, [0.0, -0.0, 448.0, -448.0, 464.0, 2.0 ** -10,
                                                                  1.5 * 2.0 ** -9, 2.5 * 2.0 ** -9]])
    x = x.astype(np.float32).astype(np.float64)
    ours = oracle.encode_e4m3(x)
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(ours, ref)


def test_e4m3_clamps_instead_of_overflowing():
    assert oracle.encode_e4m3(np.array([1000.0, 480.0, -1e6])).tolist() == [0x7E, 0x7E, 0xFE]


def test_e4m3_codes_round_trip():
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], dtype=np.uint8)
    assert np.array_equal(oracle.encode_e4m3(oracle.widen(codes, "fp8")), codes)


def _fp8_pool(rng, NB, Hkv, D, bs, gen_scale):
    """Random E4M3 pools drawn with torch's float8 conversion, logical [NB, Hkv, bs, D]."""
    torch = pytest.importorskip("torch")
    def draw():
        x = rng.standard_normal((NB, Hkv, bs, D)).astype(np.float32) / np.float32(gen_scale)
        return torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    return draw(), draw()


def test_quantised_decode_equals_decode_of_the_dequantised_pool():
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(31)
    NB, Hkv, D, bs = 24, 2, 32, 4
    kc8, vc8 = _fp8_pool(rng, NB, Hkv, D, bs, 1 / 32)
    ks, vs = 0.03, 0.05
    k8, v8 = pools_from_logical(kc8, vc8, 16)
    deq = lambda a, s: torch.from_numpy(a).view(torch.float8_e4m3fn).to(torch.float64).numpy() * s
    k64, v64 = pools_from_logical(deq(kc8, ks), deq(vc8, vs), 2)
    q = rng.standard_normal((3, 4, D)).astype(np.float16)
    bt = rng.permutation(NB)[:18].reshape(3, 6).astype(np.int32)
    L = np.array([1, 13, 24], np.int32)
    got = oracle.decode(q, k8, v8, bt, L, 0.2, "fp8", q_dtype="f16", k_scale=ks, v_scale=vs)
    ref = oracle.decode(q.astype(np.float64), k64, v64, bt, L, 0.2, "f64")
    assert np.max(np.abs(got - ref)) < 1e-13


def test_quantised_write_stores_torch_rounded_codes_of_x_over_scale():
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(32)
    NB, Hkv, D, bs, T = 10, 2, 32, 4, 9
    k = np.zeros((NB, Hkv, D // 16, bs, 16), np.uint8)
    v = np.zeros((NB, Hkv, D, bs), np.uint8)
    # |x| / scale stays inside +-448 here, where torch's conversion does not saturate
    key = rng.standard_normal((T, Hkv, D)).astype(np.float16)
    val = rng.standard_normal((T, Hkv, D)).astype(np.float16)
    slots = rng.permutation(NB * bs)[:T].astype(np.int64)
    ks, vs = 0.0125, 0.02
    oracle.reshape_and_cache_scaled(key, val, k, v, slots, "f16", "fp8", ks, vs)
    Kl, Vl = logical_from_pools(k, v)
    q8 = lambda a, s: torch.from_numpy(a.astype(np.float32) / np.float32(s)).to(torch.float8_e4m3fn) \
        .view(torch.uint8).numpy()
    for t in range(T):
        b, o = divmod(int(slots[t]), bs)
        assert np.array_equal(Kl[b, :, o], q8(key[t], ks))
        assert np.array_equal(Vl[b, :, o], q8(val[t], vs))


def test_value_scale_scales_the_output_and_key_scale_acts_like_query_scale():
    rng = np.random.default_rng(33)
    NB, Hkv, D, bs = 16, 1, 16, 4
    kc8, vc8 = _fp8_pool(rng, NB, Hkv, D, bs, 1 / 16)
    k8, v8 = pools_from_logical(kc8, vc8, 16)
    q = rng.standard_normal((2, 2, D)).astype(np.float32)
    bt = np.arange(16, dtype=np.int32).reshape(2, 8)
    L = np.array([30, 7], np.int32)
    a = oracle.decode(q, k8, v8, bt, L, 0.25, "fp8", q_dtype="f32", k_scale=0.1, v_scale=0.5)
    b = oracle.decode(q, k8, v8, bt, L, 0.25, "fp8", q_dtype="f32", k_scale=0.1, v_scale=1.0)
    c = oracle.decode(q, k8, v8, bt, L, 0.025, "fp8", q_dtype="f32", k_scale=1.0, v_scale=0.5)
    assert np.max(np.abs(a - 0.5 * b)) < 1e-14
    assert np.max(np.abs(a - c)) < 1e-12


# --- chunked prefill (the step before decode) ---------------------------------------------------

def prefill_case(rng, S, H, Hkv, D, bs, NB, max_len):
    """A tiny paged pool and, per sequence, a chunk of n_s <= L_s new query tokens."""
    q1, Kl, Vl, bt, L = tiny_case(rng, S, H, Hkv, D, bs, NB, max_len)
    n = np.array([rng.integers(0, l + 1) for l in L], np.int32)
    n[0] = L[0]                                     # one pure prefill (no cached history)
    qsl = np.concatenate([[0], np.cumsum(n)]).astype(np.int32)
    q = rng.standard_normal((int(qsl[-1]), H, D))
    return q, Kl, Vl, bt, L, qsl


@pytest.mark.parametrize("D,bs,G", [(4, 1, 1), (8, 4, 2), (4, 16, 3), (16, 2, 1)])
def test_prefill_matches_brute_force_walk_up_to_each_position(D, bs, G):
    """Row i of sequence s equals the pages' per-token walk over the first p + 1
    tokens, p = L_s - n_s + i (the causal reading of a chunk after its history)."""
    rng = np.random.default_rng(70 + D + bs + G)
    Hkv = 2
    q, Kl, Vl, bt, L, qsl = prefill_case(rng, 4, Hkv * G, Hkv, D, bs, 64, 24)
    k, v = pools_from_logical(Kl, Vl, 2)
    got = oracle.prefill(q, k, v, bt, L, qsl, 0.37, "f64")
    for s in range(len(L)):
        n = qsl[s + 1] - qsl[s]
        for i in range(n):
            p = L[s] - n + i
            for h in range(Hkv * G):
                kvh = h // G
                kb = {int(b): Kl[b, kvh].tolist() for b in bt[s] if b >= 0}
                vb = {int(b): Vl[b, kvh].tolist() for b in bt[s] if b >= 0}
                ref = brute.paged_decode_one(q[qsl[s] + i, h].tolist(), [int(b) for b in bt[s] if b >= 0], kb, vb,
                                             int(p + 1), bs, 0.37)
                assert np.max(np.abs(got[qsl[s] + i, h] - ref)) < 1e-12


def test_prefill_of_one_token_per_sequence_is_decode():
    rng = np.random.default_rng(74)
    q, Kl, Vl, bt, L = tiny_case(rng, 5, 6, 3, 8, 4, 64, 30)
    k, v = pools_from_logical(Kl, Vl, 2)
    qsl = np.arange(6, dtype=np.int32)
    got = oracle.prefill(q, k, v, bt, L, qsl, 0.3, "f64")
    assert np.max(np.abs(got - oracle.decode(q, k, v, bt, L, 0.3, "f64"))) < 1e-13


def test_a_chunk_gives_the_rows_of_the_whole_prompt():
    """Prefill of tokens a..L-1 after a cached history of a tokens gives exactly the
    rows a..L-1 of the prefill of the whole prompt."""
    rng = np.random.default_rng(75)
    q, Kl, Vl, bt, L = tiny_case(rng, 1, 4, 2, 8, 4, 32, 30)
    L = np.array([29], np.int32)
    bt = rng.permutation(32)[:8].reshape(1, 8).astype(np.int32)
    k, v = pools_from_logical(Kl, Vl, 2)
    qa = rng.standard_normal((29, 4, 8))
    full = oracle.prefill(qa, k, v, bt, L, np.array([0, 29], np.int32), 0.5, "f64")
    for a in (0, 1, 7, 16, 28):
        part = oracle.prefill(qa[a:], k, v, bt, L, np.array([0, 29 - a], np.int32), 0.5, "f64")
        assert np.array_equal(part, full[a:])


def test_prefill_rejects_a_chunk_longer_than_its_sequence():
    rng = np.random.default_rng(76)
    q, Kl, Vl, bt, L = tiny_case(rng, 2, 2, 2, 8, 4, 32, 10)
    k, v = pools_from_logical(Kl, Vl, 2)
    qsl = np.array([0, int(L[0]) + 1, int(L[0]) + 2], np.int32)
    with pytest.raises(Exception):
        oracle.prefill(np.zeros((int(qsl[-1]), 2, 8)), k, v, bt, L, qsl, 0.5, "f64")
