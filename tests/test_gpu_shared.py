"""Decode over sequences that share prefix blocks (pa_decode_shared), on the GPU
through the C ABI.

Sequences of one group hold the first prefix_blocks[s] blocks of a common prefix
("vLLM's PagedAttention: why the KV cache is paged", §4.2: forked sequences map
their first logical blocks to the same physical blocks).  pa_decode_shared reads
those blocks once per cluster of sequences, with the query heads of all members
in one tensor-core tile, and merges them with each member's own blocks.  The
result must be the plain attention of each sequence on its own: within the
decode tolerance of the oracle, with the pools written byte for byte as the
separate write path writes them.
"""
import zlib

import numpy as np
import pytest

import workloads as W
from helpers import TOL, as_f64, assert_close, max_violation, oracle_out, oracle_pools, same_bytes, upload

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

SHARED = 6  # PA_DEVERR_SHARED


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import paged_kv_cache_306_gb300 as pa
    pa.load()


def shared_call(wl, t=None, fused=True, partition_size=None, groups=None):
    """pa_decode_shared on a workload (the fused step, or decode alone after the write path)."""
    import paged_kv_cache_306_gb300 as pa
    t = upload(wl) if t is None else t
    grp, blk = W.prefix_groups(wl.block_tables, wl.seq_lens, wl.block_size) if groups is None else groups
    g, b = torch.from_numpy(np.ascontiguousarray(grp)).cuda(), torch.from_numpy(np.ascontiguousarray(blk)).cuda()
    ps = wl.partition_size if partition_size is None else partition_size
    out = torch.empty_like(t["q"])
    if not fused:
        if len(wl.cow):
            pa.pa_copy_blocks(t["k_cache"], t["v_cache"], t["cow"])
        if wl.dtype == "fp8":
            pa.pa_reshape_and_cache_scaled(t["key"], t["value"], t["k_cache"], t["v_cache"], t["slot_mapping"],
                                           wl.k_scale, wl.v_scale)
        else:
            pa.pa_reshape_and_cache(t["key"], t["value"], t["k_cache"], t["v_cache"], t["slot_mapping"])
    pa.pa_decode_shared(out, t["q"], t["key"] if fused else None, t["value"] if fused else None, t["k_cache"],
                        t["v_cache"], t["cow"] if (fused and len(wl.cow)) else None, t["block_tables"],
                        t["seq_lens"], g, b, wl.scale, wl.max_seq_len, wl.k_scale, wl.v_scale, ps)
    return out, t


def check(wl, fused=True, partition_size=None, seqs=None):
    import paged_kv_cache_306_gb300 as pa
    out, t = shared_call(wl, fused=fused, partition_size=partition_size)
    code = pa.pa_get_device_error()
    assert code == 0, f"device error {code}: {pa.DEVICE_ERRORS.get(code)}"
    k, v = oracle_pools(wl)
    assert np.array_equal(W.from_torch(t["k_cache"], wl.dtype).view(np.uint8), k.view(np.uint8))
    assert np.array_equal(W.from_torch(t["v_cache"], wl.dtype).view(np.uint8), v.view(np.uint8))
    idx = np.arange(wl.num_seqs) if seqs is None else np.asarray(seqs)
    got = as_f64(out)[idx]
    assert np.all(np.isfinite(got))
    assert_close(got, oracle_out(wl, k, v, idx), wl.dtype, with_rounding=True, what=wl.name,
                 out_dtype=wl.q_dtype)
    return out, t


def sharing_groups(dtype, bs, G, D, seed, num_groups=4, group_size=8, partition_size=-1, q_dtype=None):
    return W.make_prefix_shared(f"shared-{dtype}-G{G}", dtype, num_groups, group_size, 2 * G, 2, D, bs, seed=seed,
                                len_range=(8, 1500), prefix_range=(64, 700), partition_size=partition_size,
                                q_dtype=q_dtype)


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("bs", [16, 32])
@pytest.mark.parametrize("G", [1, 2, 4, 7, 8])
@pytest.mark.parametrize("fused", [True, False])
def test_shared_prefix_decode_matches_the_oracle(dtype, D, bs, G, fused):
    seed = zlib.crc32(repr(("shared", dtype, D, bs, G, fused)).encode())
    wl = sharing_groups(dtype, bs, G, D, seed)
    grp, blk = W.prefix_groups(wl.block_tables, wl.seq_lens, bs)
    assert (blk >= 2).sum() >= 6, "the case must share blocks"
    check(wl, fused=fused)


@pytest.mark.parametrize("part", [0, 16, 64, 256])
def test_caller_partitions_inside_shared_segments(part):
    """Partition boundaries fold running states whose columns may have seen no block."""
    wl = sharing_groups("f16", 16, 4, 128, seed=77 + part, partition_size=part)
    check(wl)


@pytest.mark.parametrize("q_dtype", ["f16", "bf16"])
@pytest.mark.parametrize("fused", [True, False])
def test_shared_prefix_decode_over_an_fp8_pool(q_dtype, fused):
    wl = sharing_groups("fp8", 16, 4, 128, seed=91 if fused else 92, q_dtype=q_dtype)
    check(wl, fused=fused)


@pytest.mark.parametrize("G,dtype", [(16, "f16"), (1, "f32"), (4, "f32")])
def test_shapes_without_clusters_run_the_plain_schedule(G, dtype):
    wl = sharing_groups(dtype, 16, G, 64, seed=5 + G)
    check(wl)


def test_short_leaders_and_members_that_share_nothing():
    """Clusters whose first sequence holds no shared block, members with 0 shared
    blocks, a group of one, and groups in any order of lengths."""
    wl = W.make_prefix_shared("short-leaders", "bf16", 6, 8, 8, 2, 128, 16, seed=123, len_range=(2, 3000),
                              prefix_range=(40, 600))
    grp, blk = W.prefix_groups(wl.block_tables, wl.seq_lens, 16)
    assert (blk == 0).any() and (blk > 8).any()
    check(wl)
    # every sequence its own group: the plain schedule's result
    check_groups = (np.arange(wl.num_seqs, dtype=np.int32), np.zeros(wl.num_seqs, np.int32))
    import paged_kv_cache_306_gb300 as pa
    out, _ = shared_call(wl, groups=check_groups)
    assert pa.pa_get_device_error() == 0
    k, v = oracle_pools(wl)
    assert_close(as_f64(out), oracle_out(wl, k, v), "bf16", with_rounding=True)


def test_bit_identical_under_a_physical_permutation():
    """The result depends on the logical order of the blocks only."""
    import paged_kv_cache_306_gb300 as pa
    wl = sharing_groups("f16", 16, 4, 128, seed=300)
    out1, _ = shared_call(wl)
    perm = np.random.default_rng(1).permutation(wl.num_blocks)
    wl2 = W.subset(wl, np.arange(wl.num_seqs))
    k2 = np.empty_like(wl.k_cache)
    v2 = np.empty_like(wl.v_cache)
    k2[perm] = wl.k_cache
    v2[perm] = wl.v_cache
    wl2.k_cache, wl2.v_cache = k2, v2
    bt = wl.block_tables.copy()
    bt[bt >= 0] = perm[bt[bt >= 0]]
    wl2.block_tables = bt
    wl2.cow = np.ascontiguousarray(perm[wl.cow]) if len(wl.cow) else wl.cow
    wl2.slot_mapping = perm[wl.slot_mapping // 16] * 16 + wl.slot_mapping % 16
    out2, _ = shared_call(wl2)
    assert pa.pa_get_device_error() == 0
    assert same_bytes(out1, out2)


def test_a_false_sharing_claim_is_reported():
    import paged_kv_cache_306_gb300 as pa
    wl = W.make_private("no-sharing", "f16", [300, 400, 500, 600], 8, 2, 128, 16, seed=9, poison=False)
    grp = np.zeros(4, np.int32)                     # one group ...
    blk = np.full(4, 10, np.int32)                  # ... claiming 10 common blocks that differ
    shared_call(wl, groups=(grp, blk))
    assert pa.pa_get_device_error() == SHARED
    assert pa.pa_get_device_error() == 0


def test_groups_across_the_launch_boundary():
    """More than 1024 sequences: a group cut by the launch boundary becomes two."""
    wl = W.make_prefix_shared("many", "f16", 138, 8, 8, 2, 64, 16, seed=44, len_range=(4, 200),
                              prefix_range=(16, 120))
    assert wl.num_seqs > 1024
    check(wl, seqs=np.r_[0:40, 1000:1060, wl.num_seqs - 40:wl.num_seqs])


@pytest.mark.parametrize("bs", [16, 32])
def test_full_size_mixed_batch(bs):
    """The prefix-sharing workload at full size in the launch configuration the
    benchmark times: pools bytewise, every sequence against the oracle."""
    wl = W.config(5, block_size=bs)
    check(wl)


def test_full_size_mixed_batch_over_an_fp8_pool():
    wl = W.config(5, block_size=16, kv_dtype="fp8")
    check(wl, seqs=np.arange(0, wl.num_seqs, 3))


def test_workspace_size_and_a_short_workspace_is_refused():
    import ctypes
    import paged_kv_cache_306_gb300 as pa
    lib = pa.load()
    need = lib.pa_decode_shared_workspace_size(256, 32, 8, 128, 8192, 16, 0, pa.PA_F16)
    plain = lib.pa_decode_workspace_size(256, 32, 8, 128, 8192, 16, 0, pa.PA_F16)
    assert need > plain > 0
    wl = sharing_groups("f16", 16, 4, 128, seed=8)
    t = upload(wl)
    grp, blk = W.prefix_groups(wl.block_tables, wl.seq_lens, 16)
    g, b = torch.from_numpy(grp).cuda(), torch.from_numpy(blk).cuda()
    out = torch.empty_like(t["q"])
    small = torch.empty(256, dtype=torch.uint8, device="cuda")
    P = ctypes.c_void_p
    n0 = lib.pa_launch_count()
    st = lib.pa_decode_shared(P(out.data_ptr()), P(t["q"].data_ptr()), None, None, P(t["k_cache"].data_ptr()),
                              P(t["v_cache"].data_ptr()), None, 0, P(t["block_tables"].data_ptr()),
                              wl.max_blocks_per_seq, P(t["seq_lens"].data_ptr()), P(g.data_ptr()), P(b.data_ptr()),
                              wl.num_seqs, wl.max_seq_len, wl.num_heads, wl.num_kv_heads, wl.head_size,
                              wl.block_size, wl.num_blocks, ctypes.c_float(wl.scale), 0, P(small.data_ptr()), 256,
                              pa.PA_F16, pa.PA_F16, ctypes.c_float(1.0), ctypes.c_float(1.0), None)
    assert st == pa.PA_ERR_WORKSPACE
    assert lib.pa_launch_count() == n0


def test_shared_workspace_covers_the_clusters():
    import paged_kv_cache_306_gb300 as pa
    lib = pa.load()
    # clusters double the segments and widen every partial slot to 16 rows
    for G in (1, 2, 4, 8):
        assert lib.pa_decode_shared_workspace_size(64, 2 * G, 2, 128, 4096, 16, 0, pa.PA_F16) > \
            lib.pa_decode_workspace_size(64, 2 * G, 2, 128, 4096, 16, 0, pa.PA_F16)
    # no clusters for fp32 or more than 8 query heads per kv head: the plain layout
    assert lib.pa_decode_shared_workspace_size(64, 32, 2, 128, 4096, 16, 0, pa.PA_F16) == \
        lib.pa_decode_workspace_size(64, 32, 2, 128, 4096, 16, 0, pa.PA_F16)
    assert lib.pa_decode_shared_workspace_size(64, 8, 2, 128, 4096, 16, 0, pa.PA_F32) == \
        lib.pa_decode_workspace_size(64, 8, 2, 128, 4096, 16, 0, pa.PA_F32)
