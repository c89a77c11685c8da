"""Host-side checks of the seeded input generator (no GPU)."""
import numpy as np
import pytest

import oracle
import workloads as W


def valid_mask_k(wl):
    """Boolean [NB, bs]: slot holds a token some sequence reads (before the step's write)."""
    m = np.zeros((wl.num_blocks, wl.block_size), bool)
    bs = wl.block_size
    for s in range(wl.num_seqs):
        L = int(wl.seq_lens[s])
        for j in range(-(-L // bs)):
            phys = int(wl.block_tables[s, j])
            n = min(bs, L - j * bs)
            m[phys, :n] = True
    return m


def test_tiny_config_shapes_and_poison():
    wl = W.config(1)
    assert wl.dtype == "f32" and wl.k_cache.shape == (128, 8, 16, 16, 4)
    assert wl.v_cache.shape == (128, 8, 64, 16)
    assert np.all((wl.seq_lens >= 1) & (wl.seq_lens <= 256))
    m = valid_mask_k(wl)
    # new-token slots are poisoned until the step writes them
    for s in range(wl.num_seqs):
        b, o = divmod(int(wl.slot_mapping[s]), wl.block_size)
        assert b == wl.block_tables[s, (wl.seq_lens[s] - 1) // wl.block_size]
        m[b, o] = False
    for b in range(wl.num_blocks):
        for o in range(wl.block_size):
            fin = np.isfinite(wl.v_cache[b, :, :, o]).all() and np.isfinite(wl.k_cache[b, :, :, o]).all()
            assert fin == m[b, o]


def test_seeded_generation_is_deterministic():
    a, b = W.config(1), W.config(1)
    assert np.array_equal(a.block_tables, b.block_tables)
    assert np.array_equal(a.k_cache, b.k_cache, equal_nan=True)
    assert np.array_equal(a.q, b.q)


def test_block_ids_distinct_for_private_sequences():
    wl = W.make_private("t", "f16", [33, 16, 1, 70], 4, 2, 64, 16, seed=3)
    ids = np.concatenate([wl.block_tables[s, :-(-int(L) // 16)] for s, L in enumerate(wl.seq_lens)])
    assert len(set(ids.tolist())) == len(ids)
    assert len(set(wl.slot_mapping.tolist())) == wl.num_seqs


@pytest.mark.parametrize("bs", [16, 32])
def test_prefix_sharing_refcounts_and_copy_on_write(bs):
    wl = W.make_prefix_shared("t", "f16", num_groups=4, group_size=8, num_heads=8, num_kv_heads=2,
                              head_size=64, block_size=bs, seed=5, len_range=(16, 600),
                              prefix_range=(40, 300))
    refs = {}
    for s in range(wl.num_seqs):
        for j in range(-(-int(wl.seq_lens[s]) // bs)):
            refs.setdefault(int(wl.block_tables[s, j]), []).append(s)
    assert any(len(v) > 1 for v in refs.values()), "no block is shared"
    dsts = set()
    for src, dst in wl.cow.tolist():
        assert src != dst and dst not in dsts
        dsts.add(dst)
        # the destination is referenced by exactly one sequence, and only at its new token
        (s,) = refs[dst]
        j = (int(wl.seq_lens[s]) - 1) // bs
        assert wl.block_tables[s, j] == dst
        assert int(wl.slot_mapping[s]) // bs == dst
        # the source is still read by a sibling
        assert len(refs.get(src, [])) >= 1
        assert np.isnan(wl.v_cache[dst].astype(np.float32)).all()
    # every write slot is distinct and lies in a block with a single reader
    assert len(set(wl.slot_mapping.tolist())) == wl.num_seqs
    for s in range(wl.num_seqs):
        b = int(wl.slot_mapping[s]) // bs
        assert refs[b] == [s]


def test_oracle_runs_one_full_step_on_a_prefix_shared_batch():
    wl = W.make_prefix_shared("t", "f16", num_groups=2, group_size=4, num_heads=4, num_kv_heads=2,
                              head_size=64, block_size=16, seed=6, len_range=(16, 200),
                              prefix_range=(20, 100))
    k, v = wl.clone_pools()
    oracle.copy_blocks(k, v, wl.cow, "f16")
    oracle.reshape_and_cache(wl.key, wl.value, k, v, wl.slot_mapping, "f16")
    out = oracle.decode(wl.q, k, v, wl.block_tables, wl.seq_lens, wl.scale, "f16")
    assert np.all(np.isfinite(out))
    # before the write the new-token slots are poisoned: the output would not be finite
    k2, v2 = wl.clone_pools()
    oracle.copy_blocks(k2, v2, wl.cow, "f16")
    bad = oracle.decode(wl.q, k2, v2, wl.block_tables, wl.seq_lens, wl.scale, "f16")
    assert not np.all(np.isfinite(bad))


def test_bf16_cast_rounds_to_nearest_even():
    torch = pytest.importorskip("torch")
    x = np.random.default_rng(0).standard_normal(10000).astype(np.float32)
    ours = W.cast(x, "bf16")
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, ref)


def test_full_size_shapes_of_the_layer_workloads():
    wl = W.config(3, poison=False)
    assert wl.num_blocks == 2048 and wl.block_tables.shape == (16, 128)
    assert sorted(wl.block_tables.ravel().tolist()) == list(range(2048))
    kv_bytes = wl.total_tokens * wl.num_kv_heads * wl.head_size * 2 * 2
    assert kv_bytes == 536_870_912


def test_fp8_workload_holds_codes_of_scaled_normal_values():
    wl = W.make_private("f8", "fp8", [40, 17, 1], 8, 2, 128, 16, seed=7, q_dtype="bf16")
    assert wl.k_cache.dtype == np.uint8 and wl.k_cache.shape == (wl.num_blocks, 2, 8, 16, 16)
    assert wl.q_dtype == "bf16" and wl.q.dtype == np.uint16 and wl.key.dtype == np.uint16
    assert wl.k_scale == wl.v_scale == W.FP8_SCALE
    m = valid_mask_k(wl)
    for s in range(wl.num_seqs):                                 # new-token slots stay poisoned until the write
        b, o = divmod(int(wl.slot_mapping[s]), wl.block_size)
        m[b, o] = False
    vals = oracle.widen(wl.v_cache, "fp8") * wl.v_scale          # [NB, Hkv, D, bs]
    live = vals.transpose(0, 3, 1, 2)[m]                         # tokens some sequence reads
    assert np.all(np.isfinite(live))
    assert 0.9 < live.std() < 1.1 and abs(live.mean()) < 0.05
    # unused slots carry the NaN code
    dead = wl.v_cache.transpose(0, 3, 1, 2)[~m]
    assert np.all(dead == W.FP8_NAN)


def test_fp8_config_keeps_the_shapes_of_its_16_bit_workload():
    a, b = W.config(3), W.config(3, kv_dtype="fp8")
    assert b.k_cache.shape[:2] == a.k_cache.shape[:2] and b.k_cache.shape[-1] == 16
    assert b.q_dtype == a.dtype and np.array_equal(a.seq_lens, b.seq_lens)
    assert np.array_equal(a.block_tables, b.block_tables)
    with pytest.raises(ValueError):
        W.config(1, kv_dtype="fp8")


@pytest.mark.parametrize("bs,seed", [(16, 1), (16, 20), (32, 8), (32, 9)])
def test_no_poison_reaches_a_read_slot_when_sharers_of_a_block_differ_in_length(bs, seed):
    """Short prefixes make sequences of one group end inside the same shared block
    with different lengths; the last sharer then writes in place into the block
    the others copy.  Before the step that slot holds a prefix token, which the
    copies carry; no poison may be read by any sequence after the step."""
    wl = W.make_prefix_shared("short", "f32", 4, 5, 4, 2, 64, bs, seed=seed, len_range=(4, 200),
                              prefix_range=(5, 120), partition_size=0)
    src = set(wl.cow[:, 0].tolist())
    k, v = wl.clone_pools()
    oracle.copy_blocks(k, v, wl.cow, "f32")
    oracle.reshape_and_cache(wl.key, wl.value, k, v, wl.slot_mapping, "f32")
    for s in range(wl.num_seqs):
        L = int(wl.seq_lens[s])
        for j in range(-(-L // bs)):
            n = min(bs, L - j * bs)
            b = int(wl.block_tables[s, j])
            assert np.all(np.isfinite(k[b, :, :, :n, :])) and np.all(np.isfinite(v[b, :, :, :n])), (s, j)
    assert np.all(np.isfinite(oracle.decode(wl.q, k, v, wl.block_tables, wl.seq_lens, wl.scale, "f32")))
    assert any(int(wl.slot_mapping[s]) // bs in src for s in range(wl.num_seqs)), "no in-place writer to test"


def test_prefix_groups_of_crafted_tables():
    bs = 16
    bt = np.array([[5, 6, 7, -1],      # group 0 (first block 5)
                   [5, 6, 9, 10],      # shares 2 with the longest of group 0 (this one: 4 blocks)
                   [5, 11, -1, -1],    # shares 1
                   [20, 21, 22, -1],   # a group of one
                   [30, 31, -1, -1],   # group 4: two sequences sharing 2 blocks
                   [30, 31, 32, -1]], dtype=np.int32)
    L = np.array([40, 60, 20, 35, 20, 40], dtype=np.int32)
    grp, blk = W.prefix_groups(bt, L, bs)
    assert grp.tolist() == [0, 0, 0, 3, 4, 4]
    assert blk.tolist() == [2, 4, 1, 0, 2, 3]


def test_prefix_groups_of_the_mixed_workload_describe_real_sharing():
    wl = W.config(5, poison=False, block_size=16)
    grp, blk = W.prefix_groups(wl.block_tables, wl.seq_lens, 16)
    for s in range(wl.num_seqs):
        for t in range(s + 1, wl.num_seqs):
            if grp[t] != grp[s]:
                break
            n = min(blk[s], blk[t])
            assert np.array_equal(wl.block_tables[s, :n], wl.block_tables[t, :n])
    # every sampling group of 8 starts a prefix group (a sibling whose only block was
    # copied on write shares nothing and stands alone)
    assert set(range(0, wl.num_seqs, 8)) <= set(np.unique(grp).tolist())
    assert (blk > 16).sum() > 100
