"""The host-side block manager (include/pa_block_manager.h), on CPU.

The manager is checked against a plain Python model of the rules the pages give
for paging ("vLLM's PagedAttention: why the KV cache is paged", §4.1 logical ->
physical mapping, §4.2 block reuse and copy-on-write) on random sequences of
operations, and against invariants that hold whatever the operations:
reference counts equal the references held by sequences, free blocks are
referenced by nobody, every block is either free or referenced, and a new
token's slot is where its sequence's block list puts it.
"""
import numpy as np
import pytest

import paged_kv_cache_306_gb300 as pa
from paged_kv_cache_306_gb300 import build as pa_build


@pytest.fixture(scope="module", autouse=True)
def _lib():
    pa_build.build()
    pa.load()


class Model:
    """The rules, written out: a stack of free ids (lowest on top), reference
    counts, and per sequence its length and block list."""

    def __init__(self, nb, bs):
        self.bs = bs
        self.free = list(range(nb - 1, -1, -1))
        self.ref = [0] * nb
        self.seqs = {}

    def take(self):
        b = self.free.pop()
        self.ref[b] = 1
        return b

    def drop(self, b):
        self.ref[b] -= 1
        if self.ref[b] == 0:
            self.free.append(b)

    def add(self, sid, n):
        need = -(-n // self.bs)
        if sid in self.seqs or need > len(self.free):
            return None
        blocks = [self.take() for _ in range(need)]
        self.seqs[sid] = [n, blocks]
        return [blocks[t // self.bs] * self.bs + t % self.bs for t in range(n)]

    def fork(self, p, c):
        n, blocks = self.seqs[p]
        for b in blocks:
            self.ref[b] += 1
        self.seqs[c] = [n, list(blocks)]

    def free_seq(self, sid):
        n, blocks = self.seqs.pop(sid)
        for b in reversed(blocks):
            self.drop(b)

    def append(self, ids):
        # feasibility, decided in batch order on the counts
        need, dropped = 0, {}
        for s in ids:
            n, blocks = self.seqs[s]
            if n % self.bs == 0:
                need += 1
            elif self.ref[blocks[-1]] - dropped.get(blocks[-1], 0) > 1:
                need += 1
                dropped[blocks[-1]] = dropped.get(blocks[-1], 0) + 1
        if need > len(self.free):
            return None
        slots, copies = [], []
        for s in ids:
            n, blocks = self.seqs[s]
            if n % self.bs == 0:
                blocks.append(self.take())
            elif self.ref[blocks[-1]] > 1:
                src, dst = blocks[-1], self.take()
                copies.append((src, dst))
                self.drop(src)
                blocks[-1] = dst
            slots.append(blocks[-1] * self.bs + n % self.bs)
            self.seqs[s][0] = n + 1
        return slots, copies


def check_state(bm, m, nb):
    assert bm.num_free_blocks == len(m.free)
    held = [0] * nb
    for sid, (n, blocks) in m.seqs.items():
        assert bm.seq_len(sid) == n
        for b in blocks:
            held[b] += 1
    for b in range(nb):
        assert bm.refcount(b) == m.ref[b] == held[b]
        assert (held[b] == 0) == (b in set(m.free))
    if m.seqs:
        ids = sorted(m.seqs)
        mb = max(1, max(len(m.seqs[s][1]) for s in ids))
        bt, sl = bm.block_tables(ids, mb)
        for i, s in enumerate(ids):
            n, blocks = m.seqs[s]
            assert sl[i] == n
            assert bt[i, :len(blocks)].tolist() == blocks
            assert np.all(bt[i, len(blocks):] == -1)


@pytest.mark.parametrize("seed", range(6))
@pytest.mark.parametrize("bs", [1, 4, 16])
def test_random_operations_match_the_model(seed, bs):
    rng = np.random.default_rng(seed * 100 + bs)
    nb = 64
    bm, m = pa.BlockManager(nb, bs), Model(nb, bs)
    next_id = 0
    for _ in range(300):
        op = rng.choice(["add", "fork", "free", "append", "append"])
        if op == "add":
            n = int(rng.integers(0, 5 * bs + 3))
            want = m.add(next_id, n)
            if want is None:
                with pytest.raises(pa.PAError) as e:
                    bm.add_sequence(next_id, n)
                assert e.value.status == pa.PA_ERR_OUT_OF_BLOCKS
            else:
                assert bm.add_sequence(next_id, n).tolist() == want
            next_id += 1
        elif op == "fork" and m.seqs:
            p = int(rng.choice(sorted(m.seqs)))
            m.fork(p, next_id)
            bm.fork(p, next_id)
            next_id += 1
        elif op == "free" and m.seqs:
            s = int(rng.choice(sorted(m.seqs)))
            m.free_seq(s)
            bm.free_sequence(s)
        elif op == "append" and m.seqs:
            ids = [int(x) for x in rng.permutation(sorted(m.seqs))[:int(rng.integers(1, len(m.seqs) + 1))]]
            want = m.append(ids)
            if want is None:
                before = bm.num_free_blocks
                with pytest.raises(pa.PAError) as e:
                    bm.append_tokens(ids)
                assert e.value.status == pa.PA_ERR_OUT_OF_BLOCKS
                assert bm.num_free_blocks == before          # nothing changed
            else:
                slots, copies = bm.append_tokens(ids)
                assert slots.tolist() == want[0]
                assert [tuple(c) for c in copies.tolist()] == want[1]
        check_state(bm, m, nb)
    bm.close()


def test_new_token_slot_follows_the_block_list():
    bs = 4
    bm = pa.BlockManager(32, bs)
    bm.add_sequence(7, 5)
    for _ in range(9):
        (slot,), copies = bm.append_tokens([7])
        assert len(copies) == 0
        n = bm.seq_len(7)
        bt, _ = bm.block_tables([7], 8)
        assert slot == bt[0, (n - 1) // bs] * bs + (n - 1) % bs


def test_fork_then_append_copies_the_shared_partial_block_once():
    bs = 4
    bm = pa.BlockManager(16, bs)
    bm.add_sequence(0, 6)                      # blocks 0, 1 (1 half full)
    bm.fork(0, 1)
    bm.fork(0, 2)
    assert bm.refcount(1) == 3
    slots, copies = bm.append_tokens([0, 1, 2])
    # two of the three sharers copy block 1, the last writes in place
    assert copies.tolist() == [[1, 2], [1, 3]]
    assert slots.tolist() == [2 * bs + 2, 3 * bs + 2, 1 * bs + 2]
    assert bm.refcount(1) == 1 and bm.refcount(0) == 3
    bt, sl = bm.block_tables([0, 1, 2], 4)
    assert bt[:, :2].tolist() == [[0, 2], [0, 3], [0, 1]] and sl.tolist() == [7, 7, 7]


def test_fork_at_a_block_boundary_needs_no_copy():
    bm = pa.BlockManager(8, 4)
    bm.add_sequence(0, 8)
    bm.fork(0, 1)
    slots, copies = bm.append_tokens([0, 1])
    assert len(copies) == 0 and slots.tolist() == [2 * 4, 3 * 4]


def test_free_returns_blocks_only_when_unreferenced():
    bm = pa.BlockManager(8, 4)
    bm.add_sequence(0, 9)                      # 3 blocks
    bm.fork(0, 1)
    assert bm.num_free_blocks == 5
    bm.free_sequence(0)
    assert bm.num_free_blocks == 5             # still held by 1
    bm.free_sequence(1)
    assert bm.num_free_blocks == 8
    # freed blocks come back lowest first
    assert bm.add_sequence(2, 4).tolist() == [0, 1, 2, 3]


def test_bad_calls_are_refused_and_change_nothing():
    bm = pa.BlockManager(4, 4)
    bm.add_sequence(0, 4)
    for call, status in [(lambda: bm.add_sequence(0, 1), pa.PA_ERR_INVALID_ARG),       # id taken
                         (lambda: bm.fork(9, 1), pa.PA_ERR_INVALID_ARG),               # no parent
                         (lambda: bm.fork(0, 0), pa.PA_ERR_INVALID_ARG),               # child exists
                         (lambda: bm.free_sequence(5), pa.PA_ERR_INVALID_ARG),
                         (lambda: bm.append_tokens([0, 0]), pa.PA_ERR_INVALID_ARG),    # listed twice
                         (lambda: bm.append_tokens([3]), pa.PA_ERR_INVALID_ARG),
                         (lambda: bm.add_sequence(1, 13), pa.PA_ERR_OUT_OF_BLOCKS),
                         (lambda: bm.block_tables([0], 0), pa.PA_ERR_INVALID_ARG),
                         (lambda: bm.refcount(4), pa.PA_ERR_INVALID_ARG)]:
        with pytest.raises(pa.PAError) as e:
            call()
        assert e.value.status == status
    assert bm.num_free_blocks == 3 and bm.seq_len(0) == 4
    with pytest.raises(pa.PAError):
        pa.BlockManager(0, 4)
    with pytest.raises(pa.PAError):
        pa.BlockManager(4, 0)


def test_exhausted_pool_refuses_the_whole_batch():
    bm = pa.BlockManager(3, 2)
    bm.add_sequence(0, 2)
    bm.add_sequence(1, 2)
    # both need a fresh block, one is free
    with pytest.raises(pa.PAError) as e:
        bm.append_tokens([0, 1])
    assert e.value.status == pa.PA_ERR_OUT_OF_BLOCKS
    assert bm.seq_len(0) == 2 and bm.seq_len(1) == 2 and bm.num_free_blocks == 1
    slots, _ = bm.append_tokens([1])
    assert slots.tolist() == [2 * 2]


def test_prefix_groups_match_the_tables():
    """The manager's description of shared prefixes agrees with one computed from
    its own block tables, after forks, appends and copy-on-write."""
    import workloads as W
    bm = pa.BlockManager(400, 16)
    bm.add_sequence(0, 100)
    for c in range(1, 6):
        bm.fork(0, c)
    bm.add_sequence(10, 40)
    bm.fork(10, 11)
    bm.add_sequence(20, 7)
    ids = [0, 1, 2, 3, 4, 5, 10, 11, 20]
    for step in range(40):
        bm.append_tokens([i for i in ids if (step + i) % 3 != 0])
    bt, sl = bm.block_tables(ids, 64)
    grp, blk = bm.prefix_groups(ids)
    g2, b2 = W.prefix_groups(bt, sl, 16)
    assert grp.tolist() == g2.tolist() and blk.tolist() == b2.tolist()
    assert grp.tolist()[:6] == [0] * 6 and blk[8] == 0
