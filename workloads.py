"""Seeded synthetic inputs for paged decode: shared by the tests, the smoke check
and the benchmark, and by both the CUDA path and the CPU oracle.

This module holds no attention arithmetic.  It draws random values, allocates
physical blocks the way a block manager would (shuffled ids, prefix sharing
with reference counts, copy-on-write decisions), and lays the values out in
the pool shapes the kernels and the oracle read:
    k_cache [num_blocks, num_kv_heads, head_size/x, block_size, x]
    v_cache [num_blocks, num_kv_heads, head_size, block_size]
with x = 16 / element_size ("Reading vLLM's PagedAttention kernel", §3.1).

One decode step of one layer is modelled ("vLLM's PagedAttention: why the KV
cache is paged", §2.3): every sequence appends one new token whose K/V rows
(`key`, `value`) are written through `slot_mapping`, after any copy-on-write
block copies (`cow`), and `seq_lens` already counts that token.  Slots that hold
no valid token are filled with NaN when `poison` is set, so a kernel that reads
them produces a visible error.

Arrays are numpy: fp32 -> float32, fp16 -> float16, bf16 -> uint16 bit patterns,
FP8 E4M3 -> uint8 codes.  An FP8 pool ("fp8") holds codes whose values times the
workload's k_scale / v_scale are the K / V values; its queries and new-token rows
are in a 16-bit `q_dtype`.
"""
from dataclasses import dataclass, field
import math

import numpy as np

ELEM_BYTES = {"f32": 4, "f16": 2, "bf16": 2, "fp8": 1}
NP_STORAGE = {"f32": np.float32, "f16": np.float16, "bf16": np.uint16, "fp8": np.uint8}
BF16_NAN = np.uint16(0x7FC0)
FP8_NAN = np.uint8(0x7F)
FP8_SCALE = 1.0 / 64   # k_scale = v_scale of the FP8 workloads: N(0,1) values span codes up to ~400
_CHUNK = 1 << 23


def pack_x(dtype):
    return 16 // ELEM_BYTES[dtype]


def _bf16_bits(f32):
    """float32 -> bfloat16 bit patterns, round to nearest even (finite inputs)."""
    u = np.ascontiguousarray(f32, dtype=np.float32).view(np.uint32)
    return ((u + (((u >> 16) & 1) + 0x7FFF)) >> 16).astype(np.uint16)


def cast(f32, dtype):
    """Round float32 values to the storage dtype (FP8: torch's float8_e4m3fn rounding)."""
    if dtype == "f32":
        return np.ascontiguousarray(f32, dtype=np.float32)
    if dtype == "f16":
        return f32.astype(np.float16)
    if dtype == "fp8":
        import torch
        x = np.clip(np.ascontiguousarray(f32, dtype=np.float32), -448.0, 448.0)
        return torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    return _bf16_bits(f32)


def fill_value(dtype, poison):
    if not poison:
        return 0
    return {"bf16": BF16_NAN, "fp8": FP8_NAN}.get(dtype, np.nan)


def randn(rng, shape, dtype, std=1.0, scale=1.0):
    """N(0, std^2) draws stored as `dtype`; FP8 stores the codes nearest to x / scale."""
    v = rng.standard_normal(shape, dtype=np.float32)
    if std != 1.0:
        v *= np.float32(std)
    if dtype == "fp8":
        v /= np.float32(scale)
    return cast(v, dtype)


@dataclass
class Workload:
    """One decode step of one attention layer over a paged pool."""
    name: str
    dtype: str
    num_seqs: int
    num_heads: int
    num_kv_heads: int
    head_size: int
    block_size: int
    num_blocks: int
    scale: float
    partition_size: int          # 0: one pass per sequence, -1: planner picks, >0: tokens
    q: np.ndarray                # [S, H, D]
    key: np.ndarray              # [S, Hkv, D], the new token of every sequence
    value: np.ndarray            # [S, Hkv, D]
    slot_mapping: np.ndarray     # int64 [S]
    k_cache: np.ndarray
    v_cache: np.ndarray
    block_tables: np.ndarray     # int32 [S, max_blocks_per_seq], unused entries -1
    seq_lens: np.ndarray         # int32 [S], includes the new token
    cow: np.ndarray = field(default_factory=lambda: np.zeros((0, 2), np.int64))
    unique_tokens: int = 0       # valid tokens summed over distinct physical blocks
    meta: dict = field(default_factory=dict)
    q_dtype: str = None          # dtype of q, key, value and out (defaults to the cache dtype)
    query_start_loc: np.ndarray = None  # prefill: int32 [S + 1], the chunk of sequence s is rows qsl[s]..qsl[s+1]-1
    k_scale: float = 1.0         # an FP8 pool reads back as code * scale
    v_scale: float = 1.0

    def __post_init__(self):
        if self.q_dtype is None:
            self.q_dtype = self.dtype

    @property
    def max_blocks_per_seq(self):
        return self.block_tables.shape[1]

    @property
    def max_seq_len(self):
        return int(self.seq_lens.max()) if self.num_seqs else 0

    @property
    def total_tokens(self):
        return int(self.seq_lens.astype(np.int64).sum())

    def clone_pools(self):
        return self.k_cache.copy(), self.v_cache.copy()


def _empty_pools(nb, hkv, d, bs, dtype, poison):
    x = pack_x(dtype)
    st = NP_STORAGE[dtype]
    k = np.empty((nb, hkv, d // x, bs, x), dtype=st)
    v = np.empty((nb, hkv, d, bs), dtype=st)
    k.fill(fill_value(dtype, poison))
    v.fill(fill_value(dtype, poison))
    return k, v


def _fill_blocks(rng, k, v, ids, dtype, std, scale=1.0):
    """Random values into whole physical blocks `ids` (chunked to bound memory)."""
    ids = np.asarray(ids, dtype=np.int64)
    per = int(np.prod(k.shape[1:]))
    step = max(1, _CHUNK // per)
    for i in range(0, len(ids), step):
        c = ids[i:i + step]
        k[c] = randn(rng, (len(c),) + k.shape[1:], dtype, std, scale)
        v[c] = randn(rng, (len(c),) + v.shape[1:], dtype, std, scale)


def _poison_tail(k, v, phys, first_invalid, dtype, poison):
    """Slots first_invalid.. of block `phys` hold no valid token."""
    fv = fill_value(dtype, poison)
    k[phys, :, :, first_invalid:, :] = fv
    v[phys, :, :, first_invalid:] = fv


def _finish(name, dtype, S, H, Hkv, D, bs, nb, tables, seq_lens, k, v, rng, partition_size,
            q_std=1.0, kv_std=1.0, poison=True, cow=None, unique_tokens=None, meta=None, q_dtype=None,
            kv_scale=1.0):
    """Common tail: new-token slots, poison, q/key/value draws."""
    mb = max(len(t) for t in tables) if S else 1
    bt = np.full((S, mb), -1, dtype=np.int32)
    for s, t in enumerate(tables):
        bt[s, :len(t)] = t
    sl = np.asarray(seq_lens, dtype=np.int32)
    slots = np.empty(S, dtype=np.int64)
    fv = fill_value(dtype, poison)
    for s in range(S):
        pos = int(sl[s]) - 1                         # position of the new token
        phys = int(bt[s, pos // bs])
        off = pos % bs
        slots[s] = phys * bs + off
        k[phys, :, :, off, :] = fv                   # written by the step itself
        v[phys, :, :, off] = fv
    qd = q_dtype or dtype
    q = randn(rng, (S, H, D), qd, q_std)
    key = randn(rng, (S, Hkv, D), qd, kv_std)
    value = randn(rng, (S, Hkv, D), qd, kv_std)
    if unique_tokens is None:
        unique_tokens = int(sl.astype(np.int64).sum())
    return Workload(name=name, dtype=dtype, num_seqs=S, num_heads=H, num_kv_heads=Hkv, head_size=D,
                    block_size=bs, num_blocks=nb, scale=1.0 / math.sqrt(D),
                    partition_size=partition_size, q=q, key=key, value=value, slot_mapping=slots,
                    k_cache=k, v_cache=v, block_tables=bt, seq_lens=sl,
                    cow=np.zeros((0, 2), np.int64) if cow is None else np.asarray(cow, np.int64).reshape(-1, 2),
                    unique_tokens=unique_tokens, meta=meta or {}, q_dtype=qd, k_scale=kv_scale,
                    v_scale=kv_scale)


def _fp8_args(dtype, q_dtype, kv_scale):
    if dtype == "fp8":
        if q_dtype not in ("f16", "bf16"):
            raise ValueError("an FP8 pool needs fp16 or bf16 queries")
        return q_dtype, FP8_SCALE if kv_scale is None else kv_scale
    return q_dtype, 1.0


def make_private(name, dtype, seq_lens, num_heads, num_kv_heads, head_size, block_size, *, seed,
                 num_blocks=None, pool_factor=1.25, placement="shuffled", q_std=1.0, kv_std=1.0,
                 poison=True, partition_size=0, q_dtype=None, kv_scale=None):
    """Sequences with private blocks only.

    placement:
      "shuffled"   -- sequence s takes blocks s*n .. s*n+n-1 of one random
                      permutation of the pool's ids (equivalently: contiguous
                      tables, then one random relabelling of physical ids);
      "contiguous" -- the identity placement, sequence after sequence.
    """
    q_dtype, kv_scale = _fp8_args(dtype, q_dtype, kv_scale)
    rng = np.random.default_rng(seed)
    seq_lens = [int(x) for x in seq_lens]
    S = len(seq_lens)
    nblk = [-(-L // block_size) for L in seq_lens]
    need = sum(nblk)
    nb = num_blocks if num_blocks is not None else max(1, math.ceil(pool_factor * need))
    if nb < need:
        raise ValueError("pool too small")
    if placement == "contiguous":
        ids = np.arange(need)
    else:
        ids = rng.permutation(nb)[:need]
    tables, c = [], 0
    for n in nblk:
        tables.append(ids[c:c + n].astype(np.int32))
        c += n
    k, v = _empty_pools(nb, num_kv_heads, head_size, block_size, dtype, poison)
    _fill_blocks(rng, k, v, ids, dtype, kv_std, kv_scale)
    for s, L in enumerate(seq_lens):
        r = L % block_size
        if r:
            _poison_tail(k, v, int(tables[s][-1]), r, dtype, poison)
    return _finish(name, dtype, S, num_heads, num_kv_heads, head_size, block_size, nb, tables, seq_lens,
                   k, v, rng, partition_size, q_std=q_std, kv_std=kv_std, poison=poison, q_dtype=q_dtype,
                   kv_scale=kv_scale)


def make_prefill(name, dtype, context_lens, query_lens, num_heads, num_kv_heads, head_size, block_size, *,
                 seed, pool_factor=1.25, poison=True):
    """Chunked prefill: sequence s has context_lens[s] cached tokens and a chunk of
    query_lens[s] new tokens (positions context .. context + n - 1), whose K/V rows
    (`key`, `value`, `slot_mapping`, one row per new token in sequence order) the
    step writes before the prefill; `q` holds one query row per new token.
    Physical blocks are a random permutation of the pool's ids; slots not yet
    written (the chunk's and those past the sequence) are poisoned.
    """
    rng = np.random.default_rng(seed)
    ctx = [int(x) for x in context_lens]
    qn = [int(x) for x in query_lens]
    S = len(ctx)
    L = [c + n for c, n in zip(ctx, qn)]
    bs = block_size
    nblk = [-(-l // bs) for l in L]
    need = sum(nblk)
    nb = max(1, math.ceil(pool_factor * need))
    ids = rng.permutation(nb)[:need]
    tables, c = [], 0
    for n in nblk:
        tables.append(ids[c:c + n].astype(np.int32))
        c += n
    k, v = _empty_pools(nb, num_kv_heads, head_size, bs, dtype, poison)
    _fill_blocks(rng, k, v, ids, dtype, 1.0)
    fv = fill_value(dtype, poison)
    slots = []
    for s in range(S):
        if L[s] % bs:
            _poison_tail(k, v, int(tables[s][-1]), L[s] % bs, dtype, poison)
        for pos in range(ctx[s], L[s]):          # the chunk: written by the step itself
            phys, off = int(tables[s][pos // bs]), pos % bs
            slots.append(phys * bs + off)
            k[phys, :, :, off, :] = fv
            v[phys, :, :, off] = fv
    mb = max(nblk) if S else 1
    bt = np.full((S, mb), -1, dtype=np.int32)
    for s, t in enumerate(tables):
        bt[s, :len(t)] = t
    T = sum(qn)
    qsl = np.concatenate([[0], np.cumsum(qn)]).astype(np.int32)
    q = randn(rng, (T, num_heads, head_size), dtype)
    key = randn(rng, (T, num_kv_heads, head_size), dtype)
    value = randn(rng, (T, num_kv_heads, head_size), dtype)
    return Workload(name=name, dtype=dtype, num_seqs=S, num_heads=num_heads, num_kv_heads=num_kv_heads,
                    head_size=head_size, block_size=bs, num_blocks=nb, scale=1.0 / math.sqrt(head_size),
                    partition_size=0, q=q, key=key, value=value, slot_mapping=np.asarray(slots, np.int64),
                    k_cache=k, v_cache=v, block_tables=bt, seq_lens=np.asarray(L, np.int32),
                    unique_tokens=int(sum(L)), meta={"context_lens": ctx, "query_lens": qn},
                    query_start_loc=qsl)


def prefill_config(*, poison=True, seed=None):
    """Chunked prefill of a Qwen2.5-7B-shaped layer (fp16, 28/4 heads, D 128, bs 16):
    16 sequences, each a chunk of 512 new tokens after U{0..3584} cached ones."""
    sd = 406 if seed is None else seed
    rng = np.random.default_rng(sd)
    ctx = rng.integers(0, 3585, size=16)
    return make_prefill("qwen2.5-7b-prefill-chunk512-f16", "f16", ctx, [512] * 16, 28, 4, 128, 16, seed=sd + 1000,
                        poison=poison)


def make_prefix_shared(name, dtype, num_groups, group_size, num_heads, num_kv_heads, head_size,
                       block_size, *, seed, len_range=(16, 8192), prefix_range=(256, 2048),
                       pool_factor=1.25, poison=True, partition_size=-1, q_dtype=None, kv_scale=None):
    """Parallel-sampling groups that share prefix blocks (refcount > 1).

    Group g has a prefix of P_g tokens.  Sequence i of the group has L_i tokens
    (log-uniform) and history L_i - 1.  It references the group's prefix blocks
    that its history reaches: every full prefix block, and the partial last one
    only while its history lies inside the prefix.  Beyond the prefix it owns
    private blocks (the private block that continues a partial prefix block
    starts with a copy of the prefix tokens).  The new token then goes to
    position L_i - 1: into a fresh block when that position starts a block, by
    copy-on-write when the target block is shared (refcount > 1), in place
    otherwise ("vLLM's PagedAttention: why the KV cache is paged", §4.2).
    """
    q_dtype, kv_scale = _fp8_args(dtype, q_dtype, kv_scale)
    rng = np.random.default_rng(seed)
    bs = block_size
    S = num_groups * group_size
    lo, hi = len_range
    L = np.exp(rng.uniform(math.log(lo), math.log(hi), size=S)).round().astype(np.int64)
    L = np.clip(L, lo, hi)
    P = rng.integers(prefix_range[0], prefix_range[1] + 1, size=num_groups)

    # logical plan: per seq a list of ("shared", g, j) or ("private", n) block refs
    prefix_nblk = [-(-int(p) // bs) for p in P]
    plans = []
    n_private = 0
    for i in range(S):
        g = i // group_size
        hist = int(L[i]) - 1
        p = int(P[g])
        refs = []
        if hist <= p:
            for j in range(-(-hist // bs)):
                refs.append(("shared", g, j))
        else:
            for j in range(p // bs):
                refs.append(("shared", g, j))
            for j in range(p // bs, -(-hist // bs)):
                refs.append(("private", n_private))
                n_private += 1
        if hist % bs == 0:                       # new token opens a fresh block
            refs.append(("private", n_private))
            n_private += 1
        plans.append(refs)
    n_shared = sum(prefix_nblk)
    # copy-on-write destinations: at most one per sequence
    need = n_shared + n_private + S
    nb = max(1, math.ceil(pool_factor * need))
    perm = rng.permutation(nb).astype(np.int64)
    shared_ids, c = [], 0
    for g in range(num_groups):
        shared_ids.append(perm[c:c + prefix_nblk[g]])
        c += prefix_nblk[g]
    private_ids = perm[c:c + n_private]
    c += n_private
    spare = list(perm[c:])

    k, v = _empty_pools(nb, num_kv_heads, head_size, bs, dtype, poison)
    # prefix content: the group's prefix tokens, partial last block poisoned past P_g
    for g in range(num_groups):
        _fill_blocks(rng, k, v, shared_ids[g], dtype, 1.0, kv_scale)
        r = int(P[g]) % bs
        if r:
            _poison_tail(k, v, int(shared_ids[g][-1]), r, dtype, poison)
    _fill_blocks(rng, k, v, private_ids, dtype, 1.0, kv_scale)

    tables = []
    refcount = {}
    for i, refs in enumerate(plans):
        g = i // group_size
        p = int(P[g])
        row = []
        for j, ref in enumerate(refs):
            if ref[0] == "shared":
                phys = int(shared_ids[ref[1]][ref[2]])
                refcount[phys] = refcount.get(phys, 0) + 1
            else:
                phys = int(private_ids[ref[1]])
                refcount[phys] = 1
                if j == p // bs and p % bs:
                    # continues the partial prefix block: starts with its prefix tokens
                    src = int(shared_ids[g][j])
                    r = p % bs
                    k[phys, :, :, :r, :] = k[src, :, :, :r, :]
                    v[phys, :, :, :r] = v[src, :, :, :r]
            row.append(phys)
        tables.append(np.asarray(row, dtype=np.int32))
        # a private block that holds the new token holds nothing past it
        Li = int(L[i])
        last = (Li - 1) // bs
        if refs[last][0] == "private" and Li % bs:
            _poison_tail(k, v, row[last], Li % bs, dtype, poison)

    # copy-on-write for new tokens that land in a shared block
    cow = []
    for i in range(S):
        pos = int(L[i]) - 1
        j = pos // bs
        phys = int(tables[i][j])
        if refcount.get(phys, 1) > 1:
            dst = int(spare.pop(0))
            cow.append((phys, dst))
            refcount[phys] -= 1
            refcount[dst] = 1
            tables[i] = tables[i].copy()
            tables[i][j] = dst
    cow = np.asarray(cow, dtype=np.int64).reshape(-1, 2)
    # the last sharer of a copied block writes its new token there in place, after
    # the copies: until then the slot holds the prefix token the copies take along
    src_before = {int(b): (k[b].copy(), v[b].copy()) for b in set(cow[:, 0].tolist())}

    # distinct physical blocks and their valid-token counts (for byte accounting)
    valid = {}
    for i in range(S):
        for j, phys in enumerate(tables[i]):
            n = min(bs, int(L[i]) - j * bs)
            valid[int(phys)] = max(valid.get(int(phys), 0), n)
    unique_tokens = int(sum(valid.values()))
    wl = _finish(name, dtype, S, num_heads, num_kv_heads, head_size, bs, nb, tables, L, k, v, rng,
                 partition_size, poison=poison, cow=None, unique_tokens=unique_tokens,
                 meta={"prefix_lens": P.tolist(), "group_size": group_size}, q_dtype=q_dtype, kv_scale=kv_scale)
    # _finish poisons the new-token slot of the (post-copy) target block; a
    # copy-on-write destination is still unwritten before the step, so the
    # poison there is what the copy must overwrite.  A copy's source keeps its
    # tokens, the slot of an in-place writer included, which the copies carry.
    for b, (kb, vb) in src_before.items():
        wl.k_cache[b] = kb
        wl.v_cache[b] = vb
    wl.cow = cow
    return wl


# --- the five decode-layer workloads -------------------------------------------------

CONFIG_NAMES = {
    1: "tiny-f32",
    2: "qwen2.5-7b-layer-f16",
    3: "llama-7b-layer-f16",
    4: "long-context-bf16",
    5: "mixed-prefix-f16",
}


def config(i, *, poison=True, block_size=None, seed=None, kv_dtype=None):
    """Workload i (1..5) at its full size; seed defaults to 306 + i.

    kv_dtype="fp8" keeps every shape and the query dtype but stores the pool as
    FP8 E4M3 codes (scales FP8_SCALE); the tiny fp32 workload has no FP8 form.
    """
    sd = 306 + i if seed is None else seed
    if kv_dtype not in (None, "fp8"):
        raise ValueError(kv_dtype)
    if kv_dtype == "fp8":
        if i == 1:
            raise ValueError("the fp32 workload has no FP8 form")
        wl0 = {2: "f16", 3: "f16", 4: "bf16", 5: "f16"}[i]
        return _config(i, sd, poison, block_size, cache="fp8", q_dtype=wl0)
    return _config(i, sd, poison, block_size)


def _config(i, sd, poison, block_size, cache=None, q_dtype=None):
    def dt(d):
        return cache or d
    suffix = "-fp8kv" if cache else ""
    if i == 1:
        rng = np.random.default_rng(sd)
        L = rng.integers(1, 257, size=4)
        wl = make_private(CONFIG_NAMES[1], "f32", L, 8, 8, 64, 16, seed=sd + 1000, num_blocks=128,
                          placement="shuffled", poison=poison, partition_size=0)
        return wl
    if i == 2:
        rng = np.random.default_rng(sd)
        L = rng.integers(512, 4097, size=64)
        return make_private(CONFIG_NAMES[2] + suffix, dt("f16"), L, 28, 4, 128, 16, seed=sd + 1000,
                            placement="shuffled", poison=poison, partition_size=-1, q_dtype=q_dtype)
    if i == 3:
        return make_private(CONFIG_NAMES[3] + suffix, dt("f16"), [2048] * 16, 32, 32, 128, 16, seed=sd,
                            num_blocks=2048, placement="shuffled", kv_std=0.5, poison=poison,
                            partition_size=-1, q_dtype=q_dtype)
    if i == 4:
        return make_private(CONFIG_NAMES[4] + suffix, dt("bf16"), [32768, 65536, 98304, 131072], 32, 8, 128,
                            16, seed=sd, pool_factor=1.25, placement="shuffled", poison=poison,
                            partition_size=512, q_dtype=q_dtype)
    if i == 5:
        return make_prefix_shared(CONFIG_NAMES[5] + f"-bs{block_size or 16}" + suffix, dt("f16"), 32, 8, 32, 8,
                                  128, block_size or 16, seed=sd, poison=poison, partition_size=-1,
                                  q_dtype=q_dtype)
    raise ValueError(i)


def prefix_groups(block_tables, seq_lens, block_size):
    """(prefix_group, prefix_blocks), int32 [S] each: runs of consecutive sequences
    whose first logical block is one physical block form a group (id: the index of
    its first sequence); prefix_blocks[s] = how many leading block-table entries
    sequence s has in common with the longest sequence of its group (0 in a group
    of one) -- the blocks a fork family still shares."""
    bt = np.asarray(block_tables)
    nblk = -(-np.asarray(seq_lens, dtype=np.int64) // block_size)
    S = len(nblk)
    grp = np.zeros(S, dtype=np.int32)
    blk = np.zeros(S, dtype=np.int32)
    i = 0
    while i < S:
        j = i + 1
        while j < S and nblk[i] > 0 and nblk[j] > 0 and bt[j, 0] == bt[i, 0]:
            j += 1
        ref = i + int(np.argmax(nblk[i:j]))
        for t in range(i, j):
            n = int(min(nblk[t], nblk[ref]))
            eq = bt[t, :n] == bt[ref, :n]
            grp[t] = i
            blk[t] = 0 if j - i == 1 else (n if eq.all() else int(np.argmin(eq)))
        i = j
    return grp, blk


def subset(wl, seqs):
    """The same pool with a sub-batch of sequences (for sampled oracle checks)."""
    seqs = np.asarray(seqs, dtype=np.int64)
    return Workload(name=wl.name + "-subset", dtype=wl.dtype, num_seqs=len(seqs),
                    num_heads=wl.num_heads, num_kv_heads=wl.num_kv_heads, head_size=wl.head_size,
                    block_size=wl.block_size, num_blocks=wl.num_blocks, scale=wl.scale,
                    partition_size=wl.partition_size, q=np.ascontiguousarray(wl.q[seqs]),
                    key=np.ascontiguousarray(wl.key[seqs]), value=np.ascontiguousarray(wl.value[seqs]),
                    slot_mapping=np.ascontiguousarray(wl.slot_mapping[seqs]), k_cache=wl.k_cache,
                    v_cache=wl.v_cache, block_tables=np.ascontiguousarray(wl.block_tables[seqs]),
                    seq_lens=np.ascontiguousarray(wl.seq_lens[seqs]), meta=dict(wl.meta), q_dtype=wl.q_dtype,
                    k_scale=wl.k_scale, v_scale=wl.v_scale)


def to_torch(a, dtype, device):
    """numpy storage array -> torch tensor of the logical dtype on `device`."""
    import torch
    if dtype == "bf16":
        t = torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16)
    elif dtype == "fp8":
        t = torch.from_numpy(np.ascontiguousarray(a).view(np.uint8)).view(torch.float8_e4m3fn)
    else:
        t = torch.from_numpy(np.ascontiguousarray(a))
    return t.to(device)


def from_torch(t, dtype):
    """torch tensor -> numpy storage array (bf16 as uint16 bits)."""
    import torch
    t = t.detach().cpu().contiguous()
    if dtype == "bf16":
        return t.view(torch.int16).numpy().view(np.uint16)
    if dtype == "fp8":
        return t.view(torch.uint8).numpy()
    return t.numpy()
