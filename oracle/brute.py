"""Pure-Python brute force for tiny paged decode cases -- TEST INFRASTRUCTURE ONLY.

This restates, in independent code, the per-token online softmax that "Reading
vLLM's PagedAttention kernel" describes (§2 flowchart, §4 CPU reference): the
tokens of a sequence are visited in logical order, each one found through the
block table (logical position t lives in slot t % block_size of physical block
block_table[t // block_size]), and folded into a running maximum, normaliser and
weighted sum of value rows; the result is the weighted sum over the normaliser.

The pool here is logical: ``k_blocks[phys][slot]`` and ``v_blocks[phys][slot]``
are lists of head_size floats.  It shares no code with the C oracle, which uses
the two-pass softmax and the real cache layouts, so agreement between the two
pins the oracle's arithmetic.
"""
import math


class RunningSoftmax:
    """Softmax-weighted sum of rows, accumulated one (score, row) pair at a time.

    Holds the largest score seen (`top`), the sum of exp(score - top) (`mass`) and
    the sum of exp(score - top) * row (`total`).  When a larger score arrives,
    what was accumulated is brought to the new reference point first.
    """

    def __init__(self, dim):
        self.top = None
        self.mass = 0.0
        self.total = [0.0] * dim

    def add(self, score, row):
        if self.top is None:
            self.top = score
        elif score > self.top:
            shrink = math.exp(self.top - score)
            self.mass *= shrink
            self.total = [x * shrink for x in self.total]
            self.top = score
        w = math.exp(score - self.top)
        self.mass += w
        self.total = [x + w * r for x, r in zip(self.total, row)]

    def result(self):
        return [x / self.mass for x in self.total]


def paged_decode_one(q, block_table, k_blocks, v_blocks, seq_len, block_size, scale):
    """Attention output of one query row over the first `seq_len` tokens of a
    paged sequence (slots past seq_len in its last block are never looked at)."""
    acc = RunningSoftmax(len(q))
    for t in range(seq_len):
        phys = block_table[t // block_size]
        slot = t % block_size
        score = scale * math.fsum(a * b for a, b in zip(q, k_blocks[phys][slot]))
        acc.add(score, v_blocks[phys][slot])
    return acc.result()


def dense_decode_one(q, keys, values, scale):
    """softmax(scale * q K^T) V over contiguous rows (two passes, fp64)."""
    scores = [scale * math.fsum(a * b for a, b in zip(q, k)) for k in keys]
    top = max(scores)
    ex = [math.exp(s - top) for s in scores]
    total = math.fsum(ex)
    dim = len(values[0])
    return [math.fsum(ex[t] / total * values[t][j] for t in range(len(values))) for j in range(dim)]
