"""Pure-Python brute force for tiny paged decode cases -- TEST INFRASTRUCTURE ONLY.

This restates, in independent code, the per-token online-softmax walk that
"Reading vLLM's PagedAttention kernel" §4 (runnable CPU reference) and its §2
flowchart describe: walk the block table in logical order, look up each
physical block, fold every token into a running maximum m, normaliser l and
accumulator acc, stop at the true sequence length, and finish with acc / l.

The pool here is logical: ``k_blocks[phys][slot]`` and ``v_blocks[phys][slot]``
are lists of head_size floats, as in the pages' dict-of-blocks.  It shares no
code with the C oracle, which uses the two-pass softmax and the real cache
layouts, so agreement between the two pins the oracle's arithmetic.
"""
import math


def paged_decode_one(q, block_table, k_blocks, v_blocks, seq_len, block_size, scale):
    """Attention output of one query row over `seq_len` paged tokens."""
    dim = len(q)
    run_max = -math.inf
    norm = 0.0
    acc = [0.0] * dim
    pos = 0
    for phys in block_table:
        if pos >= seq_len:
            break
        for slot in range(block_size):
            if pos >= seq_len:          # the last block may be partly filled
                break
            key = k_blocks[phys][slot]
            val = v_blocks[phys][slot]
            score = scale * math.fsum(a * b for a, b in zip(q, key))
            new_max = max(run_max, score)
            # rescale what was accumulated under the old maximum
            rescale = 0.0 if run_max == -math.inf else math.exp(run_max - new_max)
            weight = math.exp(score - new_max)
            norm = norm * rescale + weight
            acc = [a * rescale + weight * v for a, v in zip(acc, val)]
            run_max = new_max
            pos += 1
    return [a / norm for a in acc]


def dense_decode_one(q, keys, values, scale):
    """softmax(scale * q K^T) V over contiguous rows (two passes, fp64)."""
    scores = [scale * math.fsum(a * b for a, b in zip(q, k)) for k in keys]
    top = max(scores)
    ex = [math.exp(s - top) for s in scores]
    total = math.fsum(ex)
    dim = len(values[0])
    return [math.fsum(ex[t] / total * values[t][j] for t in range(len(values))) for j in range(dim)]
