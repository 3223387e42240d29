"""Plain float64 CPU oracle for sampled (temperature > 0) tree verification.

TEST INFRASTRUCTURE ONLY.  Only the test suite, the package's smoke check and
the benchmark's CPU-baseline / reference leg may import this module.  It
shares no code with the CUDA path and never calls it.

The rule ("Speculative decoding verify batches to amortize ANE dispatch",
Forge sampled-proposal bullet; "Speculative-decoding heads", What's not
implemented (7)): a drafted proposal is treated as deterministic; it is
accepted with its target probability, and on rejection the target
distribution with that proposal excluded is sampled.

Reading used here.  At an accepted node u, one token y_u is drawn from the
target distribution p_u = softmax(logits_u / T).  A child c of u is accepted
when its draft equals y_u; if no child matches, the walk ends at u and y_u is
the correction token (at a leaf: the bonus).  For one proposal x this is the
rule above: P(accept) = p_u(x), and given y_u != x, y_u follows p_u with x
excluded.  For several children with distinct drafts it is the same rule
applied child by child (the second child is tried against the distribution
that excludes the first, and so on).  The walk itself is the greedy one of
`tree_verify.accept` with y in place of the argmax (deepest matching node,
ties to the smallest index), which with distinct sibling drafts is exactly
the child-by-child rule.

The draw.  y_u = argmax_v (logits_u[v] / T + G_u[v]) (the Gumbel-max
construction: the argmax of Gumbel-perturbed log-weights is a sample of the
softmax), G = -log(-log U), U = ((x >> 9) + 0.5) * 2^-23 where x is word
v % 4 of Philox4x32-10 (Salmon, Moraes, Dror, Shaw, "Parallel random
numbers: as easy as 1, 2, 3", SC 2011) at counter (v // 4, r, offset_lo,
offset_hi) and key (seed_lo, seed_hi); r is the tree row's index in the
batch.  NaN logits are never drawn; the first index wins exact ties.

Parity status: Philox pinned by the generator's published known-answer
vectors; the draw by the softmax law (chi-square) and the low-temperature
limit; the step by losslessness (the emitted tokens follow the target
model's distribution whatever the drafts).
"""
from __future__ import annotations

import numpy as np

from .tree_verify import accept, commit, tree_attention

_M0, _M1 = 0xD2511F53, 0xCD9E8D57          # Philox4x32 multipliers
_W0, _W1 = 0x9E3779B9, 0xBB67AE85          # Weyl key increments
_MASK = 0xFFFFFFFF


def philox4x32_10(c0, c1, c2, c3, k0, k1):
    """Philox4x32 with 10 rounds on arrays of counters (uint32 values held in
    int64/uint64): each round multiplies words 0 and 2 by the two
    multipliers, and the new words are (hi1 ^ c1 ^ k0, lo1, hi0 ^ c3 ^ k1,
    lo0); the key is bumped by the Weyl constants between rounds."""
    c = [np.asarray(x, dtype=np.uint64) & _MASK for x in (c0, c1, c2, c3)]
    k0 = np.asarray(k0, dtype=np.uint64) & _MASK
    k1 = np.asarray(k1, dtype=np.uint64) & _MASK
    for rnd in range(10):
        if rnd:
            k0 = (k0 + _W0) & _MASK
            k1 = (k1 + _W1) & _MASK
        p0 = np.uint64(_M0) * c[0]
        p1 = np.uint64(_M1) * c[2]
        hi0, lo0 = p0 >> np.uint64(32), p0 & np.uint64(_MASK)
        hi1, lo1 = p1 >> np.uint64(32), p1 & np.uint64(_MASK)
        c = [hi1 ^ c[1] ^ k0, lo1, hi0 ^ c[3] ^ k1, lo0]
    return c


def uniforms(row, vocab, seed, offset):
    """U[v] for v in 0..vocab-1 of tree row `row`, in (0, 1), as float64: the
    top 23 bits of the Philox word plus one half, times 2^-23 (24 significant
    bits, so the value is exact in float32 as well)."""
    v = np.arange(vocab, dtype=np.uint64)
    words = philox4x32_10(v >> np.uint64(2), np.uint64(row), np.uint64(offset & _MASK),
                          np.uint64((offset >> 32) & _MASK), np.uint64(seed & _MASK),
                          np.uint64((seed >> 32) & _MASK))
    x = np.choose((v & np.uint64(3)).astype(np.int64), words)
    return ((x >> np.uint64(9)).astype(np.float64) + 0.5) * 2.0 ** -23


def gumbel(row, vocab, seed, offset):
    """G = -log(-log U) for every vocabulary entry of one row (float64)."""
    return -np.log(-np.log(uniforms(row, vocab, seed, offset)))


def perturbed(logits_row, temperature, row, seed, offset):
    """logits / T + G in float64 (NaN stays NaN)."""
    x = np.asarray(logits_row, dtype=np.float64).reshape(-1)
    return x / float(temperature) + gumbel(row, x.shape[0], seed, offset)


def draw_with_margin(logits_row, temperature, row, seed, offset):
    """(draw, margin) of one row from one evaluation of the perturbed values.
    The draw is the first index of the largest perturbed value among the
    non-NaN entries (0 for an all-NaN row); the margin is the gap between the
    largest and the second-largest of them (inf with fewer than two): a draw
    computed in lower precision agrees with this one when the gap is well
    above that precision's rounding."""
    s = perturbed(logits_row, temperature, row, seed, offset)
    ok = ~np.isnan(s)
    if not ok.any():
        return 0, float("inf")
    idx = np.flatnonzero(ok)
    y = int(idx[np.argmax(s[idx])])
    v = np.sort(s[idx])
    return y, (float(v[-1] - v[-2]) if v.shape[0] > 1 else float("inf"))


def sample_row(logits_row, temperature, row, seed, offset):
    """One draw from softmax(logits_row / T)."""
    return draw_with_margin(logits_row, temperature, row, seed, offset)[0]


def sample_rows(logits, temperature, seed, offset):
    """sample_row for every tree row r of a [R, V] logits matrix."""
    x = np.asarray(logits.float() if hasattr(logits, "float") else logits, dtype=np.float64)
    return np.array([sample_row(x[r], temperature, r, seed, offset) for r in range(x.shape[0])], dtype=np.int64)


def sample_margin(logits_row, temperature, row, seed, offset):
    """Gap between the largest and second-largest perturbed values of a row."""
    return draw_with_margin(logits_row, temperature, row, seed, offset)[1]


def verify_step_sampled(w, temperature, seed, offset, samples=None):
    """The whole step with sampled verification: attention as in the greedy
    step, one draw per tree row, the same walk with the draws in place of
    the argmax, and the same commit."""
    out = tree_attention(w, samples)
    y = sample_rows(w.logits, temperature, seed, offset)
    acc = []
    for b in range(w.batch):
        o0, o1 = w.seq_rows(b)
        acc.append(accept(w.parents[b], w.draft_tokens[o0:o1].tolist(), y[o0:o1].tolist()))
    kc, vc, new_p = commit(w, acc)
    return dict(out=out, sampled=y, accepted=acc, k_cache=kc, v_cache=vc, prefix_len=new_p)
