"""Pins of the sampled-verification oracle (CPU).

Nothing here restates the oracle's formulas: Philox is checked against the
generator's published known-answer vectors, the draw against the softmax law
it must follow (chi-square), the step against losslessness — the tokens it
emits follow the target distribution whatever the drafts propose, which is
the property the pages' rule is for ("Speculative decoding verify batches to
amortize ANE dispatch", Forge sampled-proposal bullet)."""
import os

import numpy as np
import pytest

from oracle import sampled
from oracle.tree_verify import accept, argmax_row, argmax_rows

HERE = os.path.dirname(os.path.abspath(__file__))


def softmax(x, t):
    z = np.asarray(x, dtype=np.float64) / t
    z = np.exp(z - z.max())
    return z / z.sum()


def chi2_ok(counts, probs, alpha=1e-4):
    """Pearson chi-square goodness of fit (cells with tiny expectation merged)."""
    from scipy.stats import chi2
    counts = np.asarray(counts, dtype=np.float64)
    n = counts.sum()
    exp = np.asarray(probs, dtype=np.float64) * n
    keep = exp >= 5
    c = np.append(counts[keep], counts[~keep].sum())
    e = np.append(exp[keep], exp[~keep].sum())
    c, e = c[e > 0], e[e > 0]
    stat = ((c - e) ** 2 / e).sum()
    return chi2.sf(stat, len(e) - 1) > alpha


def test_philox_known_answers(golden_dir):
    rows = [l.split() for l in open(os.path.join(golden_dir, "philox4x32_10_kat.txt")) if l.strip() and not l.startswith("#")]
    assert len(rows) == 3
    for r in rows:
        x = [int(h, 16) for h in r]
        out = sampled.philox4x32_10(*x[:6])
        assert [int(o) for o in out] == x[6:]


def test_uniforms_in_open_interval_exact_in_float32():
    u = sampled.uniforms(row=7, vocab=4096, seed=0x1234_5678_9abc, offset=99)
    assert (u > 0).all() and (u < 1).all()
    assert np.allclose(u * 2 ** 23 - 0.5, np.round(u * 2 ** 23 - 0.5))
    assert (u.astype(np.float32).astype(np.float64) == u).all()
    assert 0.45 < u.mean() < 0.55


def test_draws_follow_softmax():
    logits = np.array([0.3, -1.2, 2.0, 0.0, 1.1, -0.4])
    for t in (0.6, 1.0, 2.5):
        n = 20000
        counts = np.bincount([sampled.sample_row(logits, t, r, seed=5, offset=11) for r in range(n)],
                             minlength=6)
        assert chi2_ok(counts, softmax(logits, t)), (t, counts)


def test_low_temperature_gives_the_argmax():
    g = np.random.default_rng(3)
    for r in range(200):
        x = g.normal(size=50)
        x[g.integers(50)] += 5.0              # a clear maximum
        assert sampled.sample_row(x, 1e-3, r, seed=1, offset=2) == argmax_row(x)


def test_nan_never_drawn():
    x = np.array([np.nan, 0.0, np.nan, 0.0])
    for r in range(300):
        assert sampled.sample_row(x, 1.0, r, seed=9, offset=0) in (1, 3)
    assert sampled.sample_row(np.array([np.nan, np.nan]), 1.0, 0, seed=9, offset=0) == 0


def _walk(parents, draft, logits, t, seed, offset):
    y = [sampled.sample_row(logits[i], t, i, seed, offset) for i in range(len(parents))]
    return accept(parents, draft, y)


def test_first_token_is_lossless_whatever_the_drafts():
    # root with three children (distinct drafts), two of which have children
    V, t = 8, 0.9
    g = np.random.default_rng(7)
    parents = [-1, 0, 0, 0, 1, 2]
    logits = g.normal(size=(6, V)) * 1.5
    p0 = softmax(logits[0], t)
    for draft in ([0, 2, 5, 6, 1, 3], [0, 7, 4, 0, 0, 0]):
        n = 12000
        first = np.zeros(V)
        acc_child = np.zeros(len(parents))
        for off in range(n):
            k, path, tokens = _walk(parents, draft, logits, t, seed=123, offset=off)
            first[tokens[0]] += 1
            if k >= 1:
                acc_child[path[1]] += 1
        # the first emitted token follows p0 exactly as if no draft existed
        assert chi2_ok(first, p0), (draft, first)
        # child c is accepted with the target probability of its draft
        for c in (1, 2, 3):
            assert abs(acc_child[c] / n - p0[draft[c]]) < 4 * np.sqrt(p0[draft[c]] / n) + 1e-3


def test_second_token_follows_the_accepted_nodes_distribution():
    # chain root -> 1 -> 2: given the first draft accepted, the next emitted
    # token follows node 1's target distribution; given it rejected, the first
    # token follows p0 without the rejected draft
    V, t = 6, 1.0
    g = np.random.default_rng(11)
    parents = [-1, 0, 1]
    logits = g.normal(size=(3, V))
    logits[0, 2] += 1.0                       # make the draft likely enough
    draft = [0, 2, 4]
    second, first_rej = np.zeros(V), np.zeros(V)
    for off in range(20000):
        k, path, tokens = _walk(parents, draft, logits, t, seed=77, offset=off)
        if k >= 1:
            second[tokens[1]] += 1
        else:
            first_rej[tokens[0]] += 1
    assert chi2_ok(second, softmax(logits[1], t))
    p_ex = softmax(logits[0], t)
    p_ex[2] = 0
    p_ex /= p_ex.sum()
    assert first_rej[2] == 0 and chi2_ok(first_rej, p_ex)


def test_whole_step_is_lossless_per_sequence():
    # the step function itself (draws, walk over a batch of trees, commit):
    # over many offsets the first token each sequence emits follows that
    # sequence's root distribution, and the cache grows by the accepted rows
    from speculative_decoding_tree_gb300 import workloads as wl
    spec = wl.CONFIGS[5].replace(batch=2, hq=4, hkv=2, d=32, prefix=(3, 9), vocab=12,
                                 tree="random:5,5,3", seed=31)
    w = wl.make_workload(spec, argmax_fn=argmax_rows)
    t = 1.3
    roots = [w.seq_rows(b)[0] for b in range(w.batch)]
    logits = np.asarray(w.logits.float(), dtype=np.float64)
    first = np.zeros((w.batch, spec.vocab))
    p_before = np.asarray(w.prefix_len, dtype=np.int64).copy()
    for off in range(2500):
        st = sampled.verify_step_sampled(w, t, seed=2024, offset=off, samples=[(roots[0], 0)])
        for b, (k, path, tokens) in enumerate(st["accepted"]):
            first[b, tokens[0]] += 1
            assert int(st["prefix_len"][b]) == p_before[b] + k + 1
    for b in range(w.batch):
        assert chi2_ok(first[b], softmax(logits[roots[b]], t)), (b, first[b])
