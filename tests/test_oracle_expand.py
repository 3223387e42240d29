"""Pins of the dynamic draft-tree expansion oracle (CPU).

Top-K is checked against the pages' ordering example and a library stable
sort; log softmax against scipy; the expansion against a hand-derived tree
(the pages' grandchild-before-sibling case), against brute force over whole
candidate trees, and against invariants ("ADR-037 — EAGLE-3 with dynamic tree
port", phase rows E4a and E4b.10a, §4 Phase E4)."""
import os
import zlib

import numpy as np
import pytest
from scipy.special import log_softmax

from oracle import expand

HERE = os.path.dirname(os.path.abspath(__file__))


# ---------------------------------------------------------------- top-K

def test_topk_pages_ordering_example():
    # phase row E4b.10a: [0.0, -3e38, -2e38] must come out as 0.0, -2e38, -3e38
    # (the selection compares the raw values; nothing is clamped first)
    row = np.array([0.0, -3e38, -2e38], dtype=np.float32)
    assert expand.topk_row(row, 3) == [0, 2, 1]
    assert expand.topk_row(row, 2) == [0, 2]


def test_topk_ties_and_nan():
    assert expand.topk_row([1.0, 3.0, np.nan, 3.0, 2.0], 3) == [1, 3, 4]
    assert expand.topk_row([np.nan, np.nan], 2) == []
    assert expand.topk_row([np.nan, 5.0, np.nan], 4) == [1]
    assert expand.topk_row([-np.inf, -np.inf, 0.0], 3) == [2, 0, 1]


def test_topk_matches_a_stable_sort():
    g = np.random.default_rng(0)
    for _ in range(200):
        x = g.integers(-3, 4, size=int(g.integers(1, 40))).astype(np.float64)   # many ties
        k = int(g.integers(1, 10))
        ref = np.argsort(-x, kind="stable")[:k].tolist()
        assert expand.topk_row(x, k) == ref


# ---------------------------------------------------------------- log softmax

def test_log_softmax_matches_scipy():
    g = np.random.default_rng(1)
    for scale in (0.1, 3.0, 80.0, 1e4):
        x = g.normal(size=300) * scale
        lp = expand.log_softmax_row(x)
        assert np.allclose(lp, log_softmax(x), rtol=1e-12, atol=1e-12 * scale)
        assert abs(np.exp(lp).sum() - 1.0) < 1e-12


def test_log_softmax_special_values():
    lp = expand.log_softmax_row([0.0, np.nan, 0.0, -np.inf])
    assert np.allclose(lp[[0, 2]], np.log(0.5)) and np.isnan(lp[1]) and np.isneginf(lp[3])
    with pytest.raises(ValueError):
        expand.log_softmax_row([0.0, np.inf])


# ---------------------------------------------------------------- expansion

def _golden():
    rows, expects = {}, []
    with open(os.path.join(HERE, "golden", "expand_best_first.txt")) as f:
        lines = f.read().splitlines()
    for line in lines:
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        if line.startswith("path") or line.startswith("default"):
            key, probs = line.split("|")
            key = tuple(int(t) for t in key.split()[1:]) if key.startswith("path") else None
            rows[key] = np.log(np.array([float(p) for p in probs.split()]))
        else:
            parts = [p.split() for p in line.split("|")]
            expects.append((int(parts[0][1]), [int(t) for t in parts[1]], [int(t) for t in parts[2]],
                            [int(t) for t in parts[3]], [float(t) for t in parts[4]]))
    return rows, expects


def test_golden_grandchild_before_sibling():
    rows, expects = _golden()
    calls = []

    def logits_of(step, j, path):
        calls.append(tuple(path))
        return rows.get(tuple(path), rows[None])

    assert len(expects) == 2
    for width, tokens, parents, depths, cumprob in expects:
        calls.clear()
        t = expand.expand_tree(logits_of, 9, k=2, n_max=5, width=width, max_depth=3)
        assert t["tokens"] == tokens and t["parents"] == parents and t["depths"] == depths
        assert np.allclose(t["cum"], np.log(cumprob), rtol=0, atol=1e-12)
        # the node at the depth limit is never sent to the drafter
        assert (9, 0, 2, 0) not in calls


def _path_drafter(V, scale, salt):
    """A drafter whose logits depend on the whole token path (so the same
    node gets the same row whatever order it is reached in)."""
    def logits_of(step, j, path):
        seed = zlib.crc32(np.asarray(path, dtype=np.int64).tobytes()) ^ salt
        return np.random.default_rng(seed).normal(size=V) * scale
    return logits_of


def _all_nodes(logits_of, root, k, max_depth):
    """Every node of the full K-ary candidate tree down to max_depth, with its
    cumulative log-probability, computed with scipy and a stable sort."""
    nodes = {(root,): 0.0}
    frontier = [(root,)]
    for _ in range(max_depth):
        nxt = []
        for path in frontier:
            x = logits_of(0, 0, list(path))
            lp = log_softmax(x)
            for v in np.argsort(-x, kind="stable")[:k]:
                child = path + (int(v),)
                nodes[child] = nodes[path] + lp[v]
                nxt.append(child)
        frontier = nxt
    return nodes


@pytest.mark.parametrize("n_max", [2, 5, 13, 30, 60])
def test_best_first_is_the_best_nodes_of_the_whole_tree(n_max):
    # with W = 1 the tree is the root plus the N - 1 nodes of largest
    # cumulative log-probability in the full candidate tree (a child is never
    # more likely than its parent, so that set is a connected tree)
    k, depth, V = 3, 4, 20
    for salt in range(4):
        drafter = _path_drafter(V, 1.5, salt)
        t = expand.expand_tree(drafter, 7, k=k, n_max=n_max, width=1, max_depth=depth)
        paths = set()
        for i in range(len(t["tokens"])):
            p, u = [], i
            while u >= 0:
                p.append(t["tokens"][u])
                u = t["parents"][u]
            paths.add(tuple(p[::-1]))
        nodes = _all_nodes(drafter, 7, k, depth)
        best = sorted(nodes, key=lambda p: -nodes[p])[:n_max]
        assert paths == set(best)
        # best-first: the cumulative values leave the pool in order
        assert all(a >= b for a, b in zip(t["cum"][1:], t["cum"][2:]))


@pytest.mark.parametrize("n_max", [4, 10, 40])
def test_unbounded_width_builds_level_by_level(n_max):
    # W >= N: every pending candidate moves at once, so the tree is all of
    # levels 0..L-1 plus the best nodes of level L
    k, depth, V = 3, 5, 16
    drafter = _path_drafter(V, 2.0, 99)
    t = expand.expand_tree(drafter, 3, k=k, n_max=n_max, width=n_max, max_depth=depth)
    nodes = _all_nodes(drafter, 3, k, depth)
    want, level, need = [], 0, n_max
    while need > 0:
        lv = sorted([p for p in nodes if len(p) == level + 1], key=lambda p: -nodes[p])
        want += lv[:need]
        need -= min(need, len(lv))
        level += 1
    got = set()
    for i in range(len(t["tokens"])):
        p, u = [], i
        while u >= 0:
            p.append(t["tokens"][u])
            u = t["parents"][u]
        got.add(tuple(p[::-1]))
    assert got == set(want)


def test_invariants_on_seeded_tables():
    g = np.random.default_rng(5)
    for trial in range(30):
        k = int(g.integers(1, 9))
        width = int(g.integers(1, 9))
        n_max = int(g.integers(1, 70))
        max_depth = int(g.integers(1, 8))
        V = int(g.integers(k, 60))
        steps = n_max + 1
        table = g.normal(size=(steps, width, V)) * 2.0
        t = expand.expand_tree(expand.table_drafter(table), 5, k, n_max, width, max_depth)
        n = len(t["tokens"])
        assert 1 <= n <= n_max
        for i in range(1, n):
            p = t["parents"][i]
            assert 0 <= p < i
            assert t["depths"][i] == t["depths"][p] + 1 <= max_depth
            assert t["cum"][i] <= t["cum"][p]
        for p in set(t["parents"][1:]):
            sib = [t["tokens"][i] for i in range(n) if t["parents"][i] == p]
            assert len(sib) == len(set(sib)) <= k
        # the budget is met unless the depth limit ran the pool dry
        full = sum(min(k, V) ** d for d in range(max_depth + 1))
        assert n == min(n_max, full)


def test_token_map_renames_children_only():
    g = np.random.default_rng(8)
    V, k = 12, 3
    table = g.normal(size=(20, 2, V))
    tmap = g.permutation(1000)[:V]
    a = expand.expand_tree(expand.table_drafter(table), 4, k, 9, 2, 5)
    b = expand.expand_tree(expand.table_drafter(table), 4, k, 9, 2, 5, token_map=tmap)
    assert a["parents"] == b["parents"] and a["cum"] == b["cum"]
    assert b["tokens"] == [4] + [int(tmap[v]) for v in a["tokens"][1:]]


def test_equal_values_go_to_the_first_generated():
    # hand-derived: K = 2, W = 2, budget 5, vocabulary 2.  Root row [0, -inf]:
    # A = token 0 (log-prob 0), B = token 1 (-inf); step 0 moves both.  Step 1
    # expands A with [0, -inf] (A.0 at 0, A.1 at -inf) and B with [0, 0]
    # (B.0 and B.1 at -inf).  A.0 goes first; A.1, B.0 and B.1 tie at -inf and
    # the first generated, A.1 (expanded node 0, rank 1), wins over B.0
    # (expanded node 1, rank 0).
    ninf = -np.inf
    table = np.array([[[0.0, ninf], [0.0, ninf]],
                      [[0.0, ninf], [0.0, 0.0]]])
    t = expand.expand_tree(expand.table_drafter(table), 3, k=2, n_max=5, width=2, max_depth=4)
    assert t["tokens"] == [3, 0, 1, 0, 1]
    assert t["parents"] == [-1, 0, 0, 1, 1]
    assert t["cum"][3] == 0.0 and np.isneginf(t["cum"][4])


def test_plus_inf_row_gives_no_children():
    # hand-derived: K = 2, W = 1, budget 4, vocabulary 3.  Root row [1, 0, -inf]:
    # A = token 0 at 1 - log(e + 1), B = token 1 at -log(e + 1); step 0 moves A.
    # Step 1 expands A with a row holding +inf: outside the log-softmax's
    # domain, so A gets no children and the expansion reports it; B moves.
    # Step 2 expands B with [0, 0, 0]: B.0 (token 0, first generated) enters
    # at -log(e + 1) - log 3 and fills the budget.
    inf = np.inf
    table = np.array([[[1.0, 0.0, -inf]], [[0.0, inf, 0.0]], [[0.0, 0.0, 0.0]]])
    t = expand.expand_tree(expand.table_drafter(table), 7, k=2, n_max=4, width=1, max_depth=5)
    assert t["bad_logits"]
    assert t["tokens"] == [7, 0, 1, 0]
    assert t["parents"] == [-1, 0, 0, 2]
    assert t["depths"] == [0, 1, 1, 2]
    lse = np.log(np.e + 1.0)
    assert np.allclose(t["cum"], [0.0, 1.0 - lse, -lse, -lse - np.log(3.0)], rtol=0, atol=1e-15)
    # without the +inf entry nothing is reported
    table[1, 0, 1] = 0.0
    assert not expand.expand_tree(expand.table_drafter(table), 7, k=2, n_max=4, width=1, max_depth=5)["bad_logits"]
