"""Pins for the oracle's argmax, acceptance and commit (CPU only)."""
import itertools
import os

import numpy as np
import pytest
import torch

import oracle
from speculative_decoding_tree_gb300 import workloads as wl


# ---------------------------------------------------------------- argmax

def test_argmax_planted_and_ties():
    rng = np.random.default_rng(0)
    for _ in range(50):
        n = int(rng.integers(1, 300))
        row = rng.standard_normal(n)
        j = int(rng.integers(0, n))
        row[j] = 100.0
        assert oracle.argmax_row(row) == j
    # small integer values: many ties; reference = first index of a stable
    # sort on descending value (a different algorithm)
    for _ in range(50):
        row = rng.integers(0, 4, size=int(rng.integers(1, 40))).astype(float)
        ref = int(np.lexsort((np.arange(row.size), -row))[0])
        assert oracle.argmax_row(row) == ref


def test_argmax_nan_policy():
    nan, inf = float("nan"), float("inf")
    assert oracle.argmax_row([nan, 1.0, 3.0, 3.0]) == 2
    assert oracle.argmax_row([nan, nan]) == 0
    assert oracle.argmax_row([-inf, nan]) == 0
    assert oracle.argmax_row([nan, -inf]) == 1
    assert oracle.argmax_row([-0.0, 0.0]) == 0
    assert oracle.argmax_row([0.0, -0.0]) == 0
    assert oracle.argmax_row([-inf, -inf, -1e30]) == 2


def test_argmax_rows_matches_scan():
    rng = np.random.default_rng(1)
    x = rng.integers(-3, 3, size=(40, 57)).astype(float)
    x[rng.random(x.shape) < 0.1] = np.nan
    x[3] = np.nan
    got = oracle.argmax_rows(x)
    assert [oracle.argmax_row(r) for r in x] == got.tolist()


def test_argmax_bf16_adjacent_values():
    # values one bf16 ulp apart are distinct; widening keeps their order
    row = torch.tensor([12.0, 12.0625, 12.0, 12.0625], dtype=torch.bfloat16)
    assert oracle.argmax_rows(row[None])[0] == 1


# ---------------------------------------------------------------- acceptance

def _greedy_walk(parents, draft, am):
    """The walk of "ADR-037", phase row E5a: start at the root and move to the
    child whose draft equals the target argmax at the current node, until no
    child matches (unique when sibling drafts are distinct)."""
    children = {}
    for c in range(1, len(parents)):
        children.setdefault(parents[c], []).append(c)
    path = [0]
    while True:
        cur = path[-1]
        nxt = [c for c in children.get(cur, []) if draft[c] == am[cur]]
        if not nxt:
            return path
        assert len(nxt) == 1
        path.append(nxt[0])


def _ok_depth_rule(parents, draft, am):
    """Third formulation: ok[0]; ok[i] = ok[parent] and draft[i] == am[parent];
    k = deepest ok node's depth, end = smallest index at that depth."""
    dep = oracle.depths(parents)
    ok = [True] + [False] * (len(parents) - 1)
    for i in range(1, len(parents)):
        ok[i] = ok[parents[i]] and draft[i] == am[parents[i]]
    k = max(dep[i] for i in range(len(parents)) if ok[i])
    end = min(i for i in range(len(parents)) if ok[i] and dep[i] == k)
    return k, end


def test_tiny_workload_planted_result(golden_dir):
    fx = {}
    with open(os.path.join(golden_dir, "tiny_tree.txt")) as f:
        for line in f:
            if line.startswith("accept_k:"):
                fx["k"] = int(line.split(":")[1])
            elif line.startswith("accept_path:"):
                fx["path"] = [int(x) for x in line.split(":")[1].split()]
    w = wl.make_workload(wl.CONFIGS[1], argmax_fn=oracle.argmax_rows)
    am = oracle.argmax_rows(w.logits).tolist()
    k, path, tokens = oracle.accept(w.parents[0], w.draft_tokens.tolist(), am)
    assert k == fx["k"] and path == fx["path"]
    assert tokens == [int(w.draft_tokens[1]), int(w.draft_tokens[3]), am[3]]


def test_brute_force_equals_greedy_walk():
    rng = np.random.default_rng(2)
    gen = torch.Generator("cpu").manual_seed(3)
    for trial in range(200):
        parents = wl._tree_random(gen, 1, 30, 6)
        N = len(parents)
        am = rng.integers(0, 5, size=N).tolist()
        # distinct sibling drafts, each matching with probability 1/2
        draft = [0] * N
        used = {}
        for c in range(1, N):
            p = parents[c]
            taken = used.setdefault(p, set())
            if am[p] not in taken and rng.random() < 0.5:
                draft[c] = am[p]
            else:
                draft[c] = int(rng.integers(10, 10_000))
                while draft[c] in taken:
                    draft[c] += 1
            taken.add(draft[c])
        k, path, tokens = oracle.accept(parents, draft, am)
        assert path == _greedy_walk(parents, draft, am)
        assert (k, path[-1]) == _ok_depth_rule(parents, draft, am)
        assert tokens == [draft[c] for c in path[1:]] + [am[path[-1]]]


def test_exhaustive_match_patterns():
    # every match pattern on small trees, duplicates among siblings allowed:
    # brute force equals the ok/depth rule (deepest, then smallest index)
    for parents in ([-1, 0, 0, 1, 1, 2, 3, 5], [-1, 0, 1, 1, 0, 4], [-1, 0, 0, 0]):
        N = len(parents)
        am = [100 + i for i in range(N)]
        for pattern in itertools.product([0, 1], repeat=N - 1):
            draft = [0] + [am[parents[c]] if pattern[c - 1] else 7 for c in range(1, N)]
            k, path, _ = oracle.accept(parents, draft, am)
            assert (k, path[-1]) == _ok_depth_rule(parents, draft, am)
            assert len(path) == k + 1


def test_edge_cases():
    am = [5, 6, 7, 8]
    # empty accept: root only, correction token am[0] ("ADR-037", Phase E5)
    k, path, tok = oracle.accept([-1, 0, 0, 0], [1, 0, 0, 0], am)
    assert (k, path, tok) == (0, [0], [5])
    # full accept of a chain
    k, path, tok = oracle.accept([-1, 0, 1, 2], [1, 5, 6, 7], am)
    assert (k, path, tok) == (3, [0, 1, 2, 3], [5, 6, 7, 8])
    # two fully matching branches: the deepest wins
    k, path, _ = oracle.accept([-1, 0, 0, 2], [1, 5, 5, 7], am)
    assert (k, path) == (2, [0, 2, 3])
    # equal depth: smallest end index
    k, path, _ = oracle.accept([-1, 0, 0], [1, 5, 5], am)
    assert (k, path) == (1, [0, 1])
    # a single node
    assert oracle.accept([-1], [3], [9]) == (0, [0], [9])


def _read_burst_fixture(golden_dir):
    rows = []
    with open(os.path.join(golden_dir, "expected_tokens_per_burst.txt")) as f:
        for line in f:
            if line.strip() and not line.startswith("#"):
                K, p, v, dec = line.split()
                rows.append((int(K), float(p), float(v), int(dec)))
    return rows


def _chain_expectation(K, p):
    """Enumerate all 2^K match patterns of a K-draft chain through the oracle."""
    parents = [-1] + list(range(K))
    am = [1000 + i for i in range(K + 1)]
    e = 0.0
    for pattern in itertools.product([0, 1], repeat=K):
        prob = np.prod([p if m else 1 - p for m in pattern])
        draft = [0] + [am[c - 1] if pattern[c - 1] else -1 for c in range(1, K + 1)]
        k, _, tokens = oracle.accept(parents, draft, am)
        assert len(tokens) == k + 1
        e += prob * len(tokens)
    return e


def test_expected_tokens_per_burst(golden_dir):
    for K, p, printed, dec in _read_burst_fixture(golden_dir):
        e = _chain_expectation(K, p)
        assert round(e, dec) == printed
        assert abs(e - sum(p ** j for j in range(K + 1))) < 1e-12
    assert abs(_chain_expectation(3, 0.6) - 2.176) < 1e-12


def test_expected_tokens_monte_carlo():
    rng = np.random.default_rng(11)
    K, p, n = 3, 0.6, 40_000
    parents = [-1, 0, 1, 2]
    am = [1, 2, 3, 4]
    coins = rng.random((n, K))
    lens = []
    for t in range(n):
        draft = [0] + [am[c - 1] if coins[t, c - 1] < p else 0 for c in range(1, K + 1)]
        lens.append(oracle.accept(parents, draft, am)[0] + 1)
    lens = np.array(lens)
    se = lens.std() / np.sqrt(n)
    assert abs(lens.mean() - (1 + p + p * p + p ** 3)) < 5 * se


# ---------------------------------------------------------------- commit

@pytest.mark.parametrize("paged", [False, True])
def test_commit_touches_only_accepted_rows(paged):
    spec = wl.small_variant(5, batch=3, prefix=(17, 90), vocab=64, paged=paged)
    w = wl.make_workload(spec, canary=-7.0, argmax_fn=oracle.argmax_rows)
    res = oracle.verify_step(w, samples=[])
    kc, vc, newp = res["k_cache"], res["v_cache"], res["prefix_len"]
    changed_k = kc.view(torch.int16) != w.k_cache.view(torch.int16)
    expect = torch.zeros_like(changed_k)
    for b, (k, path, _) in enumerate(res["accepted"]):
        P = int(w.prefix_len[b])
        assert int(newp[b]) == P + k + 1
        o0, _ = w.seq_rows(b)
        for t, node in enumerate(path):
            pos = P + t
            if paged:
                pid, slot = int(w.page_table[b, pos // 16]), pos % 16
                assert torch.equal(kc[pid, :, slot], w.k_tree[:, o0 + node])
                assert torch.equal(vc[pid, :, slot], w.v_tree[:, o0 + node])
                expect[pid, :, slot] = True
            else:
                assert torch.equal(kc[b, :, pos], w.k_tree[:, o0 + node])
                expect[b, :, pos] = True
    # every changed element lies in a written row (rows may equal by chance)
    assert not (changed_k & ~expect).any()


def test_commit_k0_writes_anchor_only():
    spec = wl.CONFIGS[2].replace(prefix=(30, 30), vocab=40)
    w = wl.make_workload(spec, canary=0.5)
    am = oracle.argmax_rows(w.logits)
    w.draft_tokens = torch.tensor([0] + [int(am[i]) + 1 if int(am[i]) + 1 < 40 else 0 for i in range(3)],
                                  dtype=torch.int32)
    acc = [oracle.accept(w.parents[0], w.draft_tokens.tolist(), am.tolist())]
    assert acc[0][0] == 0
    kc, vc, newp = oracle.commit(w, acc)
    assert int(newp[0]) == 31
    assert torch.equal(kc[0, :, 30], w.k_tree[:, 0])
    assert torch.equal(kc[0, :, 31:], w.k_cache[0, :, 31:])
    assert torch.equal(kc[0, :, :30], w.k_cache[0, :, :30])


def test_commit_capacity_boundary():
    # k+1 rows fit exactly when P+k+1 == capacity; one more and nothing moves
    spec = wl.CONFIGS[2].replace(prefix=(30, 30), vocab=40, cache_margin=0)
    w = wl.make_workload(spec, argmax_fn=oracle.argmax_rows)
    acc = [(2, [0, 1, 2], [1, 2, 3])]
    w.prefix_len[0] = w.capacity - 3
    kc, vc, newp = oracle.commit(w, acc)
    assert int(newp[0]) == w.capacity
    assert torch.equal(kc[0, :, -1], w.k_tree[:, 2])
    w.prefix_len[0] = w.capacity - 2
    kc, vc, newp = oracle.commit(w, acc)
    assert int(newp[0]) == w.capacity - 2
    assert torch.equal(kc.view(torch.int16), w.k_cache.view(torch.int16))


# ---------------------------------------------------------------- tree validity

def test_check_tree_hand_cases():
    # a parent array is a tree in topological order exactly when the root's
    # parent is -1 and every other node points at an earlier node
    assert oracle.check_tree([-1])
    assert oracle.check_tree([-1, 0, 0, 1, 1, 2, 3, 5])          # the tiny workload's tree
    assert oracle.check_tree([-1, 0, 1, 2, 3])                   # a chain
    assert oracle.check_tree([-1, 0, 0, 0, 0])                   # a star
    assert not oracle.check_tree([])                             # no root
    assert not oracle.check_tree([0])                            # root with a parent
    assert not oracle.check_tree([-1, -1])                       # a second root
    assert not oracle.check_tree([-1, 1])                        # a self parent
    assert not oracle.check_tree([-1, 0, 3, 1])                  # a forward parent
    assert not oracle.check_tree([-1, 0, 0, -2])                 # a negative parent below -1
    assert not oracle.check_tree([-1, 0, 7])                     # a parent past the end
    assert not oracle.check_tree([2, -1, 0])                     # the root not first


def test_check_tree_counts_recursive_trees():
    # closed form: with parent[0] = -1 and parent[i] in {0 .. i-1}, node i has
    # i choices, so exactly (n-1)! of the (n+3)^n arrays over {-2 .. n} are
    # valid; any mistake in the bounds (<= i, >= -1, a free root) changes the count
    import math
    for n in range(1, 6):
        count = sum(oracle.check_tree(list(p)) for p in itertools.product(range(-2, n + 1), repeat=n))
        assert count == math.factorial(n - 1), n


def test_check_tree_agrees_with_the_ancestor_walk():
    # on random arrays, validity equals "every node's parent chain reaches the
    # root through strictly smaller indices", checked here by a separate walk
    rng = np.random.default_rng(11)
    seen = {True: 0, False: 0}
    for _ in range(400):
        n = int(rng.integers(1, 12))
        p = [-1] + [int(rng.integers(0, i)) for i in range(1, n)]
        if rng.random() < 0.5:
            j = int(rng.integers(0, n))
            p[j] = int(rng.integers(-2, n + 1))
        ok = True
        for i in range(n):
            j, steps = i, 0
            while j != 0 and ok:
                q = p[j]
                ok = 0 <= q < j
                j, steps = (q if ok else 0), steps + 1
            ok = ok and p[0] == -1
        assert oracle.check_tree(p) == ok
        seen[ok] += 1
    assert seen[True] > 50 and seen[False] > 50
