"""Host-side checks of the synthetic workload generator (CPU only)."""
import pytest
import torch

import oracle
from speculative_decoding_tree_gb300 import workloads as wl


def _valid(parents):
    return parents[0] == -1 and all(0 <= parents[i] < i for i in range(1, len(parents)))


@pytest.mark.parametrize("n,size,maxdepth", [(3, 64, 6), (4, 60, 6)])
def test_tree_shapes(n, size, maxdepth):
    gen = torch.Generator("cpu").manual_seed(wl.CONFIGS[n].seed)
    p = wl.make_tree(wl.CONFIGS[n], gen)
    assert len(p) == size and _valid(p)
    assert max(oracle.depths(p)) <= maxdepth
    # depth is non-decreasing in node order (renumbered by depth)
    d = oracle.depths(p)
    assert d == sorted(d)


def test_factor_tree_respects_branching():
    gen = torch.Generator("cpu").manual_seed(1004)
    p = wl.make_tree(wl.CONFIGS[4], gen)
    d = oracle.depths(p)
    factors = [4, 3, 2, 2, 1, 1]
    for i in range(len(p)):
        kids = sum(1 for c in range(1, len(p)) if p[c] == i)
        assert kids <= factors[d[i]] if d[i] < len(factors) else kids == 0


def test_eagle2_tree_is_deep():
    gen = torch.Generator("cpu").manual_seed(1003)
    p = wl.make_tree(wl.CONFIGS[3], gen)
    d = oracle.depths(p)
    assert max(d) >= 3
    # at most 8 children per node
    for i in range(len(p)):
        assert sum(1 for c in range(1, len(p)) if p[c] == i) <= 8


def test_random_trees():
    gen = torch.Generator("cpu").manual_seed(5)
    for _ in range(50):
        p = wl._tree_random(gen, 16, 64, 8)
        assert 16 <= len(p) <= 64 and _valid(p)
        assert max(oracle.depths(p)) <= 8


def test_workload_layout_and_determinism():
    spec = wl.small_variant(5, batch=3, prefix=(20, 60), vocab=100)
    a = wl.make_workload(spec)
    b = wl.make_workload(spec)
    assert torch.equal(a.q, b.q) and torch.equal(a.page_table, b.page_table)
    assert a.q.shape == (a.total_rows, spec.hq, spec.d)
    assert a.k_tree.shape == (spec.hkv, a.total_rows, spec.d)
    assert a.k_cache.shape[1:] == (spec.hkv, 16, spec.d)
    ids = a.page_table[a.page_table >= 0]
    assert ids.unique().numel() == ids.numel() == a.k_cache.shape[0]
    for bb in range(spec.batch):
        assert oracle.seq_capacity(a, bb) >= int(a.prefix_len[bb]) + len(a.parents[bb])


def test_drafts_planted_rate():
    spec = wl.small_variant(3, prefix=(8, 8), vocab=50)
    w = wl.make_workload(spec)
    am = torch.arange(w.total_rows) % 50
    d = wl.plant_drafts(w, am)
    match = [int(d[c]) == int(am[w.parents[0][c]]) for c in range(1, w.total_rows)]
    assert 0.5 < sum(match) / len(match) < 0.9
    for c in range(1, w.total_rows):
        assert 0 <= int(d[c]) < 50
