"""Pins of the tree-position RoPE oracle (CPU): the complex form of the
rotation, the relative-position property, position 0, norms, and a
hand-made tree's positions ("ADR-037 — EAGLE-3 with dynamic tree port",
phase rows E4b.5b and E6)."""
import numpy as np

from oracle import rope


def test_complex_form():
    # NeoX pairs (x[j], x[j + d/2]) as z_j = x[j] + i x[j + d/2] are multiplied
    # by exp(i * p * theta^(-2j/d))
    g = np.random.default_rng(0)
    d, theta = 16, 10000.0
    x = g.normal(size=d)
    for p in (0, 1, 7, 4096, 32767):
        z = x[:d // 2] + 1j * x[d // 2:]
        freq = np.array([theta ** (-2.0 * j / d) for j in range(d // 2)])
        w = z * np.exp(1j * p * freq)
        assert np.allclose(rope.rope_neox(x, p, theta), np.concatenate([w.real, w.imag]), rtol=0, atol=1e-12)


def test_relative_position_property():
    g = np.random.default_rng(1)
    d, theta = 64, 1e6
    q, k = g.normal(size=d), g.normal(size=d)
    for m, n, s in ((5, 3, 100), (0, 9, 4000), (20000, 19999, 777)):
        a = rope.rope_neox(q, m, theta) @ rope.rope_neox(k, n, theta)
        b = rope.rope_neox(q, m + s, theta) @ rope.rope_neox(k, n + s, theta)
        assert abs(a - b) < 1e-9


def test_position_zero_and_norms():
    g = np.random.default_rng(2)
    x = g.normal(size=(3, 128))
    assert np.array_equal(rope.rope_neox(x, 0, 1e4), x)
    y = rope.rope_neox(x, 12345, 1e4)
    pair = lambda t: t[..., :64] ** 2 + t[..., 64:] ** 2
    assert np.allclose(pair(y), pair(x))


def test_tree_positions_by_hand():
    # two sequences: b0 = the 8-node tree [-1,0,0,1,1,2,3,5] at P = 24 (depths
    # 0,1,1,2,2,2,3,3), b1 = a chain of 3 at P = 7 (depths 0,1,2)
    parents = [-1, 0, 0, 1, 1, 2, 3, 5, -1, 0, 1]
    pos = rope.tree_positions([24, 7], [0, 8, 11], parents)
    assert pos.tolist() == [24, 25, 25, 26, 26, 26, 27, 27, 7, 8, 9]


def test_scatter_layout():
    g = np.random.default_rng(3)
    R, Hq, Hkv, d = 5, 4, 2, 8
    q, k, v = g.normal(size=(R, Hq, d)), g.normal(size=(R, Hkv, d)), g.normal(size=(R, Hkv, d))
    qo, kt, vt = rope.tree_rope_scatter(q, k, v, [10], [0, R], [-1, 0, 1, 1, 0], 1e4)
    pos = [10, 11, 12, 12, 11]
    for r in range(R):
        for gg in range(Hkv):
            assert np.array_equal(vt[gg, r], v[r, gg])
            assert np.allclose(kt[gg, r], rope.rope_neox(k[r, gg], pos[r], 1e4))
        for h in range(Hq):
            assert np.allclose(qo[r, h], rope.rope_neox(q[r, h], pos[r], 1e4))
