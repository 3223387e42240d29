"""Plain float64 CPU oracle for the tree-position RoPE and K/V scatter.

TEST INFRASTRUCTURE ONLY.  Only the test suite, the package's smoke check and
the benchmark's CPU-baseline / reference leg may import this module.  It
shares no code with the CUDA path and never calls it.

What it computes ("ADR-037 — EAGLE-3 with dynamic tree port", phase row
E4b.5b: rotary embedding on Q and K at tree positions base_pos +
tree_depths[i], NeoX style, over the whole head dimension; phase row E6: the
seq-major to head-major permute and the tree K/V the attention reads):

* position of tree row i of sequence b: P_b + depth(i) (the same reading as
  the attention and the commit: the committed row t sits at P_b + t);
* NeoX rotation of a head vector x of even length d at position p: for
  j < d/2, with angle p * theta^(-2j/d), the pair (x[j], x[j + d/2]) becomes
  (x[j] cos - x[j + d/2] sin, x[j + d/2] cos + x[j] sin);
* q_out[r, h] = rot(q[r, h], pos_r); k_tree[g, r] = rot(k[r, g], pos_r);
  v_tree[g, r] = v[r, g] (head-major, as tree_verify_attn reads them).

Parity status: pinned by the complex-number form of the rotation, the
relative-position property of RoPE (q . k depends only on the position
difference), position 0 being the identity, norm preservation, and a
hand-made tree's positions.
"""
from __future__ import annotations

import numpy as np

from .tree_verify import depths


def _f64(t):
    if hasattr(t, "double"):
        return t.double().cpu().numpy()
    return np.asarray(t, dtype=np.float64)


def rope_neox(x, pos, theta):
    """x [..., d] float64 rotated at position pos (scalar or broadcastable to x[..., 0])."""
    x = np.asarray(x, dtype=np.float64)
    d = x.shape[-1]
    half = d // 2
    inv = theta ** (-2.0 * np.arange(half) / d)
    ang = np.asarray(pos, dtype=np.float64)[..., None] * inv
    c, s = np.cos(ang), np.sin(ang)
    a, b = x[..., :half], x[..., half:]
    return np.concatenate([a * c - b * s, b * c + a * s], axis=-1)


def tree_positions(prefix_len, node_offsets, parents_flat):
    """[total_rows] int64: P_b + depth(i) for every tree row."""
    off = np.asarray(node_offsets, dtype=np.int64)
    par = np.asarray(parents_flat, dtype=np.int64)
    P = np.asarray(prefix_len, dtype=np.int64)
    out = np.empty(off[-1], dtype=np.int64)
    for b in range(len(off) - 1):
        o0, o1 = off[b], off[b + 1]
        out[o0:o1] = P[b] + np.asarray(depths(par[o0:o1].tolist()), dtype=np.int64)
    return out


def tree_rope_scatter(q, k, v, prefix_len, node_offsets, parents_flat, theta):
    """(q_out [R, Hq, d], k_tree [Hkv, R, d], v_tree [Hkv, R, d]) in float64."""
    pos = tree_positions(prefix_len, node_offsets, parents_flat)
    q = _f64(q)
    k = _f64(k)
    v = _f64(v)
    q_out = rope_neox(q, pos[:, None], theta)
    k_rot = rope_neox(k, pos[:, None], theta)
    return q_out, np.transpose(k_rot, (1, 0, 2)).copy(), np.transpose(v, (1, 0, 2)).copy()
