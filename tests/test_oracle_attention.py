"""Pins for the oracle's tree-verify attention (CPU only).

Each test checks the oracle against something other than itself: a library
attention routine on a special case the pages name (tree of one node = plain
decode, chain = causal attention: "ADR-037 — EAGLE-3 with dynamic tree
port", phase rows E1.1, E1.2, E1.4), a closed form, or a hand-derived fixture.
"""
import math
import os

import numpy as np
import pytest
import torch
import torch.nn.functional as F
from scipy.special import expit

import oracle
from speculative_decoding_tree_gb300 import workloads as wl


def _sdpa(q, k, v, scale, causal=False, mask=None):
    """torch's attention in float64: q [L, d], k/v [S, d]."""
    out = F.scaled_dot_product_attention(
        torch.as_tensor(q)[None, None], torch.as_tensor(k)[None, None], torch.as_tensor(v)[None, None],
        attn_mask=None if mask is None else torch.as_tensor(mask)[None, None],
        is_causal=causal, scale=scale)
    return out[0, 0].numpy()


def _rand(rng, *shape):
    return rng.standard_normal(shape)


def test_single_node_tree_is_plain_decode():
    # tree = 1 is ordinary single-token decode over P+1 keys (phase row E1.1)
    rng = np.random.default_rng(1)
    P, d, Hq, Hkv = 37, 64, 4, 2
    q = _rand(rng, 1, Hq, d)
    kp, vp = _rand(rng, Hkv, P, d), _rand(rng, Hkv, P, d)
    kt, vt = _rand(rng, Hkv, 1, d), _rand(rng, Hkv, 1, d)
    scale = 1 / math.sqrt(d)
    out = oracle.attention_one_sequence(q, kp, vp, kt, vt, [-1], scale)
    for h in range(Hq):
        g = h // (Hq // Hkv)
        ref = _sdpa(q[:, h], np.concatenate([kp[g], kt[g]]), np.concatenate([vp[g], vt[g]]), scale)
        np.testing.assert_allclose(out[0, h], ref[0], rtol=0, atol=1e-12)


@pytest.mark.parametrize("P,N", [(0, 5), (13, 4), (508, 4), (31, 17)])
def test_chain_is_causal_attention(P, N):
    # a chain of N nodes equals causal attention over the last N rows of a
    # P+N sequence (phase row E1.2; a chain is a degenerate tree, row E1.4)
    rng = np.random.default_rng(2 + P + N)
    d, Hq, Hkv = 32, 6, 3
    qfull = _rand(rng, P + N, Hq, d)
    kfull, vfull = _rand(rng, Hkv, P + N, d), _rand(rng, Hkv, P + N, d)
    scale = 0.3
    parents = [-1] + list(range(N - 1))
    out = oracle.attention_one_sequence(qfull[P:], kfull[:, :P], vfull[:, :P], kfull[:, P:], vfull[:, P:],
                                        parents, scale)
    for h in range(Hq):
        g = h // (Hq // Hkv)
        ref = _sdpa(qfull[:, h], kfull[g], vfull[g], scale, causal=True)
        np.testing.assert_allclose(out[:, h], ref[P:], rtol=0, atol=1e-12)


def test_tree_is_union_of_chains():
    # every node sees exactly the prefix plus its root->node path, so its
    # output equals single-query attention over those keys
    rng = np.random.default_rng(3)
    spec = wl.CONFIGS[3]
    gen = torch.Generator("cpu").manual_seed(7)
    parents = wl.make_tree(spec, gen)
    N, P, d, Hq, Hkv = len(parents), 20, 16, 4, 2
    q = _rand(rng, N, Hq, d)
    kp, vp = _rand(rng, Hkv, P, d), _rand(rng, Hkv, P, d)
    kt, vt = _rand(rng, Hkv, N, d), _rand(rng, Hkv, N, d)
    out = oracle.attention_one_sequence(q, kp, vp, kt, vt, parents, 0.25)
    for i in range(N):
        path, j = [], i
        while j != -1:
            path.append(j)
            j = parents[j]
        path = path[::-1]
        for h in range(Hq):
            g = h // 2
            ref = _sdpa(q[i:i + 1, h], np.concatenate([kp[g], kt[g][path]]),
                        np.concatenate([vp[g], vt[g][path]]), 0.25)
            np.testing.assert_allclose(out[i, h], ref[0], rtol=0, atol=1e-12)


def _read_tiny_fixture(golden_dir):
    anc, dep, parents = {}, {}, None
    with open(os.path.join(golden_dir, "tiny_tree.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            if line.startswith("parents:"):
                parents = [int(x) for x in line.split(":")[1].split()]
            elif line[0].isdigit():
                node, rest = line.split(":")
                a, dd = rest.split("|")
                anc[int(node)] = set(int(x) for x in a.split())
                dep[int(node)] = int(dd)
    return parents, anc, dep


def test_visible_set_matches_hand_fixture(golden_dir):
    # zero queries make every visible score equal, so each output is the mean
    # of the visible values; one-hot values then spell out the visible set
    parents, anc, dep = _read_tiny_fixture(golden_dir)
    assert parents == wl.make_tree(wl.CONFIGS[1], None)
    N, P, Hkv = len(parents), 5, 1
    d = P + N
    q = np.zeros((N, 1, d))
    keys = np.random.default_rng(4).standard_normal((Hkv, P + N, d))
    vals = np.eye(P + N)[None]                         # value of key j = e_j
    out = oracle.attention_one_sequence(q, keys[:, :P], vals[:, :P], keys[:, P:], vals[:, P:], parents, 1.0)
    for i in range(N):
        visible = set(range(P)) | {P + j for j in anc[i]}
        expect = np.array([1.0 / len(visible) if c in visible else 0.0 for c in range(d)])
        np.testing.assert_allclose(out[i, 0], expect, rtol=0, atol=1e-15)
    assert oracle.depths(parents) == [dep[i] for i in range(N)]
    assert [oracle.ancestors(parents)[i] for i in range(N)] == [anc[i] for i in range(N)]


def test_two_keys_closed_form():
    # P = 1 prefix key plus the root: softmax of two scores is a logistic
    rng = np.random.default_rng(5)
    d, scale = 8, 0.7
    q = _rand(rng, 1, 1, d)
    k0, k1, v0, v1 = (_rand(rng, 1, 1, d) for _ in range(4))
    out = oracle.attention_one_sequence(q, k0, v0, k1, v1, [-1], scale)
    s0, s1 = scale * q[0, 0] @ k0[0, 0], scale * q[0, 0] @ k1[0, 0]
    a = expit(s0 - s1)
    np.testing.assert_allclose(out[0, 0], a * v0[0, 0] + (1 - a) * v1[0, 0], rtol=0, atol=1e-14)


def test_gqa_group_mapping():
    # query head h reads KV head h // (Hq/Hkv): with constant values per KV
    # head the output names the head it read
    rng = np.random.default_rng(6)
    N, P, d, Hq, Hkv = 3, 9, 4, 8, 2
    parents = [-1, 0, 0]
    q = _rand(rng, N, Hq, d)
    kp, kt = _rand(rng, Hkv, P, d), _rand(rng, Hkv, N, d)
    vp = np.stack([np.full((P, d), g + 1.0) for g in range(Hkv)])
    vt = np.stack([np.full((N, d), g + 1.0) for g in range(Hkv)])
    out = oracle.attention_one_sequence(q, kp, vp, kt, vt, parents, 1.0)
    for h in range(Hq):
        np.testing.assert_allclose(out[:, h], h // (Hq // Hkv) + 1.0, rtol=0, atol=1e-12)


def test_paged_equals_contiguous():
    # reading the prefix through a shuffled page table gives the same keys
    spec = wl.small_variant(5, batch=3, prefix=(20, 70), vocab=50)
    wp = wl.make_workload(spec)
    wc = wl.make_workload(spec.replace(paged=False))
    for b in range(spec.batch):
        kp, vp = oracle.prefix_kv(wp, b)
        kc, vc = oracle.prefix_kv(wc, b)
        assert kp.shape == kc.shape and np.array_equal(kp, kc) and np.array_equal(vp, vc)
    samples = [(0, 0), (5, 3), (wp.total_rows - 1, spec.hq - 1)]
    a = oracle.tree_attention(wp, samples)
    c = oracle.tree_attention(wc, samples)
    for r, h in samples:
        np.testing.assert_array_equal(a[r, h], c[r, h])


def test_sampled_equals_full():
    w = wl.make_workload(wl.small_variant(3, prefix=(40, 40)))
    full = oracle.tree_attention(w)
    samples = [(0, 0), (17, 5), (63, 31)]
    part = oracle.tree_attention(w, samples)
    for r, h in samples:
        np.testing.assert_array_equal(full[r, h], part[r, h])
    assert np.isfinite(full).all()


def test_bf16_inputs_widen_exactly():
    x = torch.tensor([1.0, 1.0078125, -3.140625, 65280.0], dtype=torch.bfloat16)
    assert oracle.tree_verify._f64(x).tolist() == [1.0, 1.0078125, -3.140625, 65280.0]


def test_large_scores_stay_finite():
    # softmax is shift-invariant; scores near 800 must not overflow
    d = 4
    q = np.full((1, 1, d), 20.0)
    k0 = np.full((1, 1, d), 10.0)      # score 800
    k1 = np.full((1, 1, d), 9.99)      # score 799.2
    v0, v1 = np.ones((1, 1, d)), -np.ones((1, 1, d))
    out = oracle.attention_one_sequence(q, k0, v0, k1, v1, [-1], 1.0)
    a = expit(800.0 - 799.2)
    np.testing.assert_allclose(out[0, 0], a - (1 - a), rtol=0, atol=1e-12)
