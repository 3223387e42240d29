"""Pins of the lm_head + argmax oracle (CPU): explicit loops on tiny inputs,
one-hot hidden rows, planted maxima and duplicated weight rows ("ADR-037 —
EAGLE-3 with dynamic tree port", phase rows E4b.9, E5a and E4b.10a)."""
import numpy as np
import torch

from oracle import lm_head


def test_explicit_loops_on_tiny_inputs():
    g = np.random.default_rng(0)
    H = g.normal(size=(3, 5))
    W = g.normal(size=(7, 5))
    ref = [[sum(H[r][k] * W[v][k] for k in range(5)) for v in range(7)] for r in range(3)]
    assert np.allclose(lm_head.lm_head_logits(H, W, block=3), ref, rtol=0, atol=1e-12)
    am, top, gap = lm_head.lm_head_argmax(H, W, block=2)
    for r in range(3):
        row = ref[r]
        best = max(range(7), key=lambda v: (row[v], -v))
        assert am[r] == best and abs(top[r] - row[best]) < 1e-12
        assert abs(gap[r] - (row[best] - max(row[v] for v in range(7) if v != best))) < 1e-12


def test_one_hot_hidden_reads_a_weight_column():
    g = np.random.default_rng(1)
    W = torch.from_numpy(g.normal(size=(300, 16))).to(torch.bfloat16)
    H = torch.zeros(16, 16, dtype=torch.bfloat16)
    H[torch.arange(16), torch.arange(16)] = 1
    logits = lm_head.lm_head_logits(H, W, block=64)
    assert np.array_equal(logits, W.double().numpy().T)
    am, _, _ = lm_head.lm_head_argmax(H, W)
    col = W.double().numpy()
    for k in range(16):
        assert am[k] == int(np.flatnonzero(col[:, k] == col[:, k].max())[0])


def test_planted_parallel_row_wins():
    # among weight rows of equal norm, the one parallel to the hidden row has
    # the largest dot product (Cauchy-Schwarz), so it is the argmax
    g = np.random.default_rng(2)
    R, Hd, V = 6, 32, 500
    H = g.normal(size=(R, Hd))
    W = g.normal(size=(V, Hd))
    W /= np.linalg.norm(W, axis=1, keepdims=True)
    planted = g.choice(V, size=R, replace=False)
    for r in range(R):
        W[planted[r]] = H[r] / np.linalg.norm(H[r])
    am, top, _ = lm_head.lm_head_argmax(H, W, block=37)
    assert np.array_equal(am, planted)
    assert np.allclose(top, np.linalg.norm(H, axis=1))


def test_duplicated_rows_go_to_the_smaller_index():
    g = np.random.default_rng(3)
    H = g.normal(size=(4, 8))
    W = g.normal(size=(50, 8))
    for r in range(4):
        v = 10 + r
        W[v] = H[r] * 10
        W[40 + r] = W[v]                      # an equal, later row
    am, _, gap = lm_head.lm_head_argmax(H, W, block=16)
    assert am.tolist() == [10, 11, 12, 13]
    assert (gap == 0).all()
