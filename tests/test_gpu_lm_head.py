"""Fused lm_head + argmax on the GPU vs the oracle (GPU).

The kernel sums bf16 products in fp32 on the tensor cores, the oracle in
float64, so the two logits of a row differ by rounding: about 1e-5 for these
sizes, bounded by TOL here.  Where the oracle's largest logit beats every
other by more than 2 * TOL the argmax must be equal; where it does not (a near
tie) the GPU's choice must be a near maximum.  Exact ties (duplicated weight
rows) must go to the smaller index."""
import numpy as np
import pytest
import torch

from oracle import lm_head
from speculative_decoding_tree_gb300 import workloads as wl
from speculative_decoding_tree_gb300.runner import DeviceLmHead

pytestmark = pytest.mark.gpu

TOL = 2e-3


def run(spec, hidden=None, weight=None):
    lm = DeviceLmHead(spec, hidden=hidden, weight=weight)
    lm.run()
    torch.cuda.synchronize()
    return lm


def check(lm, hidden, weight, rows=None):
    assert int(lm.status[0]) == 0
    h = hidden if rows is None else hidden[rows]
    am_ref, top_ref, gap = lm_head.lm_head_argmax(h, weight)
    am = lm.argmax.cpu().numpy().astype(np.int64)
    mx = lm.max_logit.cpu().numpy().astype(np.float64)
    if rows is not None:
        am, mx = am[rows], mx[rows]
    assert np.abs(mx - top_ref).max() <= TOL
    clear = gap > 2 * TOL
    assert np.array_equal(am[clear], am_ref[clear]), np.flatnonzero(am != am_ref)
    for i in np.flatnonzero(~clear):              # a near tie: the choice is a near maximum
        logit = float(h[i].double() @ weight[am[i]].double())
        assert logit >= top_ref[i] - 2 * TOL
    return clear.mean()


SMALL = [
    wl.LmHeadSpec("lm-1x64-v1", 1, 64, 1, 3.0, 11),
    wl.LmHeadSpec("lm-64x256-v1000", 64, 256, 1000, 3.0, 12),
    wl.LmHeadSpec("lm-60x512-v4099", 60, 512, 4099, 3.0, 13),
    wl.LmHeadSpec("lm-130x128-v777", 130, 128, 777, 3.0, 14),
    wl.LmHeadSpec("lm-300x192-v5000", 300, 192, 5000, 3.0, 15),
    wl.LmHeadSpec("lm-1x1024-v70000", 1, 1024, 70000, 3.0, 16),
]


@pytest.mark.parametrize("spec", SMALL, ids=[s.name for s in SMALL])
def test_small(spec):
    h, w = wl.lm_head_inputs(spec)
    assert check(run(spec, h, w), h, w) > 0.9


def test_full_size_qwen():
    spec = wl.LMHEAD_CONFIGS["qwen"]
    h, w = wl.lm_head_inputs(spec)
    assert check(run(spec, h, w), h, w) > 0.9


def test_full_size_batched_sampled_rows():
    spec = wl.LMHEAD_CONFIGS["batched"]
    h, w = wl.lm_head_inputs(spec)
    rows = np.array(sorted({0, 1, 127, 128, 129, 255, 256, 383, 511, 512, spec.rows - 1}
                           | set(np.random.default_rng(0).choice(spec.rows, 13, replace=False).tolist())))
    assert check(run(spec, h, w), h, w, rows=rows) > 0.9


def test_duplicated_rows_go_to_the_smaller_index():
    spec = wl.LmHeadSpec("lm-ties", 8, 256, 3000, 3.0, 17)
    h, w = wl.lm_head_inputs(spec)
    w = w.clone()
    for r in range(spec.rows):
        v = 100 + 300 * r
        w[v] = (h[r].float() * 0.5).to(torch.bfloat16)        # clearly the largest logit
        w[v + 257] = w[v]                                    # an equal row in a later unit
        w[v + 1] = w[v]                                      # and in the same unit
    lm = run(spec, h, w)
    assert lm.argmax.cpu().tolist() == [100 + 300 * r for r in range(spec.rows)]


def test_deterministic():
    spec = SMALL[4]
    h, w = wl.lm_head_inputs(spec)
    a, b = run(spec, h, w), run(spec, h, w)
    assert torch.equal(a.argmax, b.argmax) and torch.equal(a.max_logit, b.max_logit)
