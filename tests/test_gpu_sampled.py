"""Sampled verification on the GPU vs the oracle (GPU).

The draw is decided in float32 on the GPU and in float64 in the oracle from
the same Philox words.  Where the oracle's two largest perturbed values are
further apart than float32 noise the draws must be equal, so the parity
tests use offsets at which the oracle finds no row closer than that (the
offset is chosen from the oracle alone) and then compare every draw, the
walk, the emitted tokens and the committed cache with the oracle's own step
bit for bit.  Near ties are checked separately for validity: the GPU's draw
must then be (within the noise) a maximum.  A statistical test checks the
draws follow softmax(logits / T)."""
import numpy as np
import pytest
import torch

import oracle
from oracle import sampled
from speculative_decoding_tree_gb300 import workloads as wl
from speculative_decoding_tree_gb300.runner import DeviceStep
from gpu_helpers import workload

pytestmark = pytest.mark.gpu

NOISE = 1e-3      # float32 rounding of logit / T + G is far below this for these logits


def run_sampled(w, t, seed, offset, **kw):
    st = DeviceStep(w, **kw)
    st.mask()
    st.attn()
    st.accept_commit_sampled(t, seed, offset)
    torch.cuda.synchronize()
    return st


def oracle_draws(w, t, seed, offset):
    x = w.logits.double().numpy()
    out = [sampled.draw_with_margin(x[r], t, r, seed, offset) for r in range(w.total_rows)]
    return np.array([y for y, _ in out], dtype=np.int64), np.array([m for _, m in out])


def clear_offset(w, t, seed, start=0, tries=40):
    """First offset >= start at which no row of the oracle's draws is a near tie."""
    for off in range(start, start + tries):
        y, margin = oracle_draws(w, t, seed, off)
        if (margin > NOISE).all():
            return off, y
    raise AssertionError("every offset tried has a near tie")


def check_sampled(w, st, y_ref):
    """The whole step against the oracle's own draws, walk and commit."""
    assert int(st.status[0].item()) == 0
    y = st.argmax.cpu().numpy().astype(np.int64)
    assert np.array_equal(y, y_ref), np.flatnonzero(y != y_ref)
    acc = []
    mn = st.desc.max_nodes
    for b in range(w.batch):
        o0, o1 = w.seq_rows(b)
        k, path, tokens = oracle.accept(w.parents[b], w.draft_tokens[o0:o1].tolist(), y_ref[o0:o1].tolist())
        acc.append((k, path, tokens))
        assert int(st.accept_len[b]) == k
        assert st.path[b].cpu().tolist() == path + [-1] * (mn - len(path))
        assert st.tokens[b].cpu().tolist() == tokens + [-1] * (mn - len(tokens))
    kc, vc, new_p = oracle.commit(w, acc)
    isz = torch.int16 if st.k_cache.dtype == torch.bfloat16 else torch.int32
    assert torch.equal(st.k_cache.cpu().view(isz), kc.view(isz))
    assert torch.equal(st.v_cache.cpu().view(isz), vc.view(isz))
    assert torch.equal(st.prefix_len.cpu(), new_p)


def sampled_case(w, t, seed, start):
    off, y_ref = clear_offset(w, t, seed, start)
    check_sampled(w, run_sampled(w, t, seed, off), y_ref)


@pytest.mark.parametrize("n", [1, 2, 3, 4, 5])
@pytest.mark.parametrize("t", [0.7, 1.0, 1.6])
def test_small_variants(n, t):
    sampled_case(workload(wl.small_variant(n)), t, seed=2024 + n, start=17)


@pytest.mark.parametrize("n", [3, 4, 5])
def test_full_sizes(n):
    sampled_case(workload(wl.CONFIGS[n]), 1.0, seed=99, start=n)


def test_near_ties_draw_a_maximum():
    # a row whose two largest perturbed values are within float32 noise may
    # go either way; the GPU's draw must be one of the (near) maxima
    w = workload(wl.small_variant(5))
    x = w.logits.double().numpy()
    found = 0
    for off in range(60):
        y_ref, margin = oracle_draws(w, 1.0, 77, off)
        close = np.flatnonzero(margin <= NOISE)
        if close.size == 0:
            continue
        y = run_sampled(w, 1.0, 77, off).argmax.cpu().numpy()
        for r in close:
            s = sampled.perturbed(x[r], 1.0, int(r), 77, off)
            assert s[y[r]] >= np.nanmax(s) - NOISE, (off, r)
        far = margin > NOISE
        assert np.array_equal(y[far], y_ref[far])
        found += 1
        if found == 3:
            break
    assert found >= 1


def test_seed_and_offset_change_the_draws_deterministically():
    w = workload(wl.small_variant(3))
    a = run_sampled(w, 1.0, seed=5, offset=1).argmax.cpu()
    b = run_sampled(w, 1.0, seed=5, offset=1).argmax.cpu()
    c = run_sampled(w, 1.0, seed=5, offset=2).argmax.cpu()
    d = run_sampled(w, 1.0, seed=6, offset=1).argmax.cpu()
    assert torch.equal(a, b)
    assert not torch.equal(a, c) and not torch.equal(a, d)


def test_draws_follow_softmax():
    from scipy.stats import chi2
    spec = wl.CONFIGS[3].replace(prefix=(16, 16), vocab=24, tree="chain:1", logit_std=1.5, seed=31)
    w = workload(spec)
    st = DeviceStep(w)
    p0 = st.prefix_len.clone()
    t = 0.8
    counts = np.zeros(24)
    n = 3000
    for off in range(n):
        st.prefix_len.copy_(p0)
        st.accept_commit_sampled(t, 4321, off)
        counts[int(st.argmax[0].item())] += 1
    z = w.logits[0].double().numpy() / t
    p = np.exp(z - z.max())
    p /= p.sum()
    exp = p * n
    keep = exp >= 5
    c = np.append(counts[keep], counts[~keep].sum())
    e = np.append(exp[keep], exp[~keep].sum())
    stat = ((c - e) ** 2 / e).sum()
    assert chi2.sf(stat, len(e) - 1) > 1e-4, counts


def test_nan_logits_never_drawn():
    w = workload(wl.small_variant(2))
    x = w.logits.clone()
    x[:, ::3] = float("nan")
    w.logits = x
    st = run_sampled(w, 1.0, seed=8, offset=8)
    y = st.argmax.cpu().numpy()
    assert (y % 3 != 0).all()


def test_infinite_logits():
    # +inf wins whatever the noise (first index among several); a row of
    # -inf and NaN gives the first -inf entry, as the greedy rule does
    w = workload(wl.small_variant(2))
    x = w.logits.clone()
    x[0, 7] = float("inf")
    x[0, 3] = float("inf")
    x[1, :] = float("-inf")
    x[1, ::2] = float("nan")
    w.logits = x
    st = run_sampled(w, 1.0, seed=4, offset=4)
    y = st.argmax.cpu().numpy()
    assert y[0] == 3
    assert y[1] == 1
