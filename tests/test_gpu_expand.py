"""Dynamic draft-tree expansion on the GPU vs the oracle (GPU).

Tokens, parents, depths, node counts and the order nodes enter the tree are
compared exactly; cumulative log-probabilities within CUM_TOL.  The kernel's
log-sum-exp differs from the oracle's float64 one by rounding (float32 sums of
float32 exponentials within a warp), so every workload used here is checked
first, by the oracle alone, to make no decision between two candidates whose
values differ by less than DECIDE (a gap of exactly 0 is a tie between
siblings with equal logits, which both sides compute from identical numbers
and break by generation order)."""
import numpy as np
import pytest
import torch

from oracle import ancestors, expand
from speculative_decoding_tree_gb300 import tv_build_tree_mask, make_desc, BF16
from speculative_decoding_tree_gb300 import workloads as wl
from speculative_decoding_tree_gb300.runner import DeviceExpand

pytestmark = pytest.mark.gpu

CUM_TOL = 1e-5      # per-step lse rounding (~1e-7 to 2e-6) times the depth
DECIDE = 2e-5


def oracle_trees(spec, rows, token_map=None):
    out = []
    roots = wl.root_tokens(spec)
    for b in range(spec.batch):
        def logits_of(step, j, path, b=b):
            return rows[step][b, j]
        out.append(expand.expand_tree(logits_of, int(roots[b]), spec.top_k, spec.max_nodes, spec.width,
                                      spec.max_depth, token_map))
    return out


def run(spec, rows=None, token_map=None, steps=None):
    if rows is None:
        n = steps if steps is not None else None
        dx = DeviceExpand(spec, token_map=token_map, steps=n)
    else:
        dx = DeviceExpand(spec, rows=rows, token_map=token_map, steps=len(rows))
    dx.run()
    torch.cuda.synchronize()
    return dx


def check(spec, dx, refs, status=0):
    assert int(dx.status[0].item()) == status, int(dx.status[0].item())
    N = spec.max_nodes
    for b, t in enumerate(refs):
        g = np.asarray(t["gaps"])
        assert not ((g > 0) & (g < DECIDE)).any(), f"tree {b}: the oracle decides a near tie"
        n = len(t["tokens"])
        assert int(dx.n_nodes[b]) == n
        assert int(dx.expand_count[b]) == 0
        assert dx.tokens[b].cpu().tolist() == t["tokens"] + [-1] * (N - n)
        assert dx.parents[b].cpu().tolist() == t["parents"] + [-1] * (N - n)
        assert dx.depths[b].cpu().tolist() == t["depths"] + [-1] * (N - n)
        c = dx.cum[b].cpu().numpy()
        ref = np.asarray(t["cum"])
        fin = np.isfinite(ref)
        assert np.array_equal(np.isfinite(c[:n]), fin)
        assert np.abs(c[:n][fin] - ref[fin]).max() <= CUM_TOL
        assert np.isneginf(c[n:]).all()


def all_rows(spec, steps):
    return [wl.draft_rows(spec, s) for s in range(steps)]


SMALL = {
    "best-first": wl.ExpandSpec("x-w1", 1, 1000, 4, 1, 20, 5, "f32", 2.0, 11),
    "w3-f32": wl.ExpandSpec("x-w3", 3, 5003, 8, 3, 33, 4, "f32", 2.5, 12),
    "w16-k16-odd-vocab": wl.ExpandSpec("x-w16", 2, 777, 16, 16, 64, 10, "bf16", 3.0, 13),
    "chain-k1": wl.ExpandSpec("x-k1", 2, 300, 1, 4, 12, 20, "bf16", 1.0, 14),
    "depth-1": wl.ExpandSpec("x-d1", 2, 300, 5, 2, 30, 1, "f32", 1.0, 15),
    "budget-1": wl.ExpandSpec("x-n1", 2, 300, 5, 2, 1, 3, "f32", 1.0, 16),
    "k-above-vocab-rows": wl.ExpandSpec("x-kv", 1, 6, 8, 8, 40, 3, "f32", 1.0, 17),
    "batch-5-bf16": wl.ExpandSpec("x-b5", 5, 20011, 8, 8, 64, 6, "bf16", 3.0, 18),
}


@pytest.mark.parametrize("name", list(SMALL))
def test_small(name):
    spec = SMALL[name]
    steps = spec.max_nodes + 1          # enough steps even when the depth limit slows growth
    rows = all_rows(spec, steps)
    check(spec, run(spec, rows=rows), oracle_trees(spec, rows))


@pytest.mark.parametrize("name", list(wl.EXPAND_CONFIGS))
def test_full_size(name):
    spec = wl.EXPAND_CONFIGS[name]
    dx = run(spec)                      # the steps the benchmark runs
    rows = all_rows(spec, dx.steps)
    check(spec, dx, oracle_trees(spec, rows))


def test_steps_query_fills_unlimited_trees():
    # with no binding depth limit, tv_expand_steps steps fill every tree
    spec = SMALL["w3-f32"].replace(max_depth=64)
    dx = run(spec)
    assert (dx.n_nodes.cpu() == spec.max_nodes).all()
    check(spec, dx, oracle_trees(spec, all_rows(spec, dx.steps)))


def test_token_map():
    spec = SMALL["w3-f32"]
    g = torch.Generator().manual_seed(5)
    tmap = torch.randperm(10 * spec.vocab, generator=g)[:spec.vocab].to(torch.int32)
    rows = all_rows(spec, spec.max_nodes + 1)
    check(spec, run(spec, rows=rows, token_map=tmap), oracle_trees(spec, rows, token_map=tmap.numpy()))


def test_ties_go_to_smaller_tokens_and_first_generated():
    # every logit equal: each node's children are tokens 0..K-1 with equal
    # log-probabilities, so the tree fills in generation order
    spec = wl.ExpandSpec("x-ties", 2, 64, 3, 2, 15, 5, "bf16", 1.0, 19)
    rows = [torch.zeros_like(r) for r in all_rows(spec, spec.max_nodes + 1)]
    dx = run(spec, rows=rows)
    refs = oracle_trees(spec, rows)
    check(spec, dx, refs)
    assert refs[0]["tokens"][1:4] == [0, 1, 2]


@pytest.mark.parametrize("V,dtype", [(5000, "bf16"), (9000, "f32")])
def test_rows_of_equal_logits(V, dtype):
    # a whole chunk of equal logits (more candidates than one CTA ranks
    # directly): the smaller tokens still win, in order
    spec = wl.ExpandSpec("x-flat", 2, V, 16, 4, 30, 4, dtype, 1.0, 21)
    rows = [torch.full_like(r, 0.5) for r in all_rows(spec, spec.max_nodes + 1)]
    rows[1][1, 2, 4100:4108] = 0.75          # a few larger entries in the second chunk
    dx = run(spec, rows=rows)
    refs = oracle_trees(spec, rows)
    check(spec, dx, refs)
    assert refs[0]["tokens"][1:17] == list(range(16))


def test_nan_entries_never_chosen_and_empty_rows():
    spec = SMALL["batch-5-bf16"].replace(vocab=3001, max_nodes=40)
    rows = all_rows(spec, spec.max_nodes + 1)
    for s, r in enumerate(rows):
        r[:, :, ::3] = float("nan")
        if s == 1:
            r[0, 2, :] = float("nan")            # a node with no valid token: no children
        if s == 2:
            r[1, 0, 5:] = float("-inf")          # -inf entries are valid children of zero probability
    check(spec, run(spec, rows=rows), oracle_trees(spec, rows))


def test_plus_inf_row_flags_and_skips_the_node():
    spec = SMALL["w3-f32"]
    rows = all_rows(spec, spec.max_nodes + 1)
    rows[1][2, 1, 17] = float("inf")
    dx = run(spec, rows=rows)
    refs = oracle_trees(spec, rows)              # the oracle on the kernel's own input
    assert [t["bad_logits"] for t in refs] == [False, False, True]
    check(spec, dx, refs, status=64)


def test_out_of_order_step_is_refused():
    spec = SMALL["w3-f32"]
    dx = DeviceExpand(spec, steps=4)
    dx.step(0)
    dx.step(2)                                   # skips step 1
    torch.cuda.synchronize()
    assert int(dx.status[0]) == 128
    assert (dx.n_nodes.cpu() == min(spec.width, spec.top_k) + 1).all()


def test_deterministic():
    spec = wl.EXPAND_CONFIGS["eagle2"]
    a, b = run(spec), run(spec)
    for name in ("tokens", "parents", "depths", "cum", "n_nodes"):
        assert torch.equal(getattr(a, name), getattr(b, name))


def test_expanded_tree_feeds_the_mask():
    # the expansion's parents go straight into tv_build_tree_mask
    spec = wl.EXPAND_CONFIGS["batched"].replace(vocab=4099)
    dx = run(spec)
    B, N = spec.batch, spec.max_nodes
    assert (dx.n_nodes.cpu() == N).all()
    desc = make_desc(batch=B, num_q_heads=8, num_kv_heads=8, head_dim=128, dtype=BF16, max_nodes=N,
                     total_rows=B * N, capacity=256, max_prefix=128)
    offs = (torch.arange(B + 1, dtype=torch.int32) * N).cuda()
    anc = torch.zeros(B * N, dtype=torch.int64, device="cuda")
    depth = torch.zeros(B * N, dtype=torch.int32, device="cuda")
    st = torch.zeros(4, dtype=torch.int32, device="cuda")
    tv_build_tree_mask(desc, dx.parents.reshape(-1), offs, anc, depth, st)
    torch.cuda.synchronize()
    assert int(st[0]) == 0
    assert torch.equal(depth.reshape(B, N), dx.depths)
    par = dx.parents.cpu()
    for b in range(B):
        ref = ancestors(par[b].tolist())
        got = anc[b * N:(b + 1) * N].cpu().tolist()
        for i in range(N):
            assert (got[i] & ((1 << 64) - 1)) == sum(1 << j for j in ref[i])
