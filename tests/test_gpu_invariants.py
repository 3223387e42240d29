"""Invariants of the CUDA path that hold at any size, determinism, the
device status word, and the argmax tie / NaN policy (GPU)."""
import numpy as np
import pytest
import torch

import oracle
import speculative_decoding_tree_gb300 as tv
from speculative_decoding_tree_gb300 import workloads as wl
from speculative_decoding_tree_gb300.runner import DeviceStep
from gpu_helpers import TOL, check_step, run, workload

pytestmark = pytest.mark.gpu


def test_single_node_equals_chain_head():
    # a tree of one node and the first node of a chain see the same keys:
    # the same bytes come out (phase row E1.1: tree=1 is plain decode)
    base = wl.CONFIGS[3].replace(prefix=(333, 333), vocab=100)
    one = workload(base.replace(tree="chain:1"))
    chain = workload(base.replace(tree="chain:5"))
    a = run(one, max_nodes=5)          # same descriptor bound, same launch plan
    b = DeviceStep(chain)
    # same prefix and the same root Q/K/V: copy the single-node inputs in
    b.q[0] = a.q[0]
    b.k_tree[:, 0] = a.k_tree[:, 0]
    b.v_tree[:, 0] = a.v_tree[:, 0]
    b.k_cache[:, :, :333] = a.k_cache[:, :, :333]
    b.v_cache[:, :, :333] = a.v_cache[:, :, :333]
    b.mask()
    b.attn()
    torch.cuda.synchronize()
    assert torch.equal(a.out[0], b.out[0])


def test_determinism_repeated_calls():
    w = workload(wl.small_variant(5))
    outs = []
    for _ in range(3):
        st = DeviceStep(w)
        st.mask()
        for _ in range(5):
            st.attn()
        torch.cuda.synchronize()
        outs.append(st.out.clone())
    for o in outs[1:]:
        assert torch.equal(o.view(torch.int16), outs[0].view(torch.int16))


def test_partials_then_merge_equals_one_call():
    w = workload(wl.small_variant(4))
    a = DeviceStep(w)
    a.mask()
    a.attn()
    b = DeviceStep(w)
    b.mask()
    b.partials()
    b.merge()
    torch.cuda.synchronize()
    assert torch.equal(a.out.view(torch.int16), b.out.view(torch.int16))


def test_nan_canary_beyond_prefix_never_read():
    # every cache row past the prefix holds NaN; outputs must stay finite
    w = workload(wl.small_variant(5), canary=float("nan"))
    st = run(w)
    assert torch.isfinite(st.out.float()).all()


def test_status_bad_tree():
    w = workload(wl.small_variant(1))
    st = DeviceStep(w)
    st.parents[3] = 5            # parent index not below its own
    st.step()
    torch.cuda.synchronize()
    assert int(st.status[0]) & 1


def test_bad_tree_bit_matches_the_oracle_verdict():
    # random batches of trees, some corrupted (self, forward, out-of-range or
    # negative parents, a root with a parent): the mask kernel's bad-tree bit
    # must equal "some tree fails oracle.check_tree", and the ancestor words of
    # every valid tree must still equal the oracle's
    w = workload(wl.small_variant(5, vocab=64))
    st = DeviceStep(w)
    rng = np.random.default_rng(23)
    seen = set()
    for case in range(40):
        trees = []
        for b in range(w.batch):
            par = list(w.parents[b])
            n = len(par)
            if rng.random() < 0.3:
                j = int(rng.integers(0, n))
                par[j] = int(rng.choice([-2, -1, j, min(j + 1, n), n + 5, 0]))
            trees.append(par)
        st.parents.copy_(torch.tensor([x for t in trees for x in t], dtype=torch.int32))
        st.status.zero_()
        st.mask()
        torch.cuda.synchronize()
        want_bad = not all(oracle.check_tree(t) for t in trees)
        assert bool(int(st.status[0]) & 1) == want_bad, (case, trees)
        seen.add(want_bad)
        anc = st.anc.cpu().tolist()
        for b, t in enumerate(trees):
            if oracle.check_tree(t):
                o0, _ = w.seq_rows(b)
                for i, s in enumerate(oracle.ancestors(t)):
                    assert (anc[o0 + i] & ((1 << 64) - 1)) == sum(1 << j for j in s)
    assert seen == {True, False}


def test_status_capacity_leaves_cache():
    spec = wl.CONFIGS[2].replace(prefix=(100, 100), vocab=64, cache_margin=0, p_match=1.0)
    w = workload(spec)
    st = DeviceStep(w, max_prefix=w.capacity)
    before_k = st.k_cache.clone()
    st.prefix_len.fill_(w.capacity - 1)
    st.mask()
    st.accept_commit()
    torch.cuda.synchronize()
    k = int(st.accept_len[0])
    if k + 1 > 1:
        assert int(st.status[0]) & 16
        assert torch.equal(st.k_cache.view(torch.int16), before_k.view(torch.int16))
        assert int(st.prefix_len[0]) == w.capacity - 1


def test_status_bad_page():
    w = workload(wl.small_variant(5, batch=2))
    st = DeviceStep(w)
    st.page_table[0, 0] = 10 ** 6
    st.mask()
    st.attn()
    torch.cuda.synchronize()
    assert int(st.status[0]) & 8
    assert torch.isfinite(st.out.float()).all()


def test_status_bad_prefix():
    w = workload(wl.small_variant(3))
    st = DeviceStep(w)
    st.prefix_len[0] = -5
    st.mask()
    st.attn()
    torch.cuda.synchronize()
    assert int(st.status[0]) & 4


@pytest.mark.parametrize("V", [1, 7, 1000, 4099, 151936])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_argmax_ties_and_nan(V, dtype):
    # values from a tiny set, so maxima tie; sprinkled NaN; one all-NaN row
    g = torch.Generator("cpu").manual_seed(V)
    R = 9
    x = torch.randint(-2, 3, (R, V), generator=g).float()
    x[torch.rand(R, V, generator=g) < 0.05] = float("nan")
    x[4] = float("nan")
    if V > 3:
        x[5, 1] = -0.0
        x[5, 2] = 0.0
        x[5, 3:] = -1.0
        x[5, 0] = float("nan")
    x = x.to(torch.float32 if dtype == "f32" else torch.bfloat16)
    spec = wl.Spec("argmax", 1, 4, 4, 128, "bf16", (4, 4), f"chain:{R}", V, dtype, 1.0, 0.5)
    w = wl.make_workload(spec)
    w.logits = x
    wl.plant_drafts(w, oracle.argmax_rows(x))
    st = DeviceStep(w)
    st.mask()
    st.accept_commit()
    torch.cuda.synchronize()
    assert st.argmax.cpu().tolist() == oracle.argmax_rows(x).tolist()


def test_accept_commit_chain_of_steps():
    # two verify rounds in a row: the second reads the first one's commit
    spec = wl.CONFIGS[2].replace(prefix=(64, 64), vocab=50, p_match=0.9)
    w = workload(spec)
    st = run(w)
    ref = oracle.verify_step(w)
    check_step(w, st, ref)
    w2 = workload(spec)
    w2.k_cache, w2.v_cache, w2.prefix_len = ref["k_cache"], ref["v_cache"], ref["prefix_len"].clone()
    st2 = DeviceStep(w2)
    st2.step()
    torch.cuda.synchronize()
    ref2 = oracle.verify_step(w2)
    check_step(w2, st2, ref2)


@pytest.mark.parametrize("d,nodes,kernel", [(128, 20, 1), (256, 20, 1), (128, 40, 2), (256, 40, 2)])
def test_growing_scores_force_rescale(d, nodes, kernel):
    # prefix keys whose scores grow along the prefix: the running maximum
    # climbs tile after tile, so the tensor-core kernels must rescale O
    spec = wl.CONFIGS[3].replace(prefix=(1500, 1500), vocab=64, d=d, hq=8, hkv=2, tree=f"random:{nodes},{nodes},6",
                                 seed=4242 + d)
    w = workload(spec)
    P = 1500
    ramp = (1.0 + 0.02 * torch.arange(P, dtype=torch.float32)).view(1, 1, P, 1)
    w.k_cache[:, :, :P] = (w.k_cache[:, :, :P].float() * ramp).to(torch.bfloat16)
    st = run(w)
    assert tv.tv_attn_plan(st.desc)["kernel"] == kernel
    check_step(w, st, oracle.verify_step(w))


def test_bounded_wait_runs_out_and_the_context_stays_usable():
    # failure detection without a fault: a wait that nothing completes ends
    # after its limit with TV_DEV_TIMEOUT, and the next calls run normally
    import time
    import speculative_decoding_tree_gb300 as tv
    st = torch.zeros(4, dtype=torch.int32, device="cuda")
    t0 = time.perf_counter()
    tv.tv_check_bounded_wait(20_000_000, st)
    torch.cuda.synchronize()
    assert time.perf_counter() - t0 >= 0.019
    assert int(st[0]) == 32
    w = workload(wl.small_variant(3))
    check_step(w, run(w), oracle.verify_step(w))


@pytest.mark.parametrize("spec", [
    wl.CONFIGS[3].replace(prefix=(2000, 2000), tree="random:48,48,6", vocab=300, p_match=0.9, seed=611,
                          cache_margin=200),
    wl.CONFIGS[5].replace(batch=3, prefix=(700, 2500), vocab=300, p_match=0.9, seed=612, cache_margin=200),
], ids=["pairs-contiguous", "one-cta-paged"])
def test_attention_right_after_commit(spec):
    # accept + commit, then attention over the grown prefix, back to back on
    # one stream (no host sync): the split kernel's prefetches and loads of
    # the committed rows follow the commit kernel directly
    w = workload(spec)
    P0 = w.prefix_len.clone()
    st = DeviceStep(w, max_prefix=int(P0.max()) + 64)
    st.mask()
    st.attn()
    st.accept_commit()
    st.attn()
    torch.cuda.synchronize()
    assert int(st.status[0].item()) == 0
    ref = oracle.verify_step(w)
    assert torch.equal(st.prefix_len.cpu(), ref["prefix_len"])
    w2 = workload(spec)
    w2.k_cache, w2.v_cache, w2.prefix_len = ref["k_cache"], ref["v_cache"], ref["prefix_len"].clone()
    ref2 = oracle.verify_step(w2)
    err = np.abs(st.out.double().cpu().numpy() - ref2["out"]).max()
    assert err <= TOL[w.spec.dtype], err
