"""tree_accept_commit_argmax (GPU): the walk and commit on a caller's argmax,
against the oracle's walk and commit on the same argmax, bit for bit; and the
whole no-logits path: the fused lm_head's argmax fed straight into it."""
import numpy as np
import pytest
import torch

import oracle
from oracle import lm_head
from speculative_decoding_tree_gb300 import workloads as wl
from speculative_decoding_tree_gb300.runner import DeviceLmHead, DeviceStep
from gpu_helpers import workload

pytestmark = pytest.mark.gpu


def check_walk_commit(w, st, am):
    assert int(st.status[0]) == 0
    acc = []
    mn = st.desc.max_nodes
    for b in range(w.batch):
        o0, o1 = w.seq_rows(b)
        k, path, tokens = oracle.accept(w.parents[b], w.draft_tokens[o0:o1].tolist(), am[o0:o1].tolist())
        acc.append((k, path, tokens))
        assert int(st.accept_len[b]) == k
        assert st.path[b].cpu().tolist() == path + [-1] * (mn - len(path))
        assert st.tokens[b].cpu().tolist() == tokens + [-1] * (mn - len(tokens))
    kc, vc, new_p = oracle.commit(w, acc)
    isz = torch.int16 if st.k_cache.dtype == torch.bfloat16 else torch.int32
    assert torch.equal(st.k_cache.cpu().view(isz), kc.view(isz))
    assert torch.equal(st.v_cache.cpu().view(isz), vc.view(isz))
    assert torch.equal(st.prefix_len.cpu(), new_p)


@pytest.mark.parametrize("n", [1, 2, 3, 4, 5])
def test_given_argmax_matches_the_oracle(n):
    w = workload(wl.small_variant(n))
    am = oracle.argmax_rows(w.logits)                      # the drafts were planted against this argmax
    st = DeviceStep(w)
    st.accept_commit_argmax(torch.from_numpy(am).to(torch.int32).cuda())
    torch.cuda.synchronize()
    check_walk_commit(w, st, am)


def test_random_argmax():
    w = workload(wl.small_variant(5))
    g = np.random.default_rng(3)
    am = oracle.argmax_rows(w.logits)
    flip = g.random(am.shape[0]) < 0.3                     # a third of the rows disagree with the drafts
    am = np.where(flip, g.integers(0, w.spec.vocab, am.shape[0]), am)
    st = DeviceStep(w)
    st.accept_commit_argmax(torch.from_numpy(am).to(torch.int32).cuda())
    torch.cuda.synchronize()
    check_walk_commit(w, st, am)


def test_lm_head_argmax_feeds_the_walk():
    # hidden rows of the workload's tree rows through a random lm_head; the
    # drafts are planted against the oracle's argmax of those logits, so the
    # walk accepts deep paths only when the kernel's argmax agrees
    spec = wl.small_variant(3)
    w0 = workload(spec)
    R = w0.total_rows
    lspec = wl.LmHeadSpec("walk-lmhead", R, 512, spec.vocab, 3.0, 91)
    h, wt = wl.lm_head_inputs(lspec)
    am_ref, _, gap = lm_head.lm_head_argmax(h, wt)
    assert (gap > 4e-3).all()                              # no near ties in this fixture
    w = wl.make_workload(spec, argmax_fn=lambda logits: torch.from_numpy(am_ref))
    lm = DeviceLmHead(lspec, hidden=h, weight=wt)
    lm.run()
    st = DeviceStep(w)
    st.accept_commit_argmax(lm.argmax)
    torch.cuda.synchronize()
    assert int(lm.status[0]) == 0
    assert np.array_equal(lm.argmax.cpu().numpy(), am_ref)
    check_walk_commit(w, st, am_ref)


# Shapes of the walk's cluster (one block per (K or V, KV head) set, at most 8
# blocks, extra sets shared round-robin) and of its two commit sources: tree
# rows staged in shared memory when a block's sets fit the 160 KB budget,
# else read from the tree buffers.
@pytest.mark.parametrize("hq,hkv,d,dtype,paged", [
    (3, 1, 256, "bf16", False),    # a cluster of 2 blocks
    (6, 3, 128, "bf16", True),     # 6 blocks, paged cache
    (10, 5, 128, "bf16", False),   # 8 blocks, blocks 0 and 1 hold two sets
    (10, 5, 512, "f32", False),    # two 2 KB-row sets per block: copied from the tree buffers
])
def test_walk_cluster_shapes(hq, hkv, d, dtype, paged):
    spec = wl.small_variant(5, hq=hq, hkv=hkv, d=d, dtype=dtype, logit_dtype=dtype, paged=paged, batch=3,
                            prefix=(40, 300), vocab=2003, seed=77 + hkv + d)
    w = workload(spec)
    sets_per_block = -(-2 * hkv // min(8, 2 * hkv))
    staged = sets_per_block * w.max_nodes * d * (2 if dtype == "bf16" else 4) <= 160 * 1024
    assert staged == (d != 512)                            # each commit source is covered
    am = oracle.argmax_rows(w.logits)
    st = DeviceStep(w)
    st.accept_commit()                                     # the argmax pass, then the walk
    torch.cuda.synchronize()
    assert np.array_equal(st.argmax.cpu().numpy(), am)
    check_walk_commit(w, st, am)
    st = DeviceStep(w)
    st.accept_commit_argmax(torch.from_numpy(am).to(torch.int32).cuda())
    torch.cuda.synchronize()
    check_walk_commit(w, st, am)
