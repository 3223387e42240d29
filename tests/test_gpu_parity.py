"""CUDA path vs the oracle on the five verify workloads (GPU).

Small variants compare every attention output; full sizes compare sampled
(row, head) outputs the oracle computes one by one, and everything of the
acceptance and the commit bit for bit.  The full sizes run in the launch
configuration the benchmark times (same descriptor, same plan)."""
import numpy as np
import pytest
import torch

import oracle
from speculative_decoding_tree_gb300 import workloads as wl
from gpu_helpers import check_step, run, sample_pairs, workload

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("n", [1, 2, 3, 4, 5])
def test_small_variant(n):
    w = workload(wl.small_variant(n))
    st = run(w)
    ref = oracle.verify_step(w)
    check_step(w, st, ref)


@pytest.mark.parametrize("n", [1, 2, 3, 4, 5])
def test_full_size(n):
    w = workload(wl.CONFIGS[n])
    st = run(w)
    samples = None if n <= 2 else sample_pairs(w, 24, seed=n)
    ref = oracle.verify_step(w, samples=samples)
    check_step(w, st, ref, samples)


@pytest.mark.parametrize("P", [0, 1, 31, 32, 33, 63, 64, 65, 127, 128, 129, 255, 1000])
def test_ragged_prefixes(P):
    # prefix lengths across key-tile and chunk boundaries, with a 13-node tree
    spec = wl.CONFIGS[3].replace(prefix=(P, P), vocab=300, tree="random:13,13,5", seed=77 + P)
    w = workload(spec)
    check_step(w, run(w), oracle.verify_step(w))


@pytest.mark.parametrize("n_nodes", [1, 2, 17, 33, 64])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_tree_sizes(n_nodes, dtype):
    spec = wl.CONFIGS[4].replace(prefix=(200, 200), vocab=257, tree=f"random:{n_nodes},{n_nodes},8",
                                 dtype=dtype, logit_dtype=dtype, seed=300 + n_nodes)
    w = workload(spec)
    check_step(w, run(w), oracle.verify_step(w))


@pytest.mark.parametrize("d,hq,hkv", [(128, 8, 8), (128, 16, 2), (256, 12, 4), (512, 8, 1), (256, 4, 4)])
def test_head_shapes(d, hq, hkv):
    spec = wl.CONFIGS[5].replace(batch=3, hq=hq, hkv=hkv, d=d, prefix=(5, 300), vocab=1031, seed=900 + d + hq)
    w = workload(spec)
    check_step(w, run(w), oracle.verify_step(w))


def test_bf16_out_f32():
    w = workload(wl.small_variant(3))
    st = run(w, out_f32=True)
    assert st.out.dtype == torch.float32
    check_step(w, st, oracle.verify_step(w))


@pytest.mark.parametrize("P", [1, 512, 513, 1024, 3584, 3585, 3968, 3969, 4096])
def test_tree_split_rule(P):
    # one plan (one wave) for prefixes up to 4096; the device
    # prefix decides per sequence whether the tree joins the last chunk or
    # gets a split of its own, and how many splits the merge combines
    spec = wl.CONFIGS[3].replace(prefix=(P, P), vocab=300, tree="random:13,13,5", seed=500 + P,
                                 cache_margin=4200 - P)
    w = workload(spec)
    check_step(w, run(w, max_prefix=4096), oracle.verify_step(w))


def test_merge_in_batches():
    # one KV head, head_dim 512: more splits than one merge batch holds in
    # shared memory, so the merge keeps a running maximum across batches
    spec = wl.CONFIGS[2].replace(hq=8, hkv=1, prefix=(20000, 20000), vocab=300, seed=4242)
    w = workload(spec)
    st = run(w)
    from speculative_decoding_tree_gb300 import tv_attn_plan
    assert tv_attn_plan(st.desc)["num_splits"] > 24
    check_step(w, st, oracle.verify_step(w))


@pytest.mark.parametrize("batch,seed", [(4, 61), (6, 62)])
def test_batched_multi_chunk_every_element(batch, seed):
    # ragged paged batches whose prefixes span several key chunks (4096 to
    # 8192 keys) with random 16-64-node trees: every (row, head) output is
    # compared with the oracle, at a vocabulary small enough for the oracle
    spec = wl.CONFIGS[5].replace(batch=batch, prefix=(4096, 8192), vocab=2053, seed=seed)
    w = workload(spec)
    st = run(w)
    from speculative_decoding_tree_gb300 import tv_attn_plan
    assert tv_attn_plan(st.desc)["num_splits"] >= 3
    check_step(w, st, oracle.verify_step(w))


@pytest.mark.parametrize("paged,hq,seed", [(True, 40, 63), (False, 40, 64), (False, 32, 65)])
def test_batched_row_tile_pairs(paged, hq, seed):
    # the batch kernel computes a unit's row tiles in pairs: trees of 1 to 64
    # nodes at GQA 5 (125-row tiles, 1 to 3 per KV head) leave some pairs
    # with one live tile, or none past the last; GQA 4 gives 1 or 2 tiles.
    # Contiguous caches load 64-key halves, paged ones four pages per CTA,
    # across several key chunks
    spec = wl.CONFIGS[5].replace(batch=5, hq=hq, prefix=(1, 4500), tree="random:1,64,8", paged=paged,
                                 vocab=1031, seed=seed)
    w = workload(spec)
    st = run(w)
    from speculative_decoding_tree_gb300 import tv_attn_plan
    plan = tv_attn_plan(st.desc)
    assert plan["kernel"] == 3 and plan["grid_ctas"] % 2 == 0
    check_step(w, st, oracle.verify_step(w))
