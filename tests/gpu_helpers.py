"""Shared pieces of the GPU tests: run a workload through the C ABI and
compare with the oracle on the same seeded inputs."""
import numpy as np
import torch

import oracle
from speculative_decoding_tree_gb300 import workloads as wl
from speculative_decoding_tree_gb300.runner import DeviceStep

# attention tolerance (max-abs vs the float64 oracle): 1e-4 on the fp32 path,
# 4e-2 on the bf16 path (the pages' measured BF16 drift, "ADR-037" status
# note and phase row E6 full-layer block: 3.979e-2).
TOL = {"f32": 1e-4, "bf16": 4e-2}


def workload(spec, canary=float("nan")):
    return wl.make_workload(spec, canary=canary, argmax_fn=oracle.argmax_rows)


def run(w, **kw):
    st = DeviceStep(w, **kw)
    st.step()
    torch.cuda.synchronize()
    return st


def sample_pairs(w, n=24, seed=0):
    g = np.random.default_rng(seed)
    R, H = w.total_rows, w.spec.hq
    pairs = {(0, 0), (R - 1, H - 1), (R - 1, 0), (0, H - 1)}
    while len(pairs) < n:
        pairs.add((int(g.integers(0, R)), int(g.integers(0, H))))
    return sorted(pairs)


def check_step(w, st, ref, samples=None):
    """Bit-exact acceptance and commit; attention within tolerance."""
    assert int(st.status[0].item()) == 0, f"device status {int(st.status[0])}"
    # A0: mask bits and depths
    for b in range(w.batch):
        o0, o1 = w.seq_rows(b)
        anc = oracle.ancestors(w.parents[b])
        got = st.anc[o0:o1].cpu().tolist()
        for i, s in enumerate(anc):
            assert (got[i] & ((1 << 64) - 1)) == sum(1 << j for j in s)
        assert st.depth[o0:o1].cpu().tolist() == oracle.depths(w.parents[b])
    # A1+A2: attention
    out = st.out.double().cpu().numpy()
    exp = ref["out"]
    tol = TOL[w.spec.dtype]
    if samples is None:
        err = np.abs(out - exp).max()
    else:
        err = max(np.abs(out[r, h] - exp[r, h]).max() for r, h in samples)
    assert np.isfinite(out).all()
    assert err <= tol, f"attention max-abs error {err} > {tol}"
    # A3: argmax, bit-exact
    assert st.argmax.cpu().numpy().tolist() == ref["argmax"].tolist()
    # A4: walk
    mn = st.desc.max_nodes
    for b, (k, path, tokens) in enumerate(ref["accepted"]):
        assert int(st.accept_len[b]) == k
        assert st.path[b].cpu().tolist() == path + [-1] * (mn - len(path))
        assert st.tokens[b].cpu().tolist() == tokens + [-1] * (mn - len(tokens))
    # A5: commit, byte-exact over the whole cache
    isz = torch.int16 if st.k_cache.dtype == torch.bfloat16 else torch.int32
    assert torch.equal(st.k_cache.cpu().view(isz), ref["k_cache"].view(isz))
    assert torch.equal(st.v_cache.cpu().view(isz), ref["v_cache"].view(isz))
    assert torch.equal(st.prefix_len.cpu(), ref["prefix_len"])
    return err
