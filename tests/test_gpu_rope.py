"""Tree-position RoPE and K/V scatter on the GPU vs the oracle (GPU).

The kernel rotates in float32 (angles reduced in float64) and rounds to the
output dtype; the oracle rotates in float64.  bf16 outputs must be within one
bf16 unit in the last place of the oracle's value, fp32 outputs within 1e-5
relative; the value heads are copied bit for bit."""
import numpy as np
import pytest
import torch

from oracle import rope
from speculative_decoding_tree_gb300 import tv_build_tree_mask, tv_tree_rope_scatter
from speculative_decoding_tree_gb300 import workloads as wl
from speculative_decoding_tree_gb300.runner import DeviceStep
from gpu_helpers import workload

pytestmark = pytest.mark.gpu


def run_rope(spec, theta, in_place=False, seed=0):
    w = workload(spec)
    st = DeviceStep(w)
    st.mask()                                     # depths
    R, Hq, Hkv, d = w.total_rows, spec.hq, spec.hkv, spec.d
    g = torch.Generator().manual_seed(seed)
    dt = w.q.dtype
    q = torch.randn(R, Hq, d, generator=g).to(dt)
    k = torch.randn(R, Hkv, d, generator=g).to(dt)
    v = torch.randn(R, Hkv, d, generator=g).to(dt)
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    qo = qd if in_place else torch.empty_like(qd)
    kt = torch.empty(Hkv, R, d, dtype=dt, device="cuda")
    vt = torch.empty(Hkv, R, d, dtype=dt, device="cuda")
    tv_tree_rope_scatter(st.desc, theta, qd, kd, vd, st.prefix_len, st.node_offsets, st.depth, qo, kt, vt, st.status)
    torch.cuda.synchronize()
    assert int(st.status[0]) == 0
    ref = rope.tree_rope_scatter(q, k, v, w.prefix_len.numpy(), w.node_offsets.numpy(), w.parents_flat.numpy(), theta)
    return (qo.cpu(), kt.cpu(), vt.cpu()), ref, v


def close(got, ref, dt):
    g = got.double().numpy()
    if dt == torch.bfloat16:
        ulp = np.exp2(np.floor(np.log2(np.maximum(np.abs(ref), 1e-30))) - 7)
        return np.all(np.abs(g - ref) <= ulp + 1e-6)
    return np.all(np.abs(g - ref) <= 1e-5 * np.abs(ref) + 1e-6)


@pytest.mark.parametrize("n", [1, 2, 3, 4, 5])
@pytest.mark.parametrize("theta", [1e4, 1e6])
def test_small_variants(n, theta):
    spec = wl.small_variant(n)
    (qo, kt, vt), (qr, kr, vr), v = run_rope(spec, theta, seed=n)
    dt = qo.dtype
    assert close(qo, qr, dt) and close(kt, kr, dt)
    assert torch.equal(vt, v.transpose(0, 1).contiguous())


@pytest.mark.parametrize("n", [3, 4, 5])
def test_full_sizes(n):
    # the largest positions: 32K prefixes plus depths, and the batched workload's 16 sequences
    (qo, kt, vt), (qr, kr, vr), v = run_rope(wl.CONFIGS[n], 1e6, seed=10 + n)
    assert close(qo, qr, qo.dtype) and close(kt, kr, qo.dtype)
    assert torch.equal(vt, v.transpose(0, 1).contiguous())


def test_in_place_queries():
    spec = wl.small_variant(3)
    (qo, kt, _), (qr, kr, _), _ = run_rope(spec, 1e4, in_place=True, seed=7)
    assert close(qo, qr, qo.dtype) and close(kt, kr, qo.dtype)
