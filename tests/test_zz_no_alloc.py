"""tree_verify_attn_noalloc: attention for callers that cannot allocate
device memory (a plugin that a host framework hands only its input and
output buffers, or a loop that must not call cudaMalloc because it may
synchronise the device).  It keeps its split-KV partials in the library's
static device array instead of a workspace.

Checked through the C ABI against tree_verify_attn with a torch-allocated
workspace, on two calls in a row (the second sees the first call's leftover
scratch).  Both calls run the same launch plan and kernels, and results are
deterministic, so the outputs must be equal bit for bit.  This file is
collected last so that a failure here stops a -x run only after every other
test has run."""
import ctypes

import pytest
import torch

import speculative_decoding_tree_gb300 as tv
from speculative_decoding_tree_gb300 import _build
from speculative_decoding_tree_gb300 import workloads as wl
from speculative_decoding_tree_gb300.runner import DeviceStep
from gpu_helpers import workload

pytestmark = pytest.mark.gpu


def _noalloc():
    _build.build()
    fn = tv.lib().tree_verify_attn_noalloc
    fn.argtypes = [ctypes.POINTER(tv.TvDesc)] + [ctypes.c_void_p] * 12
    fn.restype = ctypes.c_int
    return fn


def _call(fn, st, out):
    p = lambda t: None if t is None else t.data_ptr()
    return fn(ctypes.byref(st.desc), p(st.q), p(st.k_cache), p(st.v_cache), p(st.page_table), p(st.prefix_len),
              p(st.node_offsets), p(st.k_tree), p(st.v_tree), p(st.anc), p(out), p(st.status),
              torch.cuda.current_stream().cuda_stream)


def _bits(t):
    return t.view(torch.int16 if t.dtype == torch.bfloat16 else torch.int32)


@pytest.mark.parametrize("spec", [wl.small_variant(1), wl.small_variant(3), wl.small_variant(5), wl.CONFIGS[4]],
                         ids=["tiny-f32", "eagle2-small", "batched-small", "long-full"])
def test_noalloc_matches_workspace_call(spec):
    fn = _noalloc()
    w = workload(spec)
    st = DeviceStep(w)
    # the plan's partials fit the static array (the long-context workload,
    # 19 splits of CTA-pair tiles, is the largest single-sequence case)
    assert tv.tv_workspace_size(st.desc, 0) <= 32 << 20
    st.mask()
    st.attn()                        # existing entry point, torch-allocated workspace
    torch.cuda.synchronize()
    assert int(st.status[0]) == 0
    ref = st.out.clone()
    for _ in range(2):
        out = torch.full_like(ref, float("nan"))
        assert _call(fn, st, out) == 0
        torch.cuda.synchronize()
        assert int(st.status[0]) == 0
        assert torch.equal(_bits(out), _bits(ref))


def test_noalloc_rejects_oversized_problem():
    fn = _noalloc()
    w = workload(wl.small_variant(3))
    st = DeviceStep(w)
    big = tv.make_desc(batch=64, num_q_heads=64, num_kv_heads=8, head_dim=512, dtype=tv.BF16, max_nodes=64,
                       total_rows=4096, capacity=8192, max_prefix=8000)
    assert tv.tv_workspace_size(big, 0) > 32 << 20
    st.desc = big
    assert _call(fn, st, st.out) == -10          # TV_ERR_WORKSPACE, nothing enqueued
