"""The C-ABI library loads, exports every symbol the headers under include/
declare, and rejects bad arguments on the host before any launch.  CPU only:
no call here reaches a kernel."""
import ctypes
import os
import re

import pytest

import speculative_decoding_tree_gb300 as tv
from speculative_decoding_tree_gb300 import _build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
INCLUDE = os.path.join(ROOT, "include")


@pytest.fixture(scope="module")
def L():
    _build.build()
    return tv.lib()


def declared_functions():
    text = ""
    for f in sorted(os.listdir(INCLUDE)):
        if f.endswith(".h"):
            with open(os.path.join(INCLUDE, f)) as fh:
                text += fh.read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?(?:int|size_t|char\s*\*|void)\s*\**\s*(\w+)\s*\(", text,
                                 flags=re.M)))


def test_exports_every_declared_symbol(L):
    names = declared_functions()
    assert {"tree_verify_attn", "tree_accept_commit", "tv_build_tree_mask", "tv_workspace_size",
            "tv_tree_expand_step", "tv_expand_steps", "tv_expand_workspace_size"} <= set(names)
    for n in names:
        assert hasattr(L, n), n


def test_codes_have_names(L):
    for code in range(0, -13, -1):
        assert tv.tv_status_string(code) != "unknown"
    for bit in (1, 2, 4, 8, 16, 32, 64, 128):
        assert tv.tv_status_string(bit).startswith("device:")
    assert tv.tv_status_string(12345) == "unknown"
    assert "sm_103a" in tv.tv_version()


def _desc(**kw):
    base = dict(batch=1, num_q_heads=32, num_kv_heads=8, head_dim=256, dtype=tv.BF16, max_nodes=64,
                total_rows=64, capacity=4176, max_prefix=4096)
    base.update(kw)
    return tv.make_desc(**base)


@pytest.mark.parametrize("kw,code", [
    (dict(num_kv_heads=0), -4), (dict(num_q_heads=0), -4), (dict(num_q_heads=30), -5),
    (dict(head_dim=64), -3), (dict(dtype=7), -2), (dict(max_nodes=65, total_rows=65), -7),
    (dict(total_rows=65), -7), (dict(batch=0), -6), (dict(max_prefix=5000), -6),
    (dict(page_size=8), -8), (dict(page_size=16, num_pages=0), -8), (dict(page_size=16, capacity=4177), -8),
    (dict(capacity=2 ** 62, max_prefix=4096), -9), (dict(scale=float("nan")), -6),
])
def test_descriptor_validation(L, kw, code):
    d = _desc(**kw)
    n = ctypes.c_size_t(0)
    assert L.tv_workspace_size(ctypes.byref(d), 1000, ctypes.byref(n)) == code
    # the same code from the launch entry points, which return before launching
    fake = 1 << 20
    rc = L.tree_verify_attn(ctypes.byref(d), *([fake] * 10), fake, 1 << 30, fake, None)
    assert rc == code


def test_grid_limits_refused_on_the_host(L):
    # launch grids keep sequences on z and (KV head, split) on y: extents
    # above 65535 are refused before any launch, not by the driver
    n = ctypes.c_size_t(0)
    fake = 1 << 20
    big_batch = _desc(batch=70000, total_rows=70000, max_nodes=1, capacity=64, max_prefix=64)
    assert L.tv_workspace_size(ctypes.byref(big_batch), 0, ctypes.byref(n)) == -6
    assert L.tree_verify_attn(ctypes.byref(big_batch), *([fake] * 10), fake, 1 << 30, fake, None) == -6
    # 64 KV heads x 1100 chunks of the batch chunk (1920 keys) on the one-CTA
    # tensor-core kernel (16 rows per KV head; an fp32 output keeps the batch
    # off the persistent kernel): 64 x 1100 (KV head, split) pairs exceed the
    # grid's y limit, 64 x 1000 do not
    many_splits = _desc(batch=2, num_q_heads=256, num_kv_heads=64, head_dim=128, max_nodes=4, total_rows=8,
                        capacity=1920 * 1100, max_prefix=1920 * 1100, out_f32=1)
    assert tv.tv_attn_plan(_desc(batch=2, num_q_heads=256, num_kv_heads=64, head_dim=128, max_nodes=4,
                                 total_rows=8, capacity=1920 * 1000, max_prefix=1920 * 1000,
                                 out_f32=1))["kernel"] == 1
    assert L.tv_workspace_size(ctypes.byref(many_splits), 0, ctypes.byref(n)) == -6
    ok_splits = _desc(batch=2, num_q_heads=256, num_kv_heads=64, head_dim=128, max_nodes=4, total_rows=8,
                      capacity=1920 * 1000, max_prefix=1920 * 1000, out_f32=1)
    assert tv.tv_attn_plan(ok_splits)["chunk"] == 1920 and tv.tv_attn_plan(ok_splits)["num_splits"] == 1000
    assert L.tv_workspace_size(ctypes.byref(ok_splits), 0, ctypes.byref(n)) == 0
    # the persistent batch kernel (bf16 output) counts its work units in 24 bits
    units_ok = _desc(batch=2, num_q_heads=256, num_kv_heads=64, head_dim=128, max_nodes=4, total_rows=8,
                     capacity=2048 * 1100, max_prefix=2048 * 1100)
    assert tv.tv_attn_plan(units_ok)["kernel"] == 3
    assert L.tv_workspace_size(ctypes.byref(units_ok), 0, ctypes.byref(n)) == 0
    too_many_units = _desc(batch=2, num_q_heads=256, num_kv_heads=64, head_dim=128, max_nodes=4, total_rows=8,
                           capacity=2048 * 140000, max_prefix=2048 * 140000)
    assert L.tv_workspace_size(ctypes.byref(too_many_units), 0, ctypes.byref(n)) == -6
    many_rows = _desc(batch=2000, max_nodes=64, total_rows=66000, capacity=64, max_prefix=32)
    assert L.tv_workspace_size(ctypes.byref(many_rows), 0, ctypes.byref(n)) == 0   # attention alone is fine
    args = [fake] * 15
    assert L.tree_accept_commit(ctypes.byref(many_rows), 1000, 1, *args, 1 << 30, fake, None) == -6


def test_null_and_alignment_and_workspace(L):
    d = _desc()
    fake = 1 << 20
    ptrs = [fake] * 10
    assert L.tree_verify_attn(None, *ptrs, fake, 1 << 30, fake, None) == -1
    bad = list(ptrs)
    bad[0] = None
    assert L.tree_verify_attn(ctypes.byref(d), *bad, fake, 1 << 30, fake, None) == -1
    bad[0] = fake + 8
    assert L.tree_verify_attn(ctypes.byref(d), *bad, fake, 1 << 30, fake, None) == -11
    assert L.tree_verify_attn(ctypes.byref(d), *ptrs, fake, 16, fake, None) == -10
    # paged cache requires a page table
    dp = _desc(page_size=16, num_pages=300, capacity=4176)
    bad = list(ptrs)
    bad[3] = None
    assert L.tree_verify_attn(ctypes.byref(dp), *bad, fake, 1 << 30, fake, None) == -1
    # accept: bad logits dtype, vocab, workspace
    args = [fake] * 15
    assert L.tree_accept_commit(ctypes.byref(d), 1000, 5, *args, 1 << 30, fake, None) == -2
    assert L.tree_accept_commit(ctypes.byref(d), 0, 1, *args, 1 << 30, fake, None) == -6
    assert L.tree_accept_commit(ctypes.byref(d), 1000, 1, *args, 64, fake, None) == -10


def test_workspace_and_plan(L):
    d = _desc()
    ws = tv.tv_workspace_size(d, 151936)
    assert ws > tv.tv_workspace_size(d, 0) > 0
    plan = tv.tv_attn_plan(d)
    assert plan["num_splits"] >= 1 and plan["chunk"] * plan["num_splits"] >= 4096
    assert plan["rows_per_tile"] * plan["row_tiles"] >= 64 * 4
    assert plan["kernel"] == 2                       # bf16, d256, 256 rows per KV head: CTA pairs
    assert plan["rows_per_tile"] == 128 and plan["chunk"] % 128 == 0
    assert tv.tv_attn_plan(_desc(max_nodes=16, total_rows=16))["kernel"] == 1   # 64 rows: one CTA per tile
    assert tv.tv_attn_plan(_desc(dtype=tv.F32))["kernel"] == 0
    assert tv.tv_attn_plan(_desc(head_dim=512))["kernel"] == 0
    assert tv.tv_attn_plan(_desc(max_nodes=2, total_rows=2))["kernel"] == 0   # 8 rows per KV head
    g3 = tv.tv_attn_plan(_desc(num_q_heads=24))                               # G = 3: 126-row tiles
    assert g3["kernel"] == 2 and g3["rows_per_tile"] == 126
    # batches: the persistent kernel on head_dim 128 with a bf16 output, else one CTA per tile
    bd = dict(batch=4, head_dim=128, max_nodes=64, total_rows=200, page_size=16, num_pages=2000, capacity=8192,
              max_prefix=8000)
    assert tv.tv_attn_plan(_desc(**bd))["kernel"] == 3
    assert tv.tv_attn_plan(_desc(**bd))["grid_ctas"] <= 1024
    assert tv.tv_attn_plan(_desc(**bd))["grid_ctas"] % 2 == 0                # CTA pairs
    assert tv.tv_attn_plan(_desc(**dict(bd, out_f32=1)))["kernel"] == 1
    assert tv.tv_attn_plan(_desc(**dict(bd, head_dim=256)))["kernel"] == 1


def test_sampled_rejects_bad_temperature(L):
    d = _desc()
    fake = 1 << 20
    args = [fake] * 14
    for t in (0.0, -1.0, float("nan"), float("inf"), 1e-45):
        rc = L.tree_accept_commit_sampled(ctypes.byref(d), 1000, 1, fake, t, 1, 2, *args, 1 << 30, fake, None)
        assert rc == -6, t
    # otherwise the same host checks as the greedy call
    assert L.tree_accept_commit_sampled(ctypes.byref(d), 1000, 5, fake, 1.0, 1, 2, *args, 1 << 30, fake, None) == -2
    assert L.tree_accept_commit_sampled(ctypes.byref(d), 1000, 1, fake, 1.0, 1, 2, *args, 64, fake, None) == -10


def _xdesc(**kw):
    base = dict(batch=1, vocab=151936, top_k=8, width=8, max_nodes=64, max_depth=6, logits_dtype=tv.BF16)
    base.update(kw)
    return tv.make_expand_desc(**base)


@pytest.mark.parametrize("kw,code", [
    (dict(logits_dtype=3), -2), (dict(batch=0), -6), (dict(batch=4096), -6), (dict(vocab=0), -6),
    (dict(top_k=0), -6), (dict(top_k=17), -6), (dict(width=0), -6), (dict(width=17), -6),
    (dict(max_nodes=0), -6), (dict(max_nodes=65), -6), (dict(max_depth=0), -6),
])
def test_expand_descriptor_validation(L, kw, code):
    d = _xdesc(**kw)
    n = ctypes.c_size_t(0)
    assert L.tv_expand_workspace_size(ctypes.byref(d), ctypes.byref(n)) == code
    fake = 1 << 20
    assert L.tv_tree_expand_step(ctypes.byref(d), 0, fake, 1 << 20, *([fake] * 9), 1 << 30, fake, None) == code


def test_expand_host_checks(L):
    d = _xdesc()
    fake = 1 << 20
    ptrs = [fake] * 9
    ws = tv.tv_expand_workspace_size(d)
    step = lambda s, stride, p, wsb: L.tv_tree_expand_step(ctypes.byref(d), s, p[0], stride, *p[1:], wsb, fake, None)
    assert L.tv_tree_expand_step(None, 0, fake, 151936, *ptrs, ws, fake, None) == -1
    bad = [fake] + [None] + ptrs[1:]                                   # no root tokens at step 0
    assert step(0, 151936, bad, ws) == -1
    assert step(1, 151936, bad, ws) == -6                               # (a later step may pass no roots)
    assert step(0, 151935, [fake] * 10, ws) == -6                      # rows of one tree overlap the next
    assert step(1, 151936, [fake] * 10, ws) == -6                      # a later step reads W rows per tree
    assert step(-1, 151936, [fake] * 10, ws) == -6
    assert step(0, 151936, [fake + 8] + [fake] * 9, ws) == -11
    assert step(0, 151936, [fake] * 10, ws - 1) == -10
    assert tv.tv_expand_steps(d) == 8                                  # 1 + 8 + 8 + ... + 7 nodes
    assert tv.tv_expand_steps(_xdesc(width=1)) == 63
    assert tv.tv_expand_steps(_xdesc(top_k=1, width=4)) == 63          # a chain: one node per step
    assert tv.tv_expand_steps(_xdesc(max_nodes=1)) == 1


def test_accept_commit_argmax_host_checks(L):
    d = _desc()
    fake = 1 << 20
    args = [fake] * 13                             # argmax .. tokens; then status, stream
    assert L.tree_accept_commit_argmax(None, *args, fake, None) == -1
    bad = list(args)
    bad[0] = None                                  # no argmax
    assert L.tree_accept_commit_argmax(ctypes.byref(d), *bad, fake, None) == -1
    bad[0] = fake + 4
    assert L.tree_accept_commit_argmax(ctypes.byref(d), *bad, fake, None) == -11
    assert L.tree_accept_commit_argmax(ctypes.byref(_desc(dtype=7)), *args, fake, None) == -2


def test_bounded_wait_check_host_checks(L):
    fake = 1 << 20
    assert L.tv_check_bounded_wait(999_999, fake, None) == -6
    assert L.tv_check_bounded_wait(10_000_000_001, fake, None) == -6
    assert L.tv_check_bounded_wait(20_000_000, None, None) == -1
    assert L.tv_check_bounded_wait(20_000_000, fake + 4, None) == -11
