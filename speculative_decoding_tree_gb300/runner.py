"""Device-resident buffers for one verify workload and the C-ABI calls of a
verify step, in stream order: tree mask, attention, accept + commit; and the
same for one dynamic draft-tree expansion (DeviceExpand).

Used by the benchmark, the GPU tests and the smoke check.  It only moves a
workload's tensors to the GPU, allocates the outputs and workspace with
torch, and calls the library; it computes nothing itself.
"""
from __future__ import annotations

import torch

from . import (BF16, F32, make_desc, make_expand_desc, tree_accept_commit, tree_accept_commit_sampled,
               tree_verify_attn, tv_attn_merge, tv_attn_partials, tv_build_tree_mask, tv_expand_steps,
               tv_expand_workspace_size, tv_tree_expand_step, tv_workspace_size, make_lmhead_desc,
               tv_lm_head_argmax, tv_lm_head_workspace_size, tree_accept_commit_argmax)

_DT = {torch.float32: F32, torch.bfloat16: BF16}


class DeviceStep:
    def __init__(self, w, device="cuda", out_f32=False, max_prefix=None, vocab=None, max_nodes=None):
        self.w = w
        dev = torch.device(device)
        self.device = dev
        sp = w.spec
        self.dtype = _DT[w.q.dtype]
        self.logits_dtype = _DT[w.logits.dtype]
        self.vocab = vocab if vocab is not None else w.logits.shape[1]
        mp = int(w.prefix_len.max()) if max_prefix is None else int(max_prefix)
        self.desc = make_desc(
            batch=sp.batch, num_q_heads=sp.hq, num_kv_heads=sp.hkv, head_dim=sp.d, dtype=self.dtype,
            max_nodes=w.max_nodes if max_nodes is None else int(max_nodes), total_rows=w.total_rows, capacity=w.capacity, max_prefix=mp,
            page_size=16 if w.page_table is not None else 0,
            num_pages=w.k_cache.shape[0] if w.page_table is not None else 0,
            out_f32=int(out_f32))
        to = lambda t: None if t is None else t.to(dev).contiguous()
        self.q, self.k_tree, self.v_tree = to(w.q), to(w.k_tree), to(w.v_tree)
        self.k_cache, self.v_cache = to(w.k_cache), to(w.v_cache)
        self.page_table = to(w.page_table)
        self.prefix_len = to(w.prefix_len)
        self.node_offsets = to(w.node_offsets)
        self.parents = to(w.parents_flat)
        self.logits = to(w.logits)
        self.draft = to(w.draft_tokens) if w.draft_tokens is not None else None
        R, B, mn = w.total_rows, sp.batch, self.desc.max_nodes
        self.anc = torch.zeros(R, dtype=torch.int64, device=dev)
        self.depth = torch.zeros(R, dtype=torch.int32, device=dev)
        odt = torch.float32 if (self.dtype == F32 or out_f32) else torch.bfloat16
        self.out = torch.zeros(R, sp.hq, sp.d, dtype=odt, device=dev)
        self.status = torch.zeros(4, dtype=torch.int32, device=dev)
        self.argmax = torch.zeros(R, dtype=torch.int32, device=dev)
        self.accept_len = torch.zeros(B, dtype=torch.int32, device=dev)
        self.path = torch.zeros(B, mn, dtype=torch.int32, device=dev)
        self.tokens = torch.zeros(B, mn, dtype=torch.int32, device=dev)
        self.ws_bytes = tv_workspace_size(self.desc, self.vocab)
        self.workspace = torch.empty(max(self.ws_bytes, 256), dtype=torch.uint8, device=dev)

    # one call each ------------------------------------------------------
    def mask(self, stream=None):
        tv_build_tree_mask(self.desc, self.parents, self.node_offsets, self.anc, self.depth, self.status, stream)

    def attn(self, stream=None):
        tree_verify_attn(self.desc, self.q, self.k_cache, self.v_cache, self.page_table, self.prefix_len,
                         self.node_offsets, self.k_tree, self.v_tree, self.anc, self.out, self.workspace,
                         self.ws_bytes, self.status, stream)

    def partials(self, stream=None):
        tv_attn_partials(self.desc, self.q, self.k_cache, self.v_cache, self.page_table, self.prefix_len,
                         self.node_offsets, self.k_tree, self.v_tree, self.anc, self.workspace, self.ws_bytes,
                         self.status, stream)

    def merge(self, stream=None):
        tv_attn_merge(self.desc, self.prefix_len, self.node_offsets, self.out, self.workspace, self.ws_bytes,
                      self.status, stream)

    def accept_commit(self, stream=None):
        tree_accept_commit(self.desc, self.vocab, self.logits_dtype, self.logits, self.draft, self.parents,
                           self.node_offsets, self.k_tree, self.v_tree, self.k_cache, self.v_cache,
                           self.page_table, self.prefix_len, self.argmax, self.accept_len, self.path,
                           self.tokens, self.workspace, self.ws_bytes, self.status, stream)

    def accept_commit_sampled(self, temperature, seed, offset, stream=None):
        """Sampled verification: one draw per tree row (written to self.argmax),
        then the same walk and commit."""
        tree_accept_commit_sampled(self.desc, self.vocab, self.logits_dtype, self.logits, temperature, seed, offset,
                                   self.draft, self.parents, self.node_offsets, self.k_tree, self.v_tree,
                                   self.k_cache, self.v_cache, self.page_table, self.prefix_len, self.argmax,
                                   self.accept_len, self.path, self.tokens, self.workspace, self.ws_bytes,
                                   self.status, stream)

    def accept_commit_argmax(self, argmax, stream=None):
        """The walk and commit on a given argmax [rows] int32 (device)."""
        tree_accept_commit_argmax(self.desc, argmax, self.draft, self.parents, self.node_offsets, self.k_tree,
                                  self.v_tree, self.k_cache, self.v_cache, self.page_table, self.prefix_len,
                                  self.accept_len, self.path, self.tokens, self.status, stream)

    def step(self, stream=None):
        """One verify step: mask, attention, accept + commit."""
        self.mask(stream)
        self.attn(stream)
        self.accept_commit(stream)

    def kernels_per_step(self):
        """Our kernel launches in one step: mask, split, merge (skipped when
        the plan has one key chunk), argmax, walk + commit."""
        from . import tv_attn_plan
        return 4 + (1 if tv_attn_plan(self.desc)["num_splits"] > 1 else 0)


class DeviceExpand:
    """Device buffers of one expansion workload (workloads.ExpandSpec): the
    synthetic drafter's logits of every step (resident), the roots, the tree
    outputs and the workspace; step(s) is one tv_tree_expand_step call."""

    def __init__(self, spec, device="cuda", rows=None, token_map=None, steps=None):
        from . import workloads as wl
        dev = torch.device(device)
        self.spec = spec
        dt = {"f32": F32, "bf16": BF16}[spec.dtype]
        self.desc = make_expand_desc(batch=spec.batch, vocab=spec.vocab, top_k=spec.top_k, width=spec.width,
                                     max_nodes=spec.max_nodes, max_depth=spec.max_depth, logits_dtype=dt)
        self.steps = tv_expand_steps(self.desc) if steps is None else int(steps)
        if rows is None:
            rows = [wl.draft_rows(spec, s) for s in range(self.steps)]
        self.rows = [r.to(dev).contiguous() for r in rows]
        self.roots = wl.root_tokens(spec).to(dev)
        self.token_map = None if token_map is None else token_map.to(dev).to(torch.int32).contiguous()
        B, N = spec.batch, spec.max_nodes
        self.tokens = torch.zeros(B, N, dtype=torch.int32, device=dev)
        self.parents = torch.zeros(B, N, dtype=torch.int32, device=dev)
        self.depths = torch.zeros(B, N, dtype=torch.int32, device=dev)
        self.cum = torch.zeros(B, N, dtype=torch.float64, device=dev)
        self.n_nodes = torch.zeros(B, dtype=torch.int32, device=dev)
        self.expand_count = torch.zeros(B, dtype=torch.int32, device=dev)
        self.status = torch.zeros(4, dtype=torch.int32, device=dev)
        self.ws_bytes = tv_expand_workspace_size(self.desc)
        self.workspace = torch.empty(max(self.ws_bytes, 256), dtype=torch.uint8, device=dev)

    def step(self, s, stream=None):
        x = self.rows[s]
        tv_tree_expand_step(self.desc, s, x, x.shape[1] * x.shape[2], self.roots, self.token_map, self.tokens,
                            self.parents, self.depths, self.cum, self.n_nodes, self.expand_count, self.workspace,
                            self.ws_bytes, self.status, stream)

    def run(self, stream=None):
        """Every step, in order (two kernel launches each)."""
        for s in range(self.steps):
            self.step(s, stream)


class DeviceLmHead:
    """Device buffers of one lm_head workload (workloads.LmHeadSpec): hidden
    rows and weights resident, the argmax and max-logit outputs, the
    workspace; run() is one tv_lm_head_argmax call."""

    def __init__(self, spec, device="cuda", hidden=None, weight=None):
        from . import workloads as wl
        dev = torch.device(device)
        self.spec = spec
        if hidden is None or weight is None:
            hidden, weight = wl.lm_head_inputs(spec)
        self.hidden = hidden.to(dev).contiguous()
        self.weight = weight.to(dev).contiguous()
        self.desc = make_lmhead_desc(rows=spec.rows, hidden=spec.hidden, vocab=spec.vocab)
        self.argmax = torch.zeros(spec.rows, dtype=torch.int32, device=dev)
        self.max_logit = torch.zeros(spec.rows, dtype=torch.float32, device=dev)
        self.status = torch.zeros(4, dtype=torch.int32, device=dev)
        self.ws_bytes = tv_lm_head_workspace_size(self.desc)
        self.workspace = torch.empty(max(self.ws_bytes, 256), dtype=torch.uint8, device=dev)

    def run(self, stream=None, weight=None):
        tv_lm_head_argmax(self.desc, self.hidden, self.weight if weight is None else weight, self.argmax,
                          self.max_logit, self.workspace, self.ws_bytes, self.status, stream)


def main(argv=None):
    """Run one seeded input set of a workload through the verify step a few
    times (e.g. under a profiler): python -m speculative_decoding_tree_gb300.runner
    --config 4 --steps 3.  Prints the device status word and exits non-zero
    when it is not 0."""
    import argparse

    from . import _build, workloads as wl

    ap = argparse.ArgumentParser()
    ap.add_argument("--config", type=int, default=4, help="workload 1..5")
    ap.add_argument("--steps", type=int, default=3)
    ap.add_argument("--attn-only", action="store_true", help="mask and attention only")
    ap.add_argument("--sampled", type=float, default=0.0,
                    help="temperature > 0: sampled verification (tree_accept_commit_sampled)")
    ap.add_argument("--expand", default="", help="run a dynamic-expansion workload instead (eagle2, batched)")
    ap.add_argument("--lm-head", default="", help="run a fused lm_head + argmax workload instead (qwen, batched)")
    ap.add_argument("--vocab", type=int, default=0, help="with --lm-head: a smaller vocabulary (e.g. for a profiler)")
    a = ap.parse_args(argv)
    _build.build()
    if a.lm_head:
        spec = wl.LMHEAD_CONFIGS[a.lm_head]
        lm = DeviceLmHead(spec.replace(vocab=a.vocab, name=f"{spec.name}-v{a.vocab}") if a.vocab else spec)
        for _ in range(a.steps):
            lm.run()
        torch.cuda.synchronize()
        status = int(lm.status[0].item())
        print(f"{lm.spec.name}: {a.steps} calls, device status {status}")
        return 0 if status == 0 else 1
    if a.expand:
        dx = DeviceExpand(wl.EXPAND_CONFIGS[a.expand])
        for _ in range(a.steps):
            dx.run()
        torch.cuda.synchronize()
        status = int(dx.status[0].item())
        print(f"{dx.spec.name}: {a.steps} expansions of {dx.steps} steps, {int(dx.n_nodes.sum())} nodes, "
              f"device status {status}")
        return 0 if status == 0 else 1
    w = wl.make_workload(wl.CONFIGS[a.config], canary=0.0,
                         argmax_fn=lambda x: torch.argmax(x.float(), dim=1))   # plants the draft tokens
    st = DeviceStep(w)
    p0 = st.prefix_len.clone()
    for _ in range(a.steps):
        st.prefix_len.copy_(p0)
        if a.attn_only:
            st.mask()
            st.attn()
        elif a.sampled > 0:
            st.mask()
            st.attn()
            st.accept_commit_sampled(a.sampled, 1234, _)
        else:
            st.step()
    torch.cuda.synchronize()
    status = int(st.status[0].item())
    print(f"{w.spec.name}: {a.steps} steps, device status {status}")
    return 0 if status == 0 else 1


if __name__ == "__main__":
    raise SystemExit(main())
