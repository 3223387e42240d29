"""Seeded synthetic inputs for the tree-verify step.

This module only draws random numbers and lays them out.  It holds none of
the verify step's arithmetic (no attention, no argmax, no acceptance walk, no
commit): the draft tokens, whose matching depends on the target argmax, are
composed by ``plant_drafts`` from an argmax that the caller supplies.  Both
the CUDA path's tests and the CPU oracle's tests take their inputs from here.

Workload shapes follow the five verify-step workloads of the tree-decoding
design record ("ADR-037 — EAGLE-3 with dynamic tree port", phase table rows
E1.1-E1.5, E4a and E4b.6) and the ANE verify-batching notes ("Speculative
decoding verify batches to amortize ANE dispatch", the commit-rule and
break-even bullets):

  1  tiny fp32:     B=1, Hq=Hkv=4, d=256, P=24, the 8-node asymmetric tree
                    parents [-1,0,0,1,1,2,3,5]; V=1000 fp32 logits N(0,1);
                    drafts planted so the first two levels match.
  2  chain bf16:    B=1, Hq=16, Hkv=2, d=512, P=508, chain of 4 nodes;
                    V=32000 bf16 logits N(0,2); match probability 0.6.
  3  EAGLE-2 bf16:  B=1, Hq=32, Hkv=8, d=256, P=4096, 64-node tree (top-8
                    expansion per depth to depth 6, pruned to 64 by seeded
                    confidences); V=151936 bf16 N(0,3); p=0.7.
  4  long bf16:     B=1, Hq=16, Hkv=4, d=256, P=32768, 60-node tree from
                    branching factors 4,3,2,2,1,1; V=151936 N(0,3); p=0.7.
  5  batched bf16:  B=16, P_b ~ U[512, 8192], N_b ~ U{16..64} random trees of
                    depth <= 8, Hq=32, Hkv=8, d=128, paged cache with
                    16-token pages in shuffled order; V=128256 N(0,3); p=0.7.

Draw order from ``torch.Generator('cpu').manual_seed(seed)`` (seed defaults to
1000 + workload number): tree structure (confidences or parents, and for the
batched workload N_b and P_b), Q, then per sequence the prefix K and V, the
tree K and V, the logits, the match coins, the replacement tokens, the page
permutation.  Floating values are drawn in fp32 and cast to bf16 with
round-to-nearest-even (``Tensor.to(torch.bfloat16)``); consumers read exactly
those bits.
"""
from __future__ import annotations

import dataclasses
import math
from dataclasses import dataclass, field
from typing import Callable, Optional

import torch

PAGE_SIZE = 16


@dataclass(frozen=True)
class Spec:
    name: str
    batch: int
    hq: int
    hkv: int
    d: int
    dtype: str                 # "f32" or "bf16" (Q, K, V, cache, tree K/V)
    prefix: tuple              # (lo, hi) inclusive; lo == hi for a fixed prefix
    tree: str                  # "config1" | "chain:N" | "eagle2:K,D,N" | "factors:a,b,..->N" | "random:lo,hi,maxdepth"
    vocab: int
    logit_dtype: str           # "f32" or "bf16"
    logit_std: float
    p_match: float             # per-node match probability (ignored for "config1" planting)
    paged: bool = False
    seed: int = 0
    cache_margin: int = 16     # extra cache rows beyond P_b + N_b (room for repeated commits)

    def replace(self, **kw) -> "Spec":
        return dataclasses.replace(self, **kw)


CONFIGS = {
    1: Spec("tiny-fp32-d256-p24-tree8", 1, 4, 4, 256, "f32", (24, 24), "config1",
            1000, "f32", 1.0, 1.0, seed=1001),
    2: Spec("chain-bf16-d512-p508-q4", 1, 16, 2, 512, "bf16", (508, 508), "chain:4",
            32000, "bf16", 2.0, 0.6, seed=1002),
    3: Spec("eagle2-bf16-d256-p4096-tree64", 1, 32, 8, 256, "bf16", (4096, 4096), "eagle2:8,6,64",
            151936, "bf16", 3.0, 0.7, seed=1003),
    4: Spec("long-bf16-d256-p32768-tree60", 1, 16, 4, 256, "bf16", (32768, 32768),
            "factors:4,3,2,2,1,1->60", 151936, "bf16", 3.0, 0.7, seed=1004),
    5: Spec("batched-paged-bf16-d128-b16", 16, 32, 8, 128, "bf16", (512, 8192), "random:16,64,8",
            128256, "bf16", 3.0, 0.7, paged=True, seed=1005),
}


# ----------------------------------------------------------------------------
# tree shapes (the drafter's side; here only to give the verify step realistic
# inputs).  Each returns a list of parent indices, root first, topological.
# ----------------------------------------------------------------------------

def _renumber(nodes):
    """nodes: list of (depth, -cum, gen_order, parent_gen) with gen 0 = root.
    Returns parents in order sorted by (depth, -cum, gen_order)."""
    order = sorted(range(len(nodes)), key=lambda i: (nodes[i][0], nodes[i][1], nodes[i][2]))
    new_of = {nodes[i][2]: r for r, i in enumerate(order)}
    parents = []
    for i in order:
        pg = nodes[i][3]
        parents.append(-1 if pg < 0 else new_of[pg])
    return parents


def _tree_eagle2(gen, topk, depth, budget):
    """Per-depth expansion: at each depth 1..depth take the `topk` highest
    cumulative-confidence nodes of the previous depth and give each `topk`
    children with U(0,1) confidences; keep the root plus the budget-1 best
    candidates by cumulative confidence (ancestor-closed because the
    cumulative product only falls along a path)."""
    # gen_order, depth, cum, parent_gen
    cand = [(0, 0, 1.0, -1)]
    frontier = [cand[0]]
    for dep in range(1, depth + 1):
        frontier = sorted(frontier, key=lambda t: (-t[2], t[0]))[:topk]
        conf = torch.rand(len(frontier) * topk, generator=gen, dtype=torch.float64).tolist()
        new = []
        for a, par in enumerate(frontier):
            for c in range(topk):
                g = len(cand)
                node = (g, dep, par[2] * conf[a * topk + c], par[0])
                cand.append(node)
                new.append(node)
        frontier = new
    root, rest = cand[0], cand[1:]
    keep = [root] + sorted(rest, key=lambda t: (-t[2], t[1], t[0]))[: budget - 1]
    return _renumber([(t[1], -t[2], t[0], t[3]) for t in keep])


def _tree_factors(gen, factors, budget):
    """Full expansion with per-depth branching factors, U(0,1) confidence per
    node, cumulative product along the path, keep the best `budget`."""
    cand = [(0, 0, 1.0, -1)]
    level = [cand[0]]
    for dep, f in enumerate(factors, start=1):
        conf = torch.rand(len(level) * f, generator=gen, dtype=torch.float64).tolist()
        new = []
        for a, par in enumerate(level):
            for c in range(f):
                g = len(cand)
                node = (g, dep, par[2] * conf[a * f + c], par[0])
                cand.append(node)
                new.append(node)
        level = new
    root, rest = cand[0], cand[1:]
    keep = [root] + sorted(rest, key=lambda t: (-t[2], t[1], t[0]))[: budget - 1]
    return _renumber([(t[1], -t[2], t[0], t[3]) for t in keep])


def _tree_random(gen, lo, hi, maxdepth):
    n = int(torch.randint(lo, hi + 1, (1,), generator=gen).item())
    parents, depth = [-1], [0]
    for i in range(1, n):
        allowed = [j for j in range(i) if depth[j] < maxdepth]
        pick = allowed[int(torch.randint(0, len(allowed), (1,), generator=gen).item())]
        parents.append(pick)
        depth.append(depth[pick] + 1)
    return parents


def make_tree(spec: Spec, gen) -> list:
    kind, _, arg = spec.tree.partition(":")
    if kind == "config1":
        return [-1, 0, 0, 1, 1, 2, 3, 5]
    if kind == "chain":
        return [-1] + list(range(int(arg) - 1))
    if kind == "eagle2":
        k, dep, n = (int(x) for x in arg.split(","))
        return _tree_eagle2(gen, k, dep, n)
    if kind == "factors":
        fs, n = arg.split("->")
        return _tree_factors(gen, [int(x) for x in fs.split(",")], int(n))
    if kind == "random":
        lo, hi, md = (int(x) for x in arg.split(","))
        return _tree_random(gen, lo, hi, md)
    if kind == "parents":
        return [int(x) for x in arg.split(",")]
    raise ValueError(f"unknown tree kind {spec.tree!r}")


# ----------------------------------------------------------------------------
# workload
# ----------------------------------------------------------------------------

@dataclass
class Workload:
    spec: Spec
    parents: list                      # list of per-sequence parent lists (local indices)
    node_offsets: torch.Tensor         # int32 [B+1]
    parents_flat: torch.Tensor         # int32 [sumN]
    prefix_len: torch.Tensor           # int32 [B]
    q: torch.Tensor                    # [sumN, Hq, d]
    k_tree: torch.Tensor               # [Hkv, sumN, d]
    v_tree: torch.Tensor
    k_cache: torch.Tensor              # contiguous [B, Hkv, cap, d] or paged [pages, Hkv, 16, d]
    v_cache: torch.Tensor
    page_table: Optional[torch.Tensor]  # int32 [B, max_pages] (paged only; -1 = unallocated)
    capacity: int                      # per-sequence capacity in tokens
    logits: torch.Tensor               # [sumN, V]
    coins: torch.Tensor                # float64 [sumN] U(0,1)
    repl: torch.Tensor                 # int64 [sumN] uniform in [0, V-1)
    repl_full: torch.Tensor            # int64 [sumN] uniform in [0, V)
    draft_tokens: Optional[torch.Tensor] = None   # int32 [sumN]
    extra: dict = field(default_factory=dict)

    @property
    def batch(self):
        return self.spec.batch

    @property
    def total_rows(self):
        return int(self.node_offsets[-1])

    @property
    def max_nodes(self):
        return max(len(p) for p in self.parents)

    @property
    def scale(self):
        return 1.0 / math.sqrt(self.spec.d)

    def seq_rows(self, b):
        return int(self.node_offsets[b]), int(self.node_offsets[b + 1])


def _torch_dtype(s):
    return {"f32": torch.float32, "bf16": torch.bfloat16}[s]


def make_workload(spec: Spec, canary: float = float("nan"),
                  argmax_fn: Optional[Callable] = None) -> Workload:
    """Draw one workload.  `canary` fills every cache row that holds no
    prefix token (so a kernel that reads past the prefix shows it).  If
    `argmax_fn(logits) -> int tensor [sumN]` is given, drafts are planted
    right away (see ``plant_drafts``)."""
    gen = torch.Generator("cpu").manual_seed(spec.seed)
    B, Hq, Hkv, d = spec.batch, spec.hq, spec.hkv, spec.d
    if Hkv <= 0 or Hq % Hkv:
        raise ValueError("bad head counts")
    dt = _torch_dtype(spec.dtype)

    # 1. tree structure and prefix lengths
    parents = [make_tree(spec, gen) for _ in range(B)]
    lo, hi = spec.prefix
    if lo == hi:
        plens = [lo] * B
    else:
        plens = torch.randint(lo, hi + 1, (B,), generator=gen).tolist()
    ns = [len(p) for p in parents]
    offs = [0]
    for n in ns:
        offs.append(offs[-1] + n)
    total = offs[-1]

    def randn(*shape):
        return torch.randn(*shape, generator=gen, dtype=torch.float32).to(dt)

    # 2. Q, 3. prefix K/V per sequence, 4. tree K/V
    q = randn(total, Hq, d)
    kp = [randn(Hkv, plens[b], d) for b in range(B)]
    vp = [randn(Hkv, plens[b], d) for b in range(B)]
    k_tree = randn(Hkv, total, d)
    v_tree = randn(Hkv, total, d)

    # 5. logits
    ldt = _torch_dtype(spec.logit_dtype)
    logits = (torch.randn(total, spec.vocab, generator=gen, dtype=torch.float32) * spec.logit_std).to(ldt)

    # 6. coins and replacement tokens
    coins = torch.rand(total, generator=gen, dtype=torch.float64)
    repl = torch.randint(0, max(spec.vocab - 1, 1), (total,), generator=gen)
    repl_full = torch.randint(0, spec.vocab, (total,), generator=gen)

    # cache layout
    need = [plens[b] + ns[b] + spec.cache_margin for b in range(B)]
    if not spec.paged:
        cap = -(-max(need) // PAGE_SIZE) * PAGE_SIZE
        k_cache = torch.full((B, Hkv, cap, d), canary, dtype=dt)
        v_cache = torch.full((B, Hkv, cap, d), canary, dtype=dt)
        for b in range(B):
            k_cache[b, :, : plens[b]] = kp[b]
            v_cache[b, :, : plens[b]] = vp[b]
        page_table = None
    else:
        pages_b = [-(-n // PAGE_SIZE) for n in need]
        max_pages = max(pages_b)
        cap = max_pages * PAGE_SIZE
        n_pages = sum(pages_b)
        # 7. page permutation
        perm = torch.randperm(n_pages, generator=gen)
        page_table = torch.full((B, max_pages), -1, dtype=torch.int32)
        k_cache = torch.full((n_pages, Hkv, PAGE_SIZE, d), canary, dtype=dt)
        v_cache = torch.full((n_pages, Hkv, PAGE_SIZE, d), canary, dtype=dt)
        base = 0
        for b in range(B):
            ids = perm[base: base + pages_b[b]]
            base += pages_b[b]
            page_table[b, : pages_b[b]] = ids.to(torch.int32)
            for t0 in range(0, plens[b], PAGE_SIZE):
                t1 = min(t0 + PAGE_SIZE, plens[b])
                pid = int(ids[t0 // PAGE_SIZE])
                k_cache[pid, :, : t1 - t0] = kp[b][:, t0:t1]
                v_cache[pid, :, : t1 - t0] = vp[b][:, t0:t1]

    w = Workload(
        spec=spec, parents=parents,
        node_offsets=torch.tensor(offs, dtype=torch.int32),
        parents_flat=torch.tensor([p for ps in parents for p in ps], dtype=torch.int32),
        prefix_len=torch.tensor(plens, dtype=torch.int32),
        q=q, k_tree=k_tree, v_tree=v_tree, k_cache=k_cache, v_cache=v_cache,
        page_table=page_table, capacity=cap, logits=logits,
        coins=coins, repl=repl, repl_full=repl_full,
    )
    if argmax_fn is not None:
        plant_drafts(w, argmax_fn(logits))
    return w


def plant_drafts(w: Workload, am) -> torch.Tensor:
    """Compose draft tokens from a target argmax `am` (one token per tree
    row, supplied by the caller).  Child c of parent u gets am[u] when its
    coin falls below p, else a token drawn uniformly from V minus {am[u]}.
    The root's token is the anchor (never tested), drawn uniformly.  The tiny
    workload plants a fixed pattern instead: node 1 and node 3 match, nodes
    2, 4 and 6 do not, nodes 5 and 7 are uniform draws."""
    am = torch.as_tensor(am).to(torch.int64).reshape(-1)
    V = w.spec.vocab
    out = torch.empty(w.total_rows, dtype=torch.int64)
    planted = {1: "match", 2: "miss", 3: "match", 4: "miss", 5: "any", 6: "miss", 7: "any"}
    for b, ps in enumerate(w.parents):
        o = int(w.node_offsets[b])
        out[o] = w.repl_full[o]
        for i in range(1, len(ps)):
            r = o + i
            target = int(am[o + ps[i]])
            miss = min(int(w.repl[r]) + (1 if int(w.repl[r]) >= target else 0), V - 1)
            if w.spec.tree == "config1":
                mode = planted[i]
            else:
                mode = "match" if float(w.coins[r]) < w.spec.p_match else "miss"
            out[r] = target if mode == "match" else (miss if mode == "miss" else w.repl_full[r])
    w.draft_tokens = out.to(torch.int32)
    return w.draft_tokens


def small_variant(n: int, **kw) -> Spec:
    """A workload with the shape of workload `n` but sizes the oracle finishes
    in seconds (prefix, vocabulary and batch cut down unless overridden)."""
    s = CONFIGS[n]
    defaults = {
        1: dict(),
        2: dict(),
        3: dict(prefix=(700, 700), vocab=5003),
        4: dict(prefix=(1500, 1500), vocab=5003),
        5: dict(batch=4, prefix=(40, 700), vocab=4099),
    }[n]
    defaults.update(kw)
    return s.replace(**defaults)


# ----------------------------------------------------------------------------
# dynamic draft-tree expansion: the drafter's logits, one seeded block per step
# ----------------------------------------------------------------------------

@dataclass(frozen=True)
class ExpandSpec:
    """An expansion workload ("ADR-037 — EAGLE-3 with dynamic tree port",
    phase row E4a and §4 Phase E4: top-K per expanded node, a budget of 64
    nodes; the verify workloads' EAGLE-2 tree is top-8 to depth 6)."""
    name: str
    batch: int
    vocab: int
    top_k: int
    width: int
    max_nodes: int
    max_depth: int
    dtype: str                 # draft logits: "f32" or "bf16"
    logit_std: float
    seed: int

    def replace(self, **kw) -> "ExpandSpec":
        return dataclasses.replace(self, **kw)


EXPAND_CONFIGS = {
    # one tree: top-8, 8 nodes per drafter call, 64 nodes, depth <= 6, Qwen-size vocabulary
    "eagle2": ExpandSpec("expand-eagle2-bf16-v151936-k8-w8-n64", 1, 151936, 8, 8, 64, 6, "bf16", 3.0, 2001),
    # the batched verify workload's 16 sequences, Llama-size vocabulary, depth <= 8
    "batched": ExpandSpec("expand-batched-bf16-v128256-k8-w8-n64-b16", 16, 128256, 8, 8, 64, 8, "bf16", 3.0,
                          2002),
}


def draft_rows(spec: ExpandSpec, step: int) -> torch.Tensor:
    """The synthetic drafter's logits for one expansion step: [B, R, V] with
    R = 1 at step 0 (the roots) and W after (row j = the j-th node the
    previous step moved into tree b), N(0, logit_std) drawn in fp32 from
    torch.Generator('cpu').manual_seed(seed * 1000003 + step) and cast to the
    spec's dtype.  A real drafter's row depends on the node's token path; the
    expansion never looks at that, only at the row it is given."""
    R = 1 if step == 0 else spec.width
    g = torch.Generator("cpu").manual_seed(spec.seed * 1000003 + step)
    x = torch.randn(spec.batch, R, spec.vocab, generator=g) * spec.logit_std
    return x.to(_torch_dtype(spec.dtype))


def root_tokens(spec: ExpandSpec) -> torch.Tensor:
    """[B] int32 root (anchor) tokens, uniform over the vocabulary."""
    g = torch.Generator("cpu").manual_seed(spec.seed * 1000003 - 1)
    return torch.randint(0, spec.vocab, (spec.batch,), generator=g, dtype=torch.int64).to(torch.int32)


# ----------------------------------------------------------------------------
# lm_head + argmax: the target model's final hidden rows and output weights
# ----------------------------------------------------------------------------

@dataclass(frozen=True)
class LmHeadSpec:
    """The lm_head step over a verify workload's tree rows: hidden rows
    [rows, hidden] and output weights [vocab, hidden], both bf16 (random
    weights of that shape: no trained model is used)."""
    name: str
    rows: int
    hidden: int
    vocab: int
    logit_std: float
    seed: int

    def replace(self, **kw) -> "LmHeadSpec":
        return dataclasses.replace(self, **kw)


LMHEAD_CONFIGS = {
    # the 64-node EAGLE-2 tree's rows; a Qwen-family 27B-class model (hidden 5120, vocabulary 151936)
    "qwen": LmHeadSpec("lmhead-bf16-h5120-v151936-r64", 64, 5120, 151936, 3.0, 3001),
    # the batched workload's 16 trees (612 rows); a Llama-family 8B-class model (hidden 4096, vocabulary 128256)
    "batched": LmHeadSpec("lmhead-bf16-h4096-v128256-r612", 612, 4096, 128256, 3.0, 3002),
}


def lm_head_inputs(spec: LmHeadSpec):
    """(hidden [rows, hidden] bf16, weight [vocab, hidden] bf16): hidden rows
    N(0, 1); weights N(0, logit_std^2 / hidden) so that logits have standard
    deviation about logit_std.  Drawn in fp32 from
    torch.Generator('cpu').manual_seed(seed) (hidden first, then the weights
    in blocks of 8192 rows) and cast with round-to-nearest-even."""
    g = torch.Generator("cpu").manual_seed(spec.seed)
    hidden = torch.randn(spec.rows, spec.hidden, generator=g).to(torch.bfloat16)
    w = torch.empty(spec.vocab, spec.hidden, dtype=torch.bfloat16)
    sd = spec.logit_std / math.sqrt(spec.hidden)
    for v0 in range(0, spec.vocab, 8192):
        v1 = min(spec.vocab, v0 + 8192)
        w[v0:v1] = (torch.randn(v1 - v0, spec.hidden, generator=g) * sd).to(torch.bfloat16)
    return hidden, w
