"""Plain float64 CPU oracle for dynamic draft-tree expansion (EAGLE-2 style).

TEST INFRASTRUCTURE ONLY.  Only the test suite, the package's smoke check and
the benchmark's CPU-baseline / reference leg may import this module.  It
shares no code with the CUDA path and never calls it.

What it computes ("ADR-037 — EAGLE-3 with dynamic tree port", phase rows E4a
and E4b.10a, §4 Phase E4):

* top-K of a row of draft logits: the K largest entries, largest first; equal
  values go in increasing token order (the smaller token wins ties); the
  selection compares the raw values, never a rounded or clamped copy; NaN is
  never chosen.
* log-probabilities: log softmax of the row in float64, over its non-NaN
  entries (the largest value is subtracted before the exponentials).
* expansion: a pool of pending candidates keyed by their cumulative log
  probability (float64: the parent's plus the child's log-probability).  The
  root (depth 0, cumulative 0) is expanded first.  Each step moves the best
  pending candidates into the tree, at most W of them and never more than the
  budget of N nodes (root included), best first; the nodes moved in one step
  are expanded together by the next drafter call, each adding its top-K
  children to the pool (no children at the depth limit).  Best = largest
  cumulative log-probability; equal values go to the candidate generated
  first (generation order: step, then the expanded node's place in that
  step, then the child's top-K rank).  With W = 1 this is the pages' global
  best-first expansion, in which a grandchild of A can enter the tree before
  a sibling of A.
* a drafter row holding +inf is outside the log-softmax's domain: that node
  gets no children, the rest of the expansion goes on, and the result says so
  (`bad_logits`).

The drafter is the caller's: `logits_of(step, j, path)` returns the draft
logits of the j-th node expanded at `step` (step 0 expands the root), whose
root-to-node token path is `path`.

Parity status: top-K pinned by the pages' ordering example and a library
stable sort; log softmax by scipy; the expansion by a hand-derived golden
tree (the pages' grandchild-before-sibling case), by brute force over whole
candidate trees (with W = 1 the tree is the N - 1 best nodes of the full
K-ary tree) and by invariants.
"""
from __future__ import annotations

import numpy as np


def _f64(row):
    if hasattr(row, "double"):
        row = row.double().cpu().numpy()
    return np.asarray(row, dtype=np.float64).reshape(-1)


def topk_row(row, k):
    """Indices of the k largest non-NaN values, largest first, ties to the
    smaller index: k rounds, each taking the first index of the largest value
    still available.  Fewer than k when the row has fewer non-NaN entries."""
    x = _f64(row).copy()
    out = []
    avail = ~np.isnan(x)
    for _ in range(k):
        if not avail.any():
            break
        idx = np.flatnonzero(avail)
        best = int(idx[np.argmax(x[idx])])     # first occurrence of the maximum
        out.append(best)
        avail[best] = False
    return out


def log_softmax_row(row):
    """log p_v = x_v - (m + log sum_u exp(x_u - m)), m the largest value, over
    the non-NaN entries, in float64.  NaN entries stay NaN.  A row with +inf
    is outside the domain (ValueError)."""
    x = _f64(row)
    ok = ~np.isnan(x)
    if not ok.any():
        return np.full_like(x, np.nan)
    if np.isposinf(x[ok]).any():
        raise ValueError("+inf draft logit")
    m = x[ok].max()
    if np.isneginf(m):
        return np.where(ok, -np.inf, np.nan)
    lse = m + np.log(np.exp(x[ok] - m).sum())
    return x - lse


def expand_tree(logits_of, root_token, k, n_max, width, max_depth, token_map=None):
    """The expansion above for one tree.  Returns a dict with
    tokens, parents, depths (int lists) and cum (float64 list), one entry per
    node in the order nodes entered the tree (root first, so parents[i] < i),
    the number of drafter calls, and `gaps`: for every node moved into the
    tree, the distance between its cumulative log-probability and that of the
    best candidate left behind at that moment (inf when none is left)."""
    tokens, parents, depths, cum = [int(root_token)], [-1], [0], [0.0]
    pool = []                   # [cum, generation order, parent, token, depth]
    order = 0
    expand = [0]
    gaps = []
    bad_logits = False
    step = 0
    while True:
        # expand the nodes moved in last step (step 0: the root)
        for j, u in enumerate(expand):
            if depths[u] >= max_depth:
                continue
            path = _path(u, tokens, parents)
            row = logits_of(step, j, path)
            if np.isposinf(_f64(row)).any():
                # a +inf logit is outside the log-softmax's domain: the node
                # gets no children and the expansion reports it
                bad_logits = True
                continue
            lp = log_softmax_row(row)
            for rank, v in enumerate(topk_row(row, k)):
                tok = int(token_map[v]) if token_map is not None else int(v)
                pool.append([cum[u] + lp[v], order + j * k + rank, u, tok, depths[u] + 1])
        order += len(expand) * k
        step += 1
        # move the best candidates into the tree
        expand = []
        while len(expand) < width and len(tokens) < n_max and pool:
            pool.sort(key=lambda c: (-c[0], c[1]))
            c = pool.pop(0)
            gaps.append(float("inf") if not pool else 0.0 if c[0] == pool[0][0] else c[0] - pool[0][0])
            tokens.append(c[3])
            parents.append(c[2])
            depths.append(c[4])
            cum.append(c[0])
            expand.append(len(tokens) - 1)
        if not expand or len(tokens) >= n_max:
            break
    return dict(tokens=tokens, parents=parents, depths=depths, cum=cum, calls=step, gaps=gaps,
                bad_logits=bad_logits)


def _path(u, tokens, parents):
    p = []
    while u >= 0:
        p.append(tokens[u])
        u = parents[u]
    return p[::-1]


def table_drafter(table_b):
    """The synthetic drafter used with seeded tables: the j-th node expanded
    at step s gets row table_b[s, j] ([steps, rows, V])."""
    def logits_of(step, j, path):
        return table_b[step, j]
    return logits_of


def expand_batch(table, root_tokens, k, n_max, width, max_depth, token_map=None):
    """expand_tree for every sequence b of a [B, steps, rows, V] table."""
    return [expand_tree(table_drafter(table[b]), int(root_tokens[b]), k, n_max, width, max_depth,
                        token_map) for b in range(table.shape[0])]
