"""Plain, slow, float64 CPU oracle for the tree-verify step.

TEST INFRASTRUCTURE ONLY.  Only the test suite, the package's smoke check and
the benchmark's CPU-baseline / reference leg may import this module.  It
shares no code with the CUDA path and never calls it.

Everything here is the textbook definition written out, step by step, in
float64 (inputs are the exact bf16 / fp32 values widened to double):

* ancestors / depths: walk the parent pointers ("ADR-037 — EAGLE-3 with
  dynamic tree port", §4 Phase E1 mask encoding: each tree node attends to
  the whole prefix and to its ancestors and itself; posttrainllm
  "Speculative-decoding heads", What's not implemented (1c)).
* attention: scores s_j = scale * q . k_j over the visible keys, softmax,
  weighted sum of the visible values (ADR-037 phase table E1.1-E1.5; output
  row-major [q_rows, num_heads, head_dim], phase row E1.3).  Query head h
  reads KV head h // (Hq / Hkv) (contiguous GQA groups).
* argmax: one linear scan; a strictly greater value replaces the current
  best, so the smallest index wins ties (ADR-037 phase row E4b.10a fixes
  "smaller token wins on ties" for top-K; the same rule is used here).  NaN
  is never selected; an all-NaN row gives index 0.
* acceptance: brute force over every root-to-leaf path; child c matches when
  draft[c] equals the target argmax at its parent; take the longest matching
  prefix, ties to the smallest end node; emit the accepted drafts plus the
  target argmax at the end node (ADR-037 row E5a and Phase E5 edge cases;
  "Speculative decoding verify batches to amortize ANE dispatch", commit-rule
  bullet).
* commit: a copy of the cache with rows P..P+k overwritten by the tree K/V of
  the accepted path nodes, in path order, and P' = P+k+1; nothing else moves
  (same page, KV write-before-accept and Forge accept(k) bullets).

Parity status: attention values are pinned by invariants and library
special cases (single query, chain == causal attention, union of chains,
uniform-score and two-key closed forms); acceptance by an independent greedy
walk, exhaustive match patterns and the printed expected-tokens figures.
"""
from __future__ import annotations

import numpy as np

PAGE_SIZE = 16


def _f64(t):
    """Exact widening of a torch tensor (bf16 / fp32 / int) or array to float64 numpy."""
    if hasattr(t, "detach"):
        return t.detach().cpu().double().numpy()
    return np.asarray(t, dtype=np.float64)


# ---------------------------------------------------------------------------
# tree structure
# ---------------------------------------------------------------------------

def ancestors(parents):
    """anc[i] = set of j that are i or an ancestor of i, found by walking
    the parent pointers from i up to the root."""
    out = []
    for i in range(len(parents)):
        s, j = set(), i
        while j != -1:
            s.add(j)
            j = int(parents[j])
        out.append(s)
    return out


def depths(parents):
    return [len(a) - 1 for a in ancestors(parents)]


def check_tree(parents):
    """True when parents[0] == -1 and 0 <= parents[i] < i for every i > 0."""
    if len(parents) == 0 or int(parents[0]) != -1:
        return False
    return all(0 <= int(parents[i]) < i for i in range(1, len(parents)))


# ---------------------------------------------------------------------------
# attention
# ---------------------------------------------------------------------------

def attention_one_sequence(q, k_prefix, v_prefix, k_tree, v_tree, parents, scale,
                           rows=None, heads=None):
    """Tree-verify attention for one sequence, float64.

    q        [N, Hq, d]
    k_prefix [Hkv, P, d], v_prefix [Hkv, P, d]   (committed prefix)
    k_tree   [Hkv, N, d], v_tree   [Hkv, N, d]   (this round's tree nodes)
    Returns out [N, Hq, d]; with `rows` / `heads` given, only those entries
    are computed (the rest stay NaN).
    """
    q, kp, vp, kt, vt = (_f64(x) for x in (q, k_prefix, v_prefix, k_tree, v_tree))
    N, Hq, d = q.shape
    Hkv = kp.shape[0]
    G = Hq // Hkv
    anc = ancestors(parents)
    out = np.full((N, Hq, d), np.nan)
    rows = list(range(N)) if rows is None else list(rows)
    heads = range(Hq) if heads is None else heads
    for h in heads:
        g = h // G
        # score matrix for the wanted rows: every prefix key, every tree key
        s_prefix = scale * (q[rows, h] @ kp[g].T)          # [rows, P]
        s_tree = scale * (q[rows, h] @ kt[g].T)            # [rows, N]
        for r, i in enumerate(rows):
            tree_cols = sorted(anc[i])                     # i and its ancestors only
            s = np.concatenate([s_prefix[r], s_tree[r, tree_cols]])
            w = np.exp(s - s.max())
            P = s_prefix.shape[1]
            o = w[:P] @ vp[g] + w[P:] @ vt[g][tree_cols]
            out[i, h] = o / w.sum()
    return out


def prefix_kv(w, b):
    """The committed prefix K/V of sequence b as [Hkv, P_b, d] float64,
    read from a contiguous [B, Hkv, cap, d] cache or through the page table
    of a paged [pages, Hkv, 16, d] cache."""
    P = int(w.prefix_len[b])
    if w.page_table is None:
        return _f64(w.k_cache[b, :, :P]), _f64(w.v_cache[b, :, :P])
    return gather_pages(w.k_cache, w.page_table[b], P), gather_pages(w.v_cache, w.page_table[b], P)


def gather_pages(pool, table_row, P):
    pool = _f64(pool)
    t = np.arange(P)
    ids = np.asarray(table_row)[t // PAGE_SIZE]
    return pool[ids, :, t % PAGE_SIZE, :].transpose(1, 0, 2)   # [Hkv, P, d]


def tree_attention(w, samples=None):
    """Whole-workload attention, out [sumN, Hq, d] float64.  With
    `samples` = list of (row, head) pairs (global rows) only those are computed."""
    total, Hq, d = w.q.shape
    out = np.full((total, Hq, d), np.nan)
    for b in range(w.batch):
        o0, o1 = w.seq_rows(b)
        want = None
        if samples is not None:
            want = [(r - o0, h) for (r, h) in samples if o0 <= r < o1]
            if not want:
                continue
        kp, vp = prefix_kv(w, b)
        args = (w.q[o0:o1], kp, vp, w.k_tree[:, o0:o1], w.v_tree[:, o0:o1], w.parents[b], w.scale)
        if want is None:
            out[o0:o1] = attention_one_sequence(*args)
        else:
            for (i, h) in want:
                out[o0 + i, h] = attention_one_sequence(*args, rows=[i], heads=[h])[i, h]
    return out


# ---------------------------------------------------------------------------
# acceptance
# ---------------------------------------------------------------------------

def argmax_row(row):
    """Index of the largest value; the first (smallest) index wins ties;
    NaN is never selected; an all-NaN row gives 0."""
    vals = _f64(row).reshape(-1)
    best, best_v = 0, None
    for v_idx in range(vals.shape[0]):
        x = vals[v_idx]
        if np.isnan(x):
            continue
        if best_v is None or x > best_v:
            best, best_v = v_idx, x
    return best


def argmax_rows(logits):
    """argmax_row over every row.  For long rows the scan is done with
    numpy's first-occurrence argmax over the non-NaN entries, which is the
    same rule (smallest index among the maximal values)."""
    x = _f64(logits)
    out = np.zeros(x.shape[0], dtype=np.int64)
    for r in range(x.shape[0]):
        row = x[r]
        ok = ~np.isnan(row)
        if not ok.any():
            out[r] = 0
            continue
        idx = np.flatnonzero(ok)
        out[r] = idx[np.argmax(row[idx])]
    return out


def accept(parents, draft, am):
    """Greedy acceptance by brute force.

    For every root-to-leaf path, walk from the root while each next node c
    has draft[c] == am[parent(c)].  The accepted length k is the number of
    matched drafts.  The best path has the largest k; among equal k the end
    node with the smallest index wins.  Returns (k, path, tokens) with
    path = [0, ..., end] (k+1 nodes) and tokens = drafts of path[1:] plus
    am[end] (k+1 tokens: k accepted drafts and one bonus/correction).
    """
    N = len(parents)
    children = [[] for _ in range(N)]
    for i in range(1, N):
        children[int(parents[i])].append(i)
    best_k, best_end = -1, None
    for leaf in range(N):
        if children[leaf]:
            continue
        path, j = [], leaf
        while j != -1:
            path.append(j)
            j = int(parents[j])
        path.reverse()
        L = 1
        while L < len(path) and int(draft[path[L]]) == int(am[path[L - 1]]):
            L += 1
        k, end = L - 1, path[L - 1]
        if k > best_k or (k == best_k and end < best_end):
            best_k, best_end = k, end
    path, j = [], best_end
    while j != -1:
        path.append(j)
        j = int(parents[j])
    path.reverse()
    tokens = [int(draft[c]) for c in path[1:]] + [int(am[best_end])]
    return best_k, path, tokens


def commit(w, accepted):
    """Expected cache after accept(k): copies of k_cache / v_cache with, for
    every sequence b, rows P_b .. P_b+k_b replaced by the tree K/V rows of
    the accepted path nodes (in path order), plus the new prefix lengths.
    A sequence whose P_b+k_b+1 exceeds its capacity is left untouched.
    `accepted` = list of (k, path, tokens) per sequence."""
    kc, vc = w.k_cache.clone(), w.v_cache.clone()
    new_p = w.prefix_len.clone()
    for b, (k, path, _tok) in enumerate(accepted):
        P = int(w.prefix_len[b])
        o0, _ = w.seq_rows(b)
        if P + k + 1 > seq_capacity(w, b):
            continue
        for t, node in enumerate(path):
            pos = P + t
            if w.page_table is None:
                kc[b, :, pos] = w.k_tree[:, o0 + node]
                vc[b, :, pos] = w.v_tree[:, o0 + node]
            else:
                pid = int(w.page_table[b, pos // PAGE_SIZE])
                kc[pid, :, pos % PAGE_SIZE] = w.k_tree[:, o0 + node]
                vc[pid, :, pos % PAGE_SIZE] = w.v_tree[:, o0 + node]
        new_p[b] = P + k + 1
    return kc, vc, new_p


def seq_capacity(w, b):
    """Tokens sequence b can hold: the cache's row count (contiguous) or the
    allocated pages of its page-table row times the page size (paged)."""
    if w.page_table is None:
        return w.capacity
    row = w.page_table[b]
    return int((row >= 0).sum()) * PAGE_SIZE


def verify_step(w, samples=None):
    """The whole step on one workload: attention, per-node argmax,
    acceptance and the committed cache."""
    out = tree_attention(w, samples)
    am = argmax_rows(w.logits)
    acc = []
    for b in range(w.batch):
        o0, o1 = w.seq_rows(b)
        acc.append(accept(w.parents[b], w.draft_tokens[o0:o1].tolist(), am[o0:o1].tolist()))
    kc, vc, new_p = commit(w, acc)
    return dict(out=out, argmax=am, accepted=acc, k_cache=kc, v_cache=vc, prefix_len=new_p)
