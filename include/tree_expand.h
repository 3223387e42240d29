/*
 * tree_expand.h — C ABI of dynamic draft-tree expansion (EAGLE-2 style) on
 * NVIDIA GB300 (sm_103a): the step that builds the tree tree_verify.h
 * verifies.
 *
 * What it computes ("ADR-037 — EAGLE-3 with dynamic tree port", phase rows
 * E4a and E4b.10a, §4 Phase E4):
 *
 *   A pool of pending candidates, each keyed by its cumulative log
 *   probability (float64: the parent's plus its own log-probability under the
 *   drafter).  The root (depth 0, cumulative 0) is expanded first.  Each step
 *   moves the best pending candidates into the tree, at most `width` (W) of
 *   them and never more than the budget of `max_nodes` (N) nodes, root
 *   included; the nodes moved in one step are expanded together by the next
 *   step, each adding its top-K children to the pool (none at the depth
 *   limit).  Best = largest cumulative log-probability; equal values go to
 *   the candidate generated first (in order of step, expanded node, top-K
 *   rank).  W = 1 is the pages' global best-first expansion, in which a
 *   grandchild of A can enter the tree before a sibling of A.
 *
 *   Top-K of a node's draft logits: the K largest, largest first, equal
 *   values in increasing token order (the smaller token wins ties), compared
 *   as the raw logits (never a rounded or clamped copy); NaN is never chosen.
 *   Log-probability of token v: logit[v] - log sum_u exp(logit[u]) over the
 *   non-NaN entries (computed with the maximum subtracted).  Precision: the
 *   exponentials are summed in float32 per thread and in float pairs (hi +
 *   lo, about 48 significant bits) above that; the log is M + e*ln2 (exact
 *   split) + logf(mantissa), within about 1e-7; cumulative values are float
 *   pairs inside the kernels and float64 in d_cum.
 *
 * The drafter is the caller's: between two steps it computes the draft
 * logits of the nodes the previous step moved into the tree.
 *
 * Conventions are those of tree_verify.h: caller-owned device buffers
 * (d_ prefix), 16-byte aligned device pointers, host errors as TV_ERR_*
 * before anything is enqueued, device-only faults OR-ed into *d_status as
 * TV_DEV_* bits, nothing allocated or synchronised, deterministic results.
 */
#ifndef TREE_EXPAND_H
#define TREE_EXPAND_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* device status bits of the expansion (OR-ed into *d_status; the
 * TV_DEV_* bits of tree_verify.h use 1..32) */
enum {
  TV_DEV_BAD_LOGITS = 64,  /* a draft-logit row holds +inf: that node gets no children */
  TV_DEV_BAD_STEP = 128    /* a step >= 1 on a workspace that step - 1 did not leave: nothing written */
};

typedef struct tv_expand_desc {
  int32_t batch;          /* B >= 1 independent trees */
  int32_t vocab;          /* V draft vocabulary, 1..2^30 */
  int32_t top_k;          /* K children per expanded node, 1..16 */
  int32_t width;          /* W nodes moved per step (and expanded by the next step), 1..16 */
  int32_t max_nodes;      /* N nodes per tree, root included, 1..64 (the mask of tree_verify.h holds 64) */
  int32_t max_depth;      /* deepest depth a node may have, >= 1 */
  int32_t logits_dtype;   /* TV_F32 or TV_BF16 (tree_verify.h) */
} tv_expand_desc;

/* Bytes of scratch tv_tree_expand_step needs (256-byte aligned, reused for
 * every step of one expansion; it carries the pool from step to step, so
 * one workspace serves one expansion at a time). */
int tv_expand_workspace_size(const tv_expand_desc* desc, size_t* bytes);

/* Steps after which every tree holds N nodes when neither the depth limit
 * nor rows without valid logits stop it early (step 0 included).  Each step
 * moves min(W, pending, N - size) nodes; pending starts at min(K, V) and
 * grows by K per expanded node.  With a binding depth limit a tree may stop
 * below N; further steps then do nothing. */
int tv_expand_steps(const tv_expand_desc* desc, int32_t* steps);

/* One step of the expansion for every tree b.
 *
 *  step 0: starts tree b: node 0 = root with token d_root_tokens[b],
 *          parent -1, depth 0, cumulative 0; entries 1..N-1 of the outputs
 *          are set to -1 (cum to -inf).  Then it expands the root with its
 *          draft logits (one row per tree) and moves the best candidates.
 *  step s >= 1: expands the nodes step s - 1 moved (the j-th of them reads
 *          row j), then moves the best candidates.  It must follow step s - 1
 *          on the same workspace and outputs (else TV_DEV_BAD_STEP for that
 *          tree and nothing is written).  A tree that is complete does
 *          nothing.
 *
 *   d_logits       draft logits (logits_dtype): row j of tree b starts at
 *                  element b * seq_stride + j * V; step 0 reads row 0 of each
 *                  tree, later steps rows 0..W-1 (rows beyond
 *                  d_expand_count[b] of the previous step are ignored).
 *                  seq_stride >= V at step 0 and >= W * V after.
 *   d_root_tokens  [B] int32, read at step 0 only (may be NULL after).
 *   d_token_map    NULL, or [V] int32: a child drawn at draft index v gets
 *                  token d_token_map[v] (a reduced draft vocabulary mapped to
 *                  target tokens); ties are still broken by v.
 *   d_tokens, d_parents, d_depths  [B, N] int32 (out, kept across steps):
 *                  the tree in the order nodes entered it, root first, so
 *                  parents[i] < i; tree_verify.h takes d_parents directly.
 *   d_cum          [B, N] float64 (out): cumulative log-probabilities.
 *   d_n_nodes      [B] int32 (out): nodes in tree b so far.
 *   d_expand_count [B] int32 (out): nodes the next step expands, i.e. rows
 *                  of d_logits the drafter must fill for tree b (0 once the
 *                  tree is complete); they are nodes
 *                  [d_n_nodes - d_expand_count, d_n_nodes).
 *
 * Enqueues two kernels; step 0 also enqueues a memset of 4 * B * W bytes of
 * the workspace (per-row counters that later steps find at zero again).
 *
 * Errors: TV_ERR_NULL, TV_ERR_DTYPE, TV_ERR_SHAPE (a descriptor field, step
 * or seq_stride out of range), TV_ERR_OVERFLOW, TV_ERR_WORKSPACE,
 * TV_ERR_ALIGN, TV_ERR_CUDA, as in tree_verify.h. */
int tv_tree_expand_step(const tv_expand_desc* desc, int32_t step, const void* d_logits, int64_t seq_stride,
                        const int32_t* d_root_tokens, const int32_t* d_token_map, int32_t* d_tokens,
                        int32_t* d_parents, int32_t* d_depths, double* d_cum, int32_t* d_n_nodes,
                        int32_t* d_expand_count, void* d_workspace, size_t workspace_bytes,
                        int32_t* d_status, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* TREE_EXPAND_H */
