"""Plain float64 CPU oracle for the fused lm_head + argmax step.

TEST INFRASTRUCTURE ONLY.  Only the test suite, the package's smoke check and
the benchmark's CPU-baseline / reference leg may import this module.  It
shares no code with the CUDA path and never calls it.

What it computes ("ADR-037 — EAGLE-3 with dynamic tree port", phase rows
E4b.9 (final norm + lm_head), E5a (the target argmax at every tree node) and
E4b.10a (the smaller token wins ties)): for every tree row r, the logits
logits[r, v] = sum_k hidden[r, k] * weight[v, k] over the whole vocabulary,
in float64 from the exact bf16 inputs, and the index of the largest one, the
first (smallest) index among equal maxima; NaN is never selected.  The
logits are computed one vocabulary block at a time only to bound memory:
every logit is its own dot product, so the blocks change nothing.

Parity status: pinned by explicit loops on tiny inputs, one-hot hidden rows
(the logits are a column of the weights), planted maxima (a weight row
parallel to the hidden row wins among rows of equal norm) and duplicated
weight rows (the smaller index wins).
"""
from __future__ import annotations

import numpy as np

from .tree_verify import argmax_rows


def _f64(t):
    if hasattr(t, "double"):
        return t.double().cpu().numpy()
    return np.asarray(t, dtype=np.float64)


def lm_head_logits(hidden, weight, block=8192):
    """[R, V] float64 logits, computed in vocabulary blocks of `block` rows."""
    h = _f64(hidden)
    V = weight.shape[0]
    out = np.empty((h.shape[0], V), dtype=np.float64)
    for v0 in range(0, V, block):
        w = _f64(weight[v0:v0 + block])
        out[:, v0:v0 + w.shape[0]] = h @ w.T
    return out


def lm_head_argmax(hidden, weight, block=8192):
    """(argmax [R] int64, max logit [R] float64, gap [R] float64): the gap is
    the distance from the largest logit to the largest logit of any other
    index (inf for a one-entry vocabulary); a computation in lower precision
    agrees with this argmax when the gap is well above its rounding."""
    logits = lm_head_logits(hidden, weight, block)
    am = argmax_rows(logits)
    R = logits.shape[0]
    top = logits[np.arange(R), am]
    rest = logits.copy()
    rest[np.arange(R), am] = -np.inf
    second = np.nanmax(rest, axis=1) if logits.shape[1] > 1 else np.full(R, -np.inf)
    return am, top, top - second
