"""The one exchange a vocabulary-sharded lm_head needs: each rank holds a
slice of the vocabulary, finds its rows' largest logit and first index
(tv_lm_head_argmax on its weight slice), and the ranks combine them into the
whole vocabulary's argmax with the same tie rule (largest value, then the
smallest token: "ADR-037 — EAGLE-3 with dynamic tree port", phase rows E5a
and E4b.10a).  Two all-reduces over torch.distributed (NCCL on GPUs, gloo
on CPUs): the maximum of the values, then the minimum of the indices that
attain it.  This cross-rank step of the argmax's tie rule (a comparison per
row, the NaN-means-empty convention, the index offset) is computed here in
eager torch operations around the two collectives; within a rank the argmax
is the CUDA kernel's."""
from __future__ import annotations

import torch


def allreduce_argmax(max_logit: torch.Tensor, argmax: torch.Tensor, vocab_offset: int, group=None):
    """max_logit [R] float32 and argmax [R] int32 of this rank's vocabulary
    slice (local indices; NaN max_logit = no valid entry), vocab_offset = the
    slice's first global token.  Returns (max_logit, argmax) over the whole
    vocabulary, global indices, identical on every rank."""
    import torch.distributed as dist
    v = max_logit.to(torch.float32).clone()
    valid = ~torch.isnan(v)
    v[~valid] = -float("inf")
    dist.all_reduce(v, op=dist.ReduceOp.MAX, group=group)
    big = torch.iinfo(torch.int64).max
    idx = argmax.to(torch.int64) + int(vocab_offset)
    mine = valid & (max_logit.to(torch.float32) == v)
    cand = torch.where(mine, idx, torch.full_like(idx, big))
    dist.all_reduce(cand, op=dist.ReduceOp.MIN, group=group)
    none = cand == big                             # no rank had a valid entry
    out_v = torch.where(none, torch.full_like(v, float("nan")), v)
    out_i = torch.where(none, torch.zeros_like(cand), cand).to(torch.int32)
    return out_v, out_i
