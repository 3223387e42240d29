/*
 * tree_lm_head.h — C ABI of the fused lm_head + argmax step on NVIDIA GB300
 * (sm_103a): the target model's next-token argmax at every tree row, straight
 * from the final hidden rows, without writing the [rows, vocab] logits.
 *
 * What it computes ("ADR-037 — EAGLE-3 with dynamic tree port", phase rows
 * E4b.9 (lm_head), E5a (the target argmax at every node) and E4b.10a (the
 * smaller token wins ties)): for every row r,
 *     argmax[r] = the first (smallest) v maximising sum_k hidden[r, k] * weight[v, k]
 * over v = 0..vocab-1 (NaN never wins; a row whose logits are all NaN gives 0),
 * and optionally the largest logit itself.  bf16 inputs, products exact in
 * fp32, sums in fp32 on the tensor cores (tcgen05.mma kind::f16, fp32
 * accumulators in tensor memory); the argmax is taken on those fp32 sums.
 * tree_accept_commit takes the logits instead; this call replaces the logits'
 * write and re-read with the argmax of every tile as it leaves the tensor
 * cores.
 *
 * Conventions are those of tree_verify.h: caller-owned device buffers
 * (d_ prefix), 16-byte aligned device pointers, host errors as TV_ERR_*
 * before anything is enqueued, device-only faults OR-ed into *d_status as
 * TV_DEV_* bits (here only TV_DEV_TIMEOUT, an internal bounded wait that ran
 * out), nothing allocated or synchronised, deterministic results.
 */
#ifndef TREE_LM_HEAD_H
#define TREE_LM_HEAD_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct tv_lmhead_desc {
  int32_t rows;     /* R: tree rows, 1..2048 */
  int32_t hidden;   /* Hd: hidden size, a multiple of 64, 64..65536 */
  int32_t vocab;    /* V: vocabulary rows of the weight, >= 1 */
} tv_lmhead_desc;

/* Bytes of scratch tv_lm_head_argmax needs (per-CTA partial maxima; any
 * contents; 256-byte aligned). */
int tv_lm_head_workspace_size(const tv_lmhead_desc* desc, size_t* bytes);

/* d_hidden [R, Hd] bf16 row-major, d_weight [V, Hd] bf16 row-major (the
 * lm_head / tied embedding matrix), d_argmax [R] int32 (out), d_max_logit
 * [R] float (out, may be NULL).  Errors: TV_ERR_NULL, TV_ERR_SHAPE (rows,
 * hidden or vocab out of range), TV_ERR_OVERFLOW, TV_ERR_WORKSPACE,
 * TV_ERR_ALIGN, TV_ERR_CUDA (also when the tensor maps cannot be made). */
int tv_lm_head_argmax(const tv_lmhead_desc* desc, const void* d_hidden, const void* d_weight, int32_t* d_argmax,
                      float* d_max_logit, void* d_workspace, size_t workspace_bytes, int32_t* d_status,
                      void* stream);

#ifdef __cplusplus
}
#endif

#endif /* TREE_LM_HEAD_H */
