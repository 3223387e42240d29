/*
 * tree_rope.h — C ABI of the tree-position RoPE and K/V scatter on NVIDIA
 * GB300 (sm_103a): the step between the Q/K/V projections and
 * tree_verify_attn.
 *
 * What it computes ("ADR-037 — EAGLE-3 with dynamic tree port", phase row
 * E4b.5b: rotary embedding at tree positions base_pos + tree_depths[i], NeoX
 * style over the whole head dimension; phase row E6: the seq-major to
 * head-major permute of the tree K/V): for tree row r of sequence b at
 * position p = prefix_len[b] + depth[r], and each pair j < d/2 with angle
 * p * theta^(-2j/d),
 *     out[j]       = x[j] cos - x[j + d/2] sin
 *     out[j + d/2] = x[j + d/2] cos + x[j] sin
 * applied to every query head (q_out, same [R, Hq, d] layout) and every key
 * head (k_tree, head-major [Hkv, R, d]); values are copied to v_tree
 * [Hkv, R, d] unchanged.  These are the positions tree_verify_attn and
 * tree_accept_commit assume (the committed row t sits at P + t, the depth of
 * the t-th path node), so committed K need no re-rotation.
 *
 * Precision: each angle is reduced modulo 2 pi in float64 (exact to about
 * 1e-10 rad for positions below 2^31), its sine and cosine taken in float32,
 * the rotation in float32, then rounded to the dtype (round to nearest even
 * for bf16).
 *
 * Conventions are those of tree_verify.h.  d_q_out may equal d_q_in (in
 * place); the other buffers must not overlap.
 */
#ifndef TREE_ROPE_H
#define TREE_ROPE_H

#include "tree_verify.h"

#ifdef __cplusplus
extern "C" {
#endif

/* desc: the verify descriptor (batch, heads, head_dim, dtype, max_nodes,
 * total_rows, capacity, max_prefix are used).  theta: the RoPE base, finite
 * and > 1.  d_q_in [R, Hq, d], d_k_in and d_v_in [R, Hkv, d] (dtype, seq-major
 * projection outputs); d_prefix_len [B]; d_node_offsets [B+1]; d_depth [R]
 * int32 (from tv_build_tree_mask); outputs d_q_out [R, Hq, d], d_k_tree and
 * d_v_tree [Hkv, R, d].  A row whose offsets or depth are invalid is skipped
 * (TV_DEV_BAD_OFFSETS / TV_DEV_BAD_TREE); a prefix length out of range is
 * clamped (TV_DEV_BAD_PREFIX).  Errors: those of tv_workspace_size for the
 * descriptor, TV_ERR_SHAPE for theta, TV_ERR_NULL, TV_ERR_ALIGN, TV_ERR_CUDA. */
int tv_tree_rope_scatter(const tv_desc* desc, double theta, const void* d_q_in, const void* d_k_in,
                         const void* d_v_in, const int32_t* d_prefix_len, const int32_t* d_node_offsets,
                         const int32_t* d_depth, void* d_q_out, void* d_k_tree, void* d_v_tree, int32_t* d_status,
                         void* stream);

#ifdef __cplusplus
}
#endif

#endif /* TREE_ROPE_H */
