/*
 * tree_verify.h — C ABI of the tree-verify step of tree speculative decoding
 * (EAGLE / Medusa style) on NVIDIA GB300 (sm_103a).
 *
 * The step has two halves, each one call:
 *
 *   tree_verify_attn    attention for every draft-tree query row over the
 *                       committed prefix KV cache plus the tree's own K/V,
 *                       each node seeing the whole prefix, its ancestors and
 *                       itself ("ADR-037 — EAGLE-3 with dynamic tree port",
 *                       §4 Phase E1, and phase rows E1.1-E1.5).
 *   tree_accept_commit  per-node argmax over the vocabulary, the walk for
 *                       the longest path whose drafts match the target
 *                       argmax plus one bonus/correction token (ADR-037 row
 *                       E5a, Phase E5), and the delayed write-through
 *                       accept(k) that copies only the accepted rows' K/V
 *                       into the cache ("Speculative decoding verify
 *                       batches to amortize ANE dispatch", commit-rule and
 *                       KV write-before-accept bullets).
 *
 * plus the mask build they share (tv_build_tree_mask), the two halves of the
 * split-KV attention (tv_attn_partials / tv_attn_merge), and small queries.
 *
 * Conventions for every entry point
 * ---------------------------------
 * - Pointers prefixed d_ are device pointers; the caller allocates and owns
 *   every buffer.  The library never allocates, frees or synchronises: it
 *   validates on the host, enqueues kernels on `stream` (a cudaStream_t
 *   passed as void*, NULL = legacy default stream) and returns.
 * - Device pointers must be 16-byte aligned (TV_ERR_ALIGN otherwise).
 * - Return value: TV_OK (0) or a negative TV_ERR_* found on the host BEFORE
 *   anything is enqueued (then nothing is enqueued), or TV_ERR_CUDA when a
 *   launch fails.  tv_status_string() names every code.
 * - Faults that only the device can see (a bad parent pointer, a bad node
 *   offset, a prefix length or page id out of range, a commit that does not
 *   fit) are OR-ed into *d_status as TV_DEV_* bits; the affected work is
 *   skipped or clamped, and nothing traps.  The caller zeroes d_status and
 *   reads it whenever it synchronises.
 * - Results are deterministic: the same inputs give the same output bytes.
 *   The split-KV partition depends only on the descriptor and the device
 *   prefix lengths, never on occupancy, and no float atomics are used.
 *
 * Layouts (row-major, innermost last)
 * -----------------------------------
 *   B sequences; sequence b owns tree rows [node_offsets[b], node_offsets[b+1])
 *   (N_b = node count, 1 <= N_b <= max_nodes <= 64, row 0 of each = root);
 *   total_rows = sum N_b.  Hq query heads, Hkv KV heads, G = Hq / Hkv;
 *   query head h reads KV head h / G (contiguous groups).  d = head_dim.
 *
 *   q            [total_rows, Hq, d]        dtype
 *   k/v tree     [Hkv, total_rows, d]       dtype   (this round's node K/V)
 *   k/v cache    contiguous: [B, Hkv, capacity, d]          dtype
 *                paged:      [num_pages, Hkv, 16, d]        dtype, with
 *                page_table  [B, capacity / 16] int32, position t of sequence
 *                b at page page_table[b][t / 16], slot t % 16
 *   prefix_len   [B] int32, committed tokens per sequence (P_b)
 *   parents      [total_rows] int32, local index of the parent within the
 *                sequence (-1 for the root, else 0 <= parent < own index)
 *   out          [total_rows, Hq, d]  (row r, head h at r*Hq + h: the
 *                [q_seq_len, num_heads, head_dim] layout of ADR-037 row E1.3)
 *   logits       [total_rows, vocab]  fp32 or bf16
 *
 * Positions: tree node i of sequence b carries position P_b + depth(i)
 * (RoPE is the caller's).  The committed row t sits at P_b + t, which is the
 * depth of the t-th path node, so committed K need no re-rotation.
 */
#ifndef TREE_VERIFY_H
#define TREE_VERIFY_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---------------------------------------------------------------- codes */

typedef enum {
  TV_F32 = 0,   /* IEEE fp32 */
  TV_BF16 = 1   /* bfloat16 */
} tv_dtype;

enum {
  TV_OK = 0,
  TV_ERR_NULL = -1,        /* a required pointer (or the descriptor) is NULL */
  TV_ERR_DTYPE = -2,       /* dtype / logits dtype not TV_F32 or TV_BF16 */
  TV_ERR_HEAD_DIM = -3,    /* head_dim not 128, 256 or 512 */
  TV_ERR_ZERO_HEADS = -4,  /* num_q_heads or num_kv_heads <= 0 (checked before the modulo) */
  TV_ERR_GQA = -5,         /* num_q_heads % num_kv_heads != 0 */
  TV_ERR_SHAPE = -6,       /* batch, total_rows, vocab, capacity or max_prefix out of range, or a launch
                              grid extent above 65535: batch, KV heads x splits, KV heads x row tiles,
                              or total_rows for acceptance */
  TV_ERR_TREE = -7,        /* max_nodes outside 1..64, or total_rows outside batch..batch*max_nodes */
  TV_ERR_PAGED = -8,       /* page_size not 0 or 16, capacity not a multiple of 16, or no pages */
  TV_ERR_OVERFLOW = -9,    /* a byte count overflows int64 */
  TV_ERR_WORKSPACE = -10,  /* workspace smaller than tv_workspace_size() */
  TV_ERR_ALIGN = -11,      /* a device pointer is not 16-byte aligned */
  TV_ERR_CUDA = -12        /* a CUDA launch failed */
};

/* bits OR-ed into *d_status by the kernels */
enum {
  TV_DEV_BAD_TREE = 1,     /* parents[root] != -1 or a parent outside [0, own index) */
  TV_DEV_BAD_OFFSETS = 2,  /* node_offsets not starting at 0, N_b outside 1..max_nodes, or sum != total_rows */
  TV_DEV_BAD_PREFIX = 4,   /* prefix_len[b] < 0, > max_prefix or > capacity (clamped) */
  TV_DEV_BAD_PAGE = 8,     /* a page-table entry outside [0, num_pages) (page read as zeros / commit skipped) */
  TV_DEV_CAPACITY = 16,    /* accept(k) skipped: prefix_len + k + 1 > capacity */
  TV_DEV_TIMEOUT = 32      /* a kernel's bounded wait ran out (internal error; results invalid) */
};

/* ----------------------------------------------------------- descriptor */

typedef struct tv_desc {
  int32_t batch;          /* B >= 1 */
  int32_t num_q_heads;    /* Hq >= 1 */
  int32_t num_kv_heads;   /* Hkv >= 1, Hq % Hkv == 0 */
  int32_t head_dim;       /* d: 128, 256 or 512 */
  int32_t dtype;          /* tv_dtype of q, tree K/V and cache */
  int32_t out_f32;        /* bf16 inputs: 1 = write fp32 out, 0 = bf16 out. fp32 inputs: fp32 out */
  float   scale;          /* softmax scale; 0 = 1/sqrt(head_dim) */
  int32_t max_nodes;      /* upper bound on N_b, 1..64 */
  int32_t total_rows;     /* sum over b of N_b */
  int32_t page_size;      /* 0 = contiguous cache, 16 = paged cache */
  int64_t capacity;       /* tokens one sequence can hold: contiguous = cache rows per (b, head);
                             paged = page-table columns * 16 */
  int64_t num_pages;      /* paged: pages in the pool; ignored when contiguous */
  int64_t max_prefix;     /* host upper bound on every prefix_len[b] (sizes the grid only) */
} tv_desc;

/* How tree_verify_attn will run a descriptor (for inspection and for
 * counting algorithmic work; filled by tv_attn_plan). */
typedef struct tv_plan {
  int32_t kernel;         /* 0 = CUDA-core split kernel, 1 = tcgen05 kernel (one CTA per query tile),
                             2 = tcgen05 kernel on CTA pairs (two query tiles share each K/V tile),
                             3 = persistent tcgen05 kernel on CTA pairs for batches at head_dim 128
                             (units of (sequence, KV head, two query tiles, chunk) from a counter) */
  int32_t num_splits;     /* KV chunks per (sequence, KV head) at the longest prefix */
  int32_t chunk;          /* keys per chunk (the last chunk of a sequence also takes its tree keys) */
  int32_t row_tiles;      /* query-row tiles per (sequence, KV head) */
  int32_t rows_per_tile;  /* query rows (node x group head) per tile */
  int32_t grid_ctas;      /* CTAs launched by the split kernel */
} tv_plan;

/* ------------------------------------------------------------- queries */

/* Bytes of scratch that tree_verify_attn, tv_attn_partials/_merge and
 * tree_accept_commit need for this descriptor and vocabulary (vocab may be 0
 * when only attention is used).  The caller allocates it once (256-byte
 * aligned) and may reuse it across calls on the same stream; its contents
 * need no initialisation.  Returns TV_OK or a TV_ERR_* for a bad descriptor. */
int tv_workspace_size(const tv_desc* desc, int32_t vocab, size_t* bytes);

/* Fill *plan with the launch plan tree_verify_attn uses for desc. */
int tv_attn_plan(const tv_desc* desc, tv_plan* plan);

/* Static name of a TV_OK / TV_ERR_* code or of a single TV_DEV_* bit
 * (pass the bit as a positive value); "unknown" otherwise. */
const char* tv_status_string(int code);

/* Library version string, e.g. "treeverify 0.1 sm_103a". */
const char* tv_version(void);

/* Failure detection check: launches one CTA whose thread waits, with the
 * bounded wait every tensor-core kernel of the library uses, on a shared
 * memory barrier that nothing completes.  After limit_ns (1 ms .. 10 s) of
 * GPU time the wait gives up, the kernel ORs TV_DEV_TIMEOUT into *d_status
 * and ends; the context stays usable.  Returns TV_ERR_SHAPE for a limit out
 * of range, TV_ERR_NULL / TV_ERR_ALIGN for d_status, TV_ERR_CUDA if the
 * launch fails, else TV_OK. */
int tv_check_bounded_wait(int64_t limit_ns, int32_t* d_status, void* stream);

/* ------------------------------------------------------- A0: tree mask */

/* For every node i of every sequence: d_anc[row] has bit j set iff j == i or
 * j is an ancestor of i (j local index), and d_depth[row] = number of edges
 * to the root.  A row whose parent chain is invalid gets only its own bit
 * and TV_DEV_BAD_TREE.  Mask rule: ADR-037 §4 Phase E1 (mask encoding) and
 * row E6 v2 (ancestors + self); a uint64 per row replaces the pages' f32
 * [seq+tree, tree] mask for trees of at most 64 nodes.
 *   d_parents [total_rows] int32, d_node_offsets [B+1] int32,
 *   d_anc [total_rows] uint64 (out), d_depth [total_rows] int32 (out, may be NULL). */
int tv_build_tree_mask(const tv_desc* desc, const int32_t* d_parents, const int32_t* d_node_offsets,
                       uint64_t* d_anc, int32_t* d_depth, int32_t* d_status, void* stream);

/* ------------------------------------------------- A1+A2: attention */

/* out[r, h, :] = sum_j softmax_j(scale * q[r,h,:] . k_j) v_j over the keys
 * j visible to row r: every prefix position 0..P_b-1 of its sequence and
 * every tree node in d_anc[r] (from tv_build_tree_mask).  fp32 inputs are
 * computed in fp32 (no TF32); bf16 inputs are multiplied in bf16 with fp32
 * accumulation and an fp32 softmax.  d_page_table is NULL for a contiguous
 * cache.  The cache is only read.  Runs tv_attn_partials then tv_attn_merge.
 * ADR-037 phase rows E1.1-E1.5 and E4b.6 (tree attention as flash-decode
 * with a reduce kernel merging the split-KV partials). */
int tree_verify_attn(const tv_desc* desc, const void* d_q, const void* d_k_cache, const void* d_v_cache,
                     const int32_t* d_page_table, const int32_t* d_prefix_len,
                     const int32_t* d_node_offsets, const void* d_k_tree, const void* d_v_tree,
                     const uint64_t* d_anc, void* d_out, void* d_workspace, size_t workspace_bytes,
                     int32_t* d_status, void* stream);

/* First half of tree_verify_attn: the split-KV pass.  For every chunk of
 * keys it leaves in the workspace the unnormalised partial output, the
 * running maximum and the running sum of that chunk (the partials a second
 * GPU holding another range of the prefix would exchange). */
int tv_attn_partials(const tv_desc* desc, const void* d_q, const void* d_k_cache, const void* d_v_cache,
                     const int32_t* d_page_table, const int32_t* d_prefix_len,
                     const int32_t* d_node_offsets, const void* d_k_tree, const void* d_v_tree,
                     const uint64_t* d_anc, void* d_workspace, size_t workspace_bytes,
                     int32_t* d_status, void* stream);

/* Second half: the log-sum-exp merge of the partials left by
 * tv_attn_partials (same descriptor, prefix lengths and workspace) into
 * d_out, cast to the output dtype.  The pages' "reduce kernel" (ADR-037 rows
 * E1.2 and E4b.6). */
int tv_attn_merge(const tv_desc* desc, const int32_t* d_prefix_len, const int32_t* d_node_offsets,
                  void* d_out, const void* d_workspace, size_t workspace_bytes, int32_t* d_status,
                  void* stream);

/* ------------------------------------------- A3+A4+A5: accept + commit */

/* Greedy acceptance and delayed write-through, per sequence b:
 *  1. d_argmax[r] = argmax over v of logits[r, v]; the smallest index wins
 *     ties, NaN never wins, an all-NaN row gives 0 (ADR-037 row E4b.10a
 *     fixes this tie rule for top-K; it is used here for argmax).
 *  2. node c (c > 0) matches when draft[c] == argmax[parent(c)]; the
 *     accepted path is the deepest node whose whole root path matches (ties:
 *     smallest node index); k = its depth (ADR-037 row E5a and Phase E5
 *     edge cases; the ANE page's commit-rule bullet).
 *     d_accept_len[b] = k; d_path[b, 0..k] = the path's local node indices;
 *     d_tokens[b, 0..k] = drafts of path[1..k] then argmax[path[k]] (the
 *     bonus or correction token); both rows are -1 padded to max_nodes.
 *  3. if P_b + k + 1 <= capacity (and every page needed is valid): for
 *     t = 0..k copy tree K/V row path[t] (all KV heads) to cache position
 *     P_b + t, then prefix_len[b] = P_b + k + 1.  No other cache byte is
 *     written, so rejected drafts never touch the cache (the ANE page's
 *     KV write-before-accept bullet and Forge's accept(k)).  Otherwise the
 *     cache and prefix_len are left as they were and TV_DEV_CAPACITY (or
 *     TV_DEV_BAD_PAGE) is set.
 *   d_logits [total_rows, vocab] (logits_dtype), d_draft_tokens [total_rows]
 *   int32 (the root's entry is ignored), d_parents [total_rows] int32,
 *   d_prefix_len in/out, d_argmax [total_rows] int32 out, d_accept_len [B]
 *   out, d_path and d_tokens [B, max_nodes] int32 out. */
int tree_accept_commit(const tv_desc* desc, int32_t vocab, int32_t logits_dtype, const void* d_logits,
                       const int32_t* d_draft_tokens, const int32_t* d_parents,
                       const int32_t* d_node_offsets, const void* d_k_tree, const void* d_v_tree,
                       void* d_k_cache, void* d_v_cache, const int32_t* d_page_table,
                       int32_t* d_prefix_len, int32_t* d_argmax, int32_t* d_accept_len,
                       int32_t* d_path, int32_t* d_tokens, void* d_workspace, size_t workspace_bytes,
                       int32_t* d_status, void* stream);

/* Sampled verification (temperature > 0): the same walk, outputs and commit
 * as tree_accept_commit, with step 1's argmax replaced by one draw per tree
 * row from the target distribution softmax(logits[r, :] / temperature).
 * The rule ("Speculative decoding verify batches to amortize ANE dispatch",
 * Forge sampled-proposal bullet; "Speculative-decoding heads", What's not
 * implemented (7)): a drafted proposal is accepted with its target
 * probability, and on rejection the target distribution with the proposal
 * excluded is sampled.  Drawing y_u from p_u at an accepted node u and
 * accepting the child whose draft equals y_u is that rule (child by child,
 * for siblings with distinct drafts); if no child matches, y_u is the
 * correction token.  The emitted tokens therefore follow the target model's
 * distribution whatever the drafts propose.
 *   The draw: d_sampled[r] = argmax over v of logits[r, v] / temperature +
 *   G(r, v), G = -log(-log U), U = ((x >> 9) + 0.5) * 2^-23 with x word v % 4
 *   of Philox4x32-10 (Salmon et al., SC 2011) at counter (v / 4, r,
 *   offset low, offset high) and key (seed low, seed high); NaN logits are
 *   never drawn; computed in float32.  Pass a new offset (or seed) for every
 *   step to draw fresh noise; the same (seed, offset) gives the same draws.
 *   temperature must be finite and > 0 (TV_ERR_SHAPE otherwise); every other
 *   argument, the workspace and the errors are as for tree_accept_commit, with
 *   d_sampled in place of d_argmax. */
int tree_accept_commit_sampled(const tv_desc* desc, int32_t vocab, int32_t logits_dtype, const void* d_logits,
                               float temperature, uint64_t seed, uint64_t offset, const int32_t* d_draft_tokens,
                               const int32_t* d_parents, const int32_t* d_node_offsets, const void* d_k_tree,
                               const void* d_v_tree, void* d_k_cache, void* d_v_cache, const int32_t* d_page_table,
                               int32_t* d_prefix_len, int32_t* d_sampled, int32_t* d_accept_len, int32_t* d_path,
                               int32_t* d_tokens, void* d_workspace, size_t workspace_bytes, int32_t* d_status,
                               void* stream);

/* Steps 2 and 3 of tree_accept_commit with the target argmax given instead
 * of logits, e.g. from tv_lm_head_argmax (tree_lm_head.h), which never
 * writes the logits: d_argmax [total_rows] int32 is read (not written) and
 * every other argument, output and error is as for tree_accept_commit.  No
 * workspace is used. */
int tree_accept_commit_argmax(const tv_desc* desc, const int32_t* d_argmax, const int32_t* d_draft_tokens,
                              const int32_t* d_parents, const int32_t* d_node_offsets, const void* d_k_tree,
                              const void* d_v_tree, void* d_k_cache, void* d_v_cache, const int32_t* d_page_table,
                              int32_t* d_prefix_len, int32_t* d_accept_len, int32_t* d_path, int32_t* d_tokens,
                              int32_t* d_status, void* stream);

/* ------------------------------------- attention without a workspace */

/* Size in bytes of the library's static scratch array (file-scope device
 * memory) that tree_verify_attn_noalloc uses instead of a caller workspace. */
#define TV_NOALLOC_SCRATCH_BYTES (32u << 20)

/* tree_verify_attn for callers that cannot allocate device memory: a
 * plugin that a host framework hands only its input and output buffers, or
 * a loop that must not call cudaMalloc (it may synchronise the device).
 * The pages have no counterpart of this call; it exists for such callers.
 * Same arguments and results as tree_verify_attn minus the workspace: the
 * split-KV partials go to a static __device__ array of
 * TV_NOALLOC_SCRATCH_BYTES (32 MiB), which every GPU that loads this part of
 * the library keeps until the process exits.
 * - Returns TV_ERR_WORKSPACE, enqueuing nothing, when the descriptor needs
 *   more partials than the array holds (tv_workspace_size(desc, 0) above
 *   TV_NOALLOC_SCRATCH_BYTES).
 * - Every call looks up the array's device address in the caller's current
 *   context (`stream` must belong to that device); TV_ERR_CUDA if the lookup
 *   fails.  The address is not kept between calls, so a context torn down
 *   and made again (cudaDeviceReset) is handled.
 * - The first call on each device loads this part of the library's device
 *   code (CUDA loads modules lazily by default): that is when the driver
 *   reserves the 32 MiB array, and the load may synchronise the device.
 *   Warm up with one call (or one tv_workspace_size plus one call) before a
 *   loop that must not synchronise, and before any stream capture.
 * - Allocates nothing itself: no cudaMalloc, cudaFree or allocating library
 *   call.
 * - Every call shares the one array and it keeps the last call's contents;
 *   nothing in it needs to start at zero (each call writes every partial it
 *   reads).  Calls whose kernels overlap on the GPU (other streams, other
 *   host threads) race on the array: serialise them. */
int tree_verify_attn_noalloc(const tv_desc* desc, const void* d_q, const void* d_k_cache, const void* d_v_cache,
                             const int32_t* d_page_table, const int32_t* d_prefix_len,
                             const int32_t* d_node_offsets, const void* d_k_tree, const void* d_v_tree,
                             const uint64_t* d_anc, void* d_out, int32_t* d_status, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* TREE_VERIFY_H */
