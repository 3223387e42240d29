// Internal declarations shared by the CUDA translation units of the
// tree-verify library.  Not part of the C ABI (include/tree_verify.h is).
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include "tree_verify.h"

namespace tv {

constexpr int kPageSize = 16;
constexpr int kMaxNodes = 64;
constexpr int kNumSMsDefault = 148;
constexpr int kMaxVChunks = 32;      // vocabulary chunks per row in the argmax pass

// Everything the split-KV attention kernels read, resolved on the host.
struct AttnParams {
  const void* q;             // [R, Hq, d]
  const void* k_cache;       // contiguous [B, Hkv, cap, d] or paged [pages, Hkv, 16, d]
  const void* v_cache;
  const int32_t* page_table; // [B, max_pages] or nullptr
  const int32_t* prefix_len; // [B]
  const int32_t* node_offsets;  // [B+1]
  const void* k_tree;        // [Hkv, R, d]
  const void* v_tree;
  const uint64_t* anc;       // [R]
  float* o_part;             // [tiles, tile_stride, d]  unnormalised partial output, tile-major:
                             // tile = ((split * B + b) * Hkv + g) * row_tiles + row_tile
  float2* ml_part;           // [tiles, tile_stride]     (running max in log2 units, running sum)
  void* out;                 // [R, Hq, d] or nullptr: a sequence with one key chunk writes its
                             // normalised rows here instead of partials (the merge skips it)
  int out_bf16;
  int32_t* status;
  int B, Hq, Hkv, G, d, R, max_nodes;
  int paged;
  int64_t capacity, num_pages, max_pages, max_prefix;
  float scale_log2;          // softmax scale * log2(e): scores are kept in base-2 units
  int chunk;                 // keys per split (multiple of the kernel's key tile)
  int splits;                // splits in the grid (covers max_prefix)
  int rows_per_tile;         // query rows per row tile (node x group head)
  int row_tiles;
  int tile_stride;           // partial rows reserved per tile (>= rows_per_tile)
};

// Partial-row index of query row m_in of row tile rt of (split, b, g).
__host__ __device__ inline int64_t partial_row(int split, int b, int g, int rt, int m_in, int B, int Hkv,
                                               int row_tiles, int tile_stride) {
  return ((((int64_t)split * B + b) * Hkv + g) * row_tiles + rt) * tile_stride + m_in;
}

struct MergeParams {
  const int32_t* prefix_len;
  const int32_t* node_offsets;
  const float* o_part;
  const float2* ml_part;
  void* out;
  int32_t* status;
  int B, Hq, d, R, max_nodes, out_bf16;
  int skip_single;           // rows of one-chunk sequences were written by the split pass
  int Hkv, G, rows_per_tile, row_tiles, tile_stride;
  int64_t max_prefix, capacity;
  int chunk, splits;
};

// Number of key chunks sequence b is split into, from its (clamped) prefix
// length.  The last chunk also takes the tree keys.  Host and device use the
// same formula so the merge reads exactly the partials the split pass wrote.
__host__ __device__ inline int num_chunks(int64_t P, int chunk) {
  int64_t n = (P + chunk - 1) / chunk;
  return n < 1 ? 1 : (int)n;
}

__host__ __device__ inline int64_t clamp_prefix(int64_t P, int64_t max_prefix, int64_t capacity) {
  int64_t hi = max_prefix < capacity ? max_prefix : capacity;
  return P < 0 ? 0 : (P > hi ? hi : P);
}

__device__ inline void set_status(int32_t* status, int bits) {
  if (status) atomicOr(status, bits);
}

// Reads node_offsets for sequence b with every check the kernels need:
// returns false (and flags TV_DEV_BAD_OFFSETS) when the sequence's rows are
// not a valid range, in which case the caller skips the sequence.
__device__ inline bool seq_rows(const int32_t* offs, int b, int R, int max_nodes, int32_t* status,
                                int* o0, int* n) {
  int a = offs[b], c = offs[b + 1];
  int cnt = c - a;
  if (a < 0 || cnt < 1 || cnt > max_nodes || c > R || (b == 0 && a != 0)) {
    set_status(status, TV_DEV_BAD_OFFSETS);
    return false;
  }
  *o0 = a;
  *n = cnt;
  return true;
}

// Launchers (return cudaError_t of the launch).
cudaError_t launch_attn_simt(const AttnParams& p, int dtype, cudaStream_t s);
cudaError_t launch_attn_tc(const AttnParams& p, cudaStream_t s);
cudaError_t launch_attn_tc2(const AttnParams& p, cudaStream_t s);
cudaError_t launch_merge(const MergeParams& p, cudaStream_t s);
cudaError_t launch_tree_mask(const int32_t* parents, const int32_t* offs, uint64_t* anc, int32_t* depth,
                             int32_t* status, int B, int R, int max_nodes, cudaStream_t s);

struct AcceptParams {
  const void* logits;        // [R, V]
  int logits_bf16;
  int V;
  const int32_t* draft;
  const int32_t* parents;
  const int32_t* node_offsets;
  const void* k_tree;
  const void* v_tree;
  void* k_cache;
  void* v_cache;
  const int32_t* page_table;
  int32_t* prefix_len;
  int32_t* argmax;
  int32_t* accept_len;
  int32_t* path;
  int32_t* tokens;
  float* am_val;             // workspace [R, vchunks]
  int32_t* am_idx;           // workspace [R, vchunks]
  int32_t* status;
  int B, R, Hkv, d, esize, max_nodes, paged;
  int64_t capacity, num_pages, max_pages;
  int vchunks;               // vocab chunks per row in the argmax pass
  int vchunk_len;            // elements per chunk (multiple of 8)
};

cudaError_t launch_accept_commit(const AcceptParams& p, cudaStream_t s);

// tcgen05 kernel availability for a descriptor (head_dim, group size).
bool tc_supported(const tv_desc* d, int G);
int tc_key_tile(int d);

}  // namespace tv
