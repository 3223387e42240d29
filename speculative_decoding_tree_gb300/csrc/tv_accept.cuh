// Parameters of the acceptance kernels (argmax or sampled draw, then the
// walk and commit), resolved on the host.  Internal to the library.
#pragma once
#include "tv_internal.cuh"

namespace tv {

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
  int sampled;               // draw per row (Gumbel-max) instead of the argmax
  float inv_temp;            // 1 / temperature (sampled)
  uint32_t seed_lo, seed_hi, off_lo, off_hi;   // Philox key and counter words 2, 3 (sampled)
  int given_argmax;          // argmax is an input (no logits pass): only the walk and commit run
  int stage_bytes;           // shared memory per walk block for its staged tree rows (0: copy from the tree buffers)
};

// Blocks per sequence in the walk and commit: one per (K or V, KV head) set
// of rows, at most 8 (a portable cluster).
inline int walk_cluster(int Hkv) { return 2 * Hkv < 8 ? 2 * Hkv : 8; }

// Shared memory a walk block needs to stage its sets' tree rows (max_nodes
// rows of row_bytes per set), or 0 when that exceeds the staging budget.
inline int walk_stage_bytes(int Hkv, int max_nodes, int64_t row_bytes) {
  constexpr int64_t kStageBudget = 160 * 1024;
  const int C = walk_cluster(Hkv);
  const int64_t sets = (2 * (int64_t)Hkv + C - 1) / C;
  const int64_t bytes = sets * max_nodes * row_bytes;
  return bytes <= kStageBudget ? (int)bytes : 0;
}

cudaError_t launch_accept_commit(const AcceptParams& p, cudaStream_t s);

}  // namespace tv
