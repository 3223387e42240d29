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
};

cudaError_t launch_accept_commit(const AcceptParams& p, cudaStream_t s);

}  // namespace tv
