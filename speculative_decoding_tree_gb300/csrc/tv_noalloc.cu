// tree_verify_attn without a caller workspace, for callers that cannot
// allocate device memory (a plugin given only its input and output buffers,
// or a loop where cudaMalloc's possible device synchronisation is not
// allowed).  The split-KV partials live in a file-scope device array instead.
//
// In host code `g_noalloc_scratch` names a host-side stand-in, not device
// memory: its device address is looked up with cudaGetSymbolAddress (the
// caller's device current) on every call and passed to the kernels.  The
// lookup allocates nothing once this file's module is loaded; it is not
// cached, so that a context torn down and made again (cudaDeviceReset)
// never leaves a stale address behind.
#include "tv_internal.cuh"

namespace {

static __device__ __align__(256) unsigned char g_noalloc_scratch[TV_NOALLOC_SCRATCH_BYTES];

// Device address of the scratch array in the current context, or nullptr
// when the lookup fails.
void* scratch_on_current_device() {
  void* ptr = nullptr;
  if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess) return nullptr;
  return ptr;
}

}  // namespace

extern "C" int tree_verify_attn_noalloc(const tv_desc* desc, const void* d_q, const void* d_k_cache,
                                        const void* d_v_cache, const int32_t* d_page_table,
                                        const int32_t* d_prefix_len, const int32_t* d_node_offsets,
                                        const void* d_k_tree, const void* d_v_tree, const uint64_t* d_anc,
                                        void* d_out, int32_t* d_status, void* stream) {
  void* scratch = scratch_on_current_device();
  if (!scratch) {
    cudaGetLastError();
    return TV_ERR_CUDA;
  }
  // tree_verify_attn checks the descriptor, the pointers and that the plan's
  // partials fit TV_NOALLOC_SCRATCH_BYTES (TV_ERR_WORKSPACE otherwise)
  return tree_verify_attn(desc, d_q, d_k_cache, d_v_cache, d_page_table, d_prefix_len, d_node_offsets, d_k_tree,
                          d_v_tree, d_anc, d_out, scratch, TV_NOALLOC_SCRATCH_BYTES, d_status, stream);
}
