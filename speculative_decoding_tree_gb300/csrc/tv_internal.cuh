// Internal declarations shared by the CUDA translation units of the
// tree-verify library.  Not part of the C ABI (include/tree_verify.h is).
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include <atomic>

#include "tree_verify.h"

namespace tv {

constexpr int kPageSize = 16;
constexpr int kMaxNodes = 64;
constexpr int kNumSMsDefault = 148;
constexpr int kMaxVChunks = 32;      // vocabulary chunks per row in the argmax pass
constexpr int64_t kMaxGridYZ = 65535;   // CUDA's limit on a launch grid's y and z extents

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
  float* o_part;             // [slots, d] partial output O_s / l_s at partial_slot(); fp32, or
                             // bf16 when part_bf16 (then the rows are d bf16 wide)
  float2* ml_part;           // [slots] (running max in log2 units, running sum)
  int part_bf16;             // partials stored as bf16 (tensor-core kernels with bf16 output)
  void* out;                 // [R, Hq, d] or nullptr: a sequence with one key chunk writes its
                             // normalised rows here instead of partials (the merge skips it)
  int out_bf16;
  int32_t* status;
  unsigned long long* work_counter;   // workspace word of the persistent kernel's work queue
  int B, Hq, Hkv, G, d, R, max_nodes;
  int paged;
  int64_t capacity, num_pages, max_pages, max_prefix;
  float scale_log2;          // softmax scale * log2(e): scores are kept in base-2 units
  int chunk;                 // keys per split (multiple of the kernel's key tile)
  int tree_tile;             // 0, or the key tile when the tree may take a split of its own (num_chunks)
  int splits;                // splits in the grid (covers max_prefix)
  int rows_per_tile;         // query rows per row tile (node x group head)
  int row_tiles;
  int tile_stride;           // partial rows reserved per tile (>= rows_per_tile)
};

// Slot of the partial of query row m_in of row tile rt of (sequence b, KV
// head g) from split s.  The splits of one row are adjacent, and the rows of
// a row tile follow each other, so the partials a merge CTA combines (a slab
// of rows, every split) are one contiguous block.
__host__ __device__ inline int64_t partial_slot(int s, int b, int g, int rt, int m_in, int Hkv, int row_tiles,
                                                int tile_stride, int splits) {
  return ((((int64_t)b * Hkv + g) * row_tiles + rt) * tile_stride + m_in) * splits + s;
}

struct MergeParams {
  const int32_t* prefix_len;
  const int32_t* node_offsets;
  const float* o_part;       // fp32 or (part_bf16) bf16 rows of d values
  const float2* ml_part;
  int part_bf16;
  void* out;
  int32_t* status;
  int B, Hq, d, R, max_nodes, out_bf16;
  int skip_single;           // rows of one-chunk sequences were written by the split pass
  int Hkv, G, rows_per_tile, row_tiles, tile_stride;
  int64_t max_prefix, capacity;
  int chunk, tree_tile, splits;
  int early_reads;           // launched right after the split pass of the same call
  int slab_rows;             // rows per merge CTA (2..32, a power of two, <= tile_stride)
  int batch_splits;          // splits gathered into shared memory at once
};

// Merge CTA shape for `tiles` (sequence, KV head, row tile) triples.
void merge_shape(int tiles, int tile_stride, int d, int esize, int splits, int sms, int* slab_rows,
                 int* batch_splits);

// Number of key chunks (splits) of a sequence with a (clamped) prefix of P
// keys: the prefix in chunks of `chunk` keys, the tree keys with the last of
// them.  With tree_tile > 0 (one-wave plans) and a prefix of two or more
// chunks, the tree gets a split of its own when the last prefix chunk already
// has chunk / tree_tile key tiles, so that no split has more tiles than a full
// chunk.  Host and device use the same formula, so the merge reads exactly the
// partials the split pass wrote; it never decreases as P grows.
__host__ __device__ inline int num_chunks(int64_t P, int chunk, int tree_tile) {
  int64_t n = (P + chunk - 1) / chunk;
  if (n < 1) return 1;
  if (tree_tile > 0 && n >= 2) {
    const int64_t last = P - (n - 1) * chunk;
    if ((last + tree_tile - 1) / tree_tile >= chunk / tree_tile) ++n;
  }
  return (int)n;
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

// Programmatic dependent launch.  Every kernel of the library is launched
// with programmatic stream serialization, so its CTAs may start while the
// previous kernel of the stream is still running.  dep_wait() returns once
// the previous grid has completed and its writes are visible; every CTA
// calls it, and calls it before dep_launch(), so a grid never completes
// before its predecessor, and when a kernel's CTAs start, every kernel
// before its predecessor has completed.  Before dep_wait() a kernel
// therefore reads only what its immediate predecessor does not write: the
// caller's inputs (sequence lengths, parents, logits), state an earlier
// kernel of its own call sequence left two launches back (read from L2,
// never from L1), and L2 / TMA prefetches, which only warm caches; it writes
// nothing global.  dep_launch() lets the next kernel's CTAs be scheduled
// early (they wait in their own dep_wait for this grid to finish).
__device__ __forceinline__ void dep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void dep_launch() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// Workspace words that need no zeroing between launches: a word holds a tag
// (the low 40 bits of the launch's %gridid) above a 24-bit count.  Every
// user first raises the word to (tag, 0) with an atomic maximum (an earlier
// launch's word has a smaller tag; memory never written by a launch, with a
// larger one, is replaced by compare-and-swap) and only then counts with
// atomic adds.
__device__ __forceinline__ unsigned long long launch_tag() {
  unsigned long long g;
  asm volatile("mov.u64 %0, %%gridid;" : "=l"(g));
  return (g & ((1ull << 40) - 1)) << 24;
}

__device__ __forceinline__ void arm_counter(unsigned long long* cnt, unsigned long long tag) {
  unsigned long long old = atomicMax(cnt, tag);
  while ((old >> 24) > (tag >> 24)) {               // not an earlier launch's word: replace it
    const unsigned long long prev = atomicCAS(cnt, old, tag);
    if (prev == old) break;
    old = prev;                                     // changed meanwhile (another CTA may have armed it)
  }
}

// L2 prefetch of the line holding ptr: no effect on memory ordering, so a
// kernel may issue it before dep_wait() (it only warms L2 and the TLB for
// what the kernel reads first, while the previous kernel still runs).
__device__ __forceinline__ void prefetch_l2(const void* ptr) {
  asm volatile("prefetch.global.L2 [%0];" ::"l"(reinterpret_cast<uint64_t>(ptr)));
}

template <typename... KArgs, typename... Args>
cudaError_t launch_dep(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                       Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<Args&&>(args)...);
}

// SMs of the current device (cached; a default when no device answers).
int num_sms();

// Devices whose launch attributes are tracked per device (larger ordinals set
// the attribute on every launch).
constexpr int kAttrDevices = 64;

// Raises kernel K's dynamic shared memory limit to at least `bytes` on the
// current device.  A function attribute belongs to a device's context, so it
// is tracked per device: the largest size set so far, kept per kernel
// instantiation (one static array per K).  Safe to call from several host
// threads (setting the same attribute twice is harmless).
template <auto K>
cudaError_t ensure_max_dynamic_smem(int bytes) {
  static std::atomic<int> set_bytes[kAttrDevices];   // zero-initialised
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const bool tracked = dev >= 0 && dev < kAttrDevices;
  if (tracked && set_bytes[dev].load(std::memory_order_acquire) >= bytes) return cudaSuccess;
  e = cudaFuncSetAttribute(K, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e != cudaSuccess || !tracked) return e;
  int cur = set_bytes[dev].load(std::memory_order_relaxed);
  while (cur < bytes && !set_bytes[dev].compare_exchange_weak(cur, bytes, std::memory_order_release)) {
  }
  return cudaSuccess;
}

// Launchers (return cudaError_t of the launch).
cudaError_t launch_attn_simt(const AttnParams& p, int dtype, cudaStream_t s);
cudaError_t launch_attn_tc(const AttnParams& p, cudaStream_t s);
cudaError_t launch_attn_tc2(const AttnParams& p, cudaStream_t s);
cudaError_t launch_attn_tcp(const AttnParams& p, cudaStream_t s);
int64_t tcp_units(const AttnParams& p);
cudaError_t launch_merge(const MergeParams& p, cudaStream_t s);
cudaError_t launch_tree_mask(const int32_t* parents, const int32_t* offs, uint64_t* anc, int32_t* depth,
                             int32_t* status, int B, int R, int max_nodes, cudaStream_t s);



// tcgen05 kernel availability for a descriptor (head_dim, group size).
bool tc_supported(const tv_desc* d, int G);
int tc_key_tile(int d);

}  // namespace tv
