// Tree-position RoPE and K/V scatter ("ADR-037 — EAGLE-3 with dynamic tree
// port", phase rows E4b.5b and E6): one CTA per tree row.  The row's
// position is prefix_len[b] + depth[r]; the d/2 angles are reduced modulo
// 2 pi in float64 once per row (shared by every head), their sines and
// cosines go to shared memory, and the CTA then rotates every query and key
// head of the row and copies its value heads into the head-major tree
// buffers.  Bound by latency (a few KB per row).
#include <cmath>
#include <cstdint>

#include "tree_rope.h"
#include "tv_internal.cuh"

namespace tv {
namespace {

constexpr int kRThreads = 256;

struct RopeParams {
  const void* q_in;
  const void* k_in;
  const void* v_in;
  const int32_t* prefix_len;
  const int32_t* node_offsets;
  const int32_t* depth;
  void* q_out;
  void* k_tree;
  void* v_tree;
  int32_t* status;
  int B, R, Hq, Hkv, d, max_nodes;
  int64_t max_prefix, capacity;
  double inv_freq[256];      // theta^(-2j/d), j < d/2
};

template <bool BF16>
__device__ __forceinline__ float ld(const void* p, int64_t i) {
  if (BF16) return __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(p)[i]);
  return reinterpret_cast<const float*>(p)[i];
}

template <bool BF16>
__device__ __forceinline__ void st(void* p, int64_t i, float x) {
  if (BF16) reinterpret_cast<__nv_bfloat16*>(p)[i] = __float2bfloat16_rn(x);
  else reinterpret_cast<float*>(p)[i] = x;
}

template <bool BF16>
__global__ void __launch_bounds__(kRThreads) tree_rope_kernel(const __grid_constant__ RopeParams p) {
  __shared__ float s_cos[256], s_sin[256];
  __shared__ int s_pos;
  const int r = blockIdx.x, tid = threadIdx.x;
  dep_wait();
  dep_launch();
  if (tid == 0) {
    // the row's sequence: the last b with node_offsets[b] <= r
    int lo = 0, hi = p.B;                         // offsets[lo] <= r < offsets[hi] if valid
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (p.node_offsets[mid] <= r) lo = mid;
      else hi = mid;
    }
    int o0 = 0, n = 0, pos = -1;
    if (seq_rows(p.node_offsets, lo, p.R, p.max_nodes, p.status, &o0, &n) && r >= o0 && r < o0 + n) {
      const int dp = p.depth[r];
      if (dp < 0 || dp >= n) {
        set_status(p.status, TV_DEV_BAD_TREE);
      } else {
        const int64_t P0 = p.prefix_len[lo];
        const int64_t P = clamp_prefix(P0, p.max_prefix, p.capacity);
        if (P != P0) set_status(p.status, TV_DEV_BAD_PREFIX);
        pos = (int)(P + dp);
      }
    } else {
      set_status(p.status, TV_DEV_BAD_OFFSETS);
    }
    s_pos = pos;
  }
  __syncthreads();
  const int pos = s_pos;
  if (pos < 0) return;
  const int half = p.d / 2;
  if (tid < half) {
    // angle modulo 2 pi in float64, then float32 sine and cosine
    const double ang = (double)pos * p.inv_freq[tid];
    const double two_pi = 6.283185307179586;
    const double k = rint(ang * (1.0 / two_pi));
    const float red = (float)fma(-k, two_pi, ang);
    float sn, cs;
    sincosf(red, &sn, &cs);
    s_cos[tid] = cs;
    s_sin[tid] = sn;
  }
  __syncthreads();
  // query heads: [R, Hq, d] in and out
  const int64_t qrow = (int64_t)r * p.Hq * p.d;
  for (int e = tid; e < p.Hq * half; e += blockDim.x) {
    const int h = e / half, j = e - h * half;
    const int64_t i0 = qrow + (int64_t)h * p.d + j;
    const float a = ld<BF16>(p.q_in, i0), b = ld<BF16>(p.q_in, i0 + half);
    const float c = s_cos[j], s = s_sin[j];
    st<BF16>(p.q_out, i0, a * c - b * s);
    st<BF16>(p.q_out, i0 + half, b * c + a * s);
  }
  // key heads rotated into [Hkv, R, d]; value heads copied
  const int64_t krow = (int64_t)r * p.Hkv * p.d;
  for (int e = tid; e < p.Hkv * half; e += blockDim.x) {
    const int g = e / half, j = e - g * half;
    const int64_t i0 = krow + (int64_t)g * p.d + j;
    const int64_t o0 = ((int64_t)g * p.R + r) * p.d + j;
    const float a = ld<BF16>(p.k_in, i0), b = ld<BF16>(p.k_in, i0 + half);
    const float c = s_cos[j], s = s_sin[j];
    st<BF16>(p.k_tree, o0, a * c - b * s);
    st<BF16>(p.k_tree, o0 + half, b * c + a * s);
  }
  const int ES = BF16 ? 2 : 4;
  const int units = p.d * ES / 16;                // 16-byte units per head vector
  for (int e = tid; e < p.Hkv * units; e += blockDim.x) {
    const int g = e / units, u = e - g * units;
    const uint4* src = reinterpret_cast<const uint4*>(reinterpret_cast<const char*>(p.v_in) + (krow + (int64_t)g * p.d) * ES) + u;
    uint4* dst = reinterpret_cast<uint4*>(reinterpret_cast<char*>(p.v_tree) + (((int64_t)g * p.R + r) * p.d) * ES) + u;
    *dst = *src;
  }
}

bool aligned16(const void* q) { return (reinterpret_cast<uintptr_t>(q) & 15u) == 0; }

}  // namespace
}  // namespace tv

using namespace tv;

extern "C" {

int tv_tree_rope_scatter(const tv_desc* desc, double theta, const void* d_q_in, const void* d_k_in,
                         const void* d_v_in, const int32_t* d_prefix_len, const int32_t* d_node_offsets,
                         const int32_t* d_depth, void* d_q_out, void* d_k_tree, void* d_v_tree, int32_t* d_status,
                         void* stream) {
  size_t ws = 0;
  int rc = tv_workspace_size(desc, 0, &ws);        // the descriptor's own checks
  if (rc) return rc;
  if (!(theta > 1.0) || !std::isfinite(theta)) return TV_ERR_SHAPE;
  if (!d_q_in || !d_k_in || !d_v_in || !d_prefix_len || !d_node_offsets || !d_depth || !d_q_out || !d_k_tree ||
      !d_v_tree || !d_status)
    return TV_ERR_NULL;
  const void* ptrs[] = {d_q_in, d_k_in, d_v_in, d_prefix_len, d_node_offsets, d_depth, d_q_out, d_k_tree, d_v_tree,
                        d_status};
  for (const void* q : ptrs)
    if (!aligned16(q)) return TV_ERR_ALIGN;
  RopeParams p;
  p.q_in = d_q_in;
  p.k_in = d_k_in;
  p.v_in = d_v_in;
  p.prefix_len = d_prefix_len;
  p.node_offsets = d_node_offsets;
  p.depth = d_depth;
  p.q_out = d_q_out;
  p.k_tree = d_k_tree;
  p.v_tree = d_v_tree;
  p.status = d_status;
  p.B = desc->batch;
  p.R = desc->total_rows;
  p.Hq = desc->num_q_heads;
  p.Hkv = desc->num_kv_heads;
  p.d = desc->head_dim;
  p.max_nodes = desc->max_nodes;
  p.max_prefix = desc->max_prefix;
  p.capacity = desc->capacity;
  for (int j = 0; j < 256; ++j) p.inv_freq[j] = j < p.d / 2 ? std::pow(theta, -2.0 * j / p.d) : 0.0;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const cudaError_t e = desc->dtype == TV_BF16
                            ? launch_dep(tree_rope_kernel<true>, dim3(p.R), dim3(kRThreads), 0, s, p)
                            : launch_dep(tree_rope_kernel<false>, dim3(p.R), dim3(kRThreads), 0, s, p);
  return e == cudaSuccess ? TV_OK : TV_ERR_CUDA;
}

}  // extern "C"
