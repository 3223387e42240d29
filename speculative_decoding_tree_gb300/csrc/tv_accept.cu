// Tree mask (A0), per-node argmax (A3), acceptance walk (A4) and the delayed
// KV commit (A5) of the tree-verify step.
//
// Mask rule: "ADR-037 — EAGLE-3 with dynamic tree port", §4 Phase E1 (each
// node sees the prefix, its ancestors and itself).  Acceptance: ADR-037 row
// E5a and Phase E5 (longest matching path from the root; empty accept = root
// only; full accept = deepest), "Speculative decoding verify batches to
// amortize ANE dispatch" (commit-rule bullet: target argmax per row decides;
// longest matching prefix plus one bonus/correction token; accept(k) commits
// only the accepted prefix so rejected drafts never touch the cache).
#include <cfloat>
#include <climits>

#include "tv_internal.cuh"

namespace tv {
namespace {

// ----------------------------------------------------------------- A0

// One block per sequence, one thread per node: walk the parent chain.
__global__ void tree_mask_kernel(const int32_t* __restrict__ parents, const int32_t* __restrict__ offs,
                                 uint64_t* __restrict__ anc, int32_t* __restrict__ depth, int32_t* status,
                                 int B, int R, int max_nodes) {
  const int b = blockIdx.x;
  if (b == B - 1 && threadIdx.x == 0 && offs[B] != R) set_status(status, TV_DEV_BAD_OFFSETS);
  int o0, n;
  if (!seq_rows(offs, b, R, max_nodes, status, &o0, &n)) return;
  const int i = threadIdx.x;
  if (i >= n) return;
  uint64_t bits = 0;
  int dep = 0, j = i;
  bool ok = true;
  while (true) {                       // terminates: the chain index strictly falls
    bits |= 1ull << j;
    const int p = parents[o0 + j];
    if (j == 0) {
      ok = (p == -1);
      break;
    }
    if (p < 0 || p >= j) {
      ok = false;
      break;
    }
    j = p;
    ++dep;
  }
  if (!ok) {
    set_status(status, TV_DEV_BAD_TREE);
    bits = 1ull << i;
    dep = 0;
  }
  anc[o0 + i] = bits;
  if (depth) depth[o0 + i] = dep;
}

// ----------------------------------------------------------------- A3

struct Best {
  float v;
  int i;   // -1 = no non-NaN value seen
};

// max value, smallest index among equal values; NaN never enters.
__device__ __forceinline__ Best better(Best a, Best b) {
  if (a.i < 0) return b;
  if (b.i < 0) return a;
  if (a.v > b.v) return a;
  if (b.v > a.v) return b;
  return a.i <= b.i ? a : b;
}

__device__ __forceinline__ void consider(Best& bst, float x, int idx) {
  if (x != x) return;                               // NaN
  if (bst.i < 0 || x > bst.v || (x == bst.v && idx < bst.i)) {
    bst.v = x;
    bst.i = idx;
  }
}

template <bool BF16>
__device__ __forceinline__ float load_elem(const void* base, int64_t e) {
  if (BF16) return __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(base)[e]);
  return reinterpret_cast<const float*>(base)[e];
}

// grid (vchunks, R): block reduces one vocab chunk of one row with 16-byte
// loads over the aligned body and scalar loads at the ragged ends.
template <bool BF16>
__global__ __launch_bounds__(256) void argmax_partial_kernel(const void* __restrict__ logits, int V, int vlen,
                                                             int vchunks, float* __restrict__ am_val,
                                                             int32_t* __restrict__ am_idx) {
  constexpr int ES = BF16 ? 2 : 4;
  constexpr int PER = 16 / ES;                       // elements per 16-byte load
  const int row = blockIdx.y, c = blockIdx.x;
  const int v0 = c * vlen;
  const int v1 = min(V, v0 + vlen);
  const int64_t rbase = (int64_t)row * V;            // element index of the row start
  Best bst{-FLT_MAX, -1};
  // first element index >= v0 whose address is 16-byte aligned
  const uintptr_t addr0 = reinterpret_cast<uintptr_t>(logits) + (uintptr_t)((rbase + v0) * ES);
  int head = (int)(((16 - (addr0 & 15)) & 15) / ES);
  if ((addr0 & (ES - 1)) != 0) head = v1 - v0;       // cannot align: all scalar
  int a0 = min(v0 + head, v1);
  int nvec = (v1 - a0) / PER;
  int a1 = a0 + nvec * PER;
  for (int e = v0 + threadIdx.x; e < a0; e += blockDim.x) consider(bst, load_elem<BF16>(logits, rbase + e), e);
  const uint4* vp = reinterpret_cast<const uint4*>(reinterpret_cast<const char*>(logits) + (rbase + a0) * ES);
  for (int k = threadIdx.x; k < nvec; k += blockDim.x) {
    uint4 u = __ldcs(vp + k);                        // streamed once: do not keep in L1
    const int e0 = a0 + k * PER;
    if (BF16) {
      const __nv_bfloat162* h2 = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
      for (int t = 0; t < 4; ++t) {
        float2 f = __bfloat1622float2(h2[t]);
        consider(bst, f.x, e0 + 2 * t);
        consider(bst, f.y, e0 + 2 * t + 1);
      }
    } else {
      const float* f = reinterpret_cast<const float*>(&u);
#pragma unroll
      for (int t = 0; t < 4; ++t) consider(bst, f[t], e0 + t);
    }
  }
  for (int e = a1 + threadIdx.x; e < v1; e += blockDim.x) consider(bst, load_elem<BF16>(logits, rbase + e), e);
  // warp then block reduction
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    Best o;
    o.v = __shfl_xor_sync(0xffffffffu, bst.v, off);
    o.i = __shfl_xor_sync(0xffffffffu, bst.i, off);
    bst = better(bst, o);
  }
  __shared__ Best red[8];
  const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (lane == 0) red[w] = bst;
  __syncthreads();
  if (threadIdx.x == 0) {
    Best r = red[0];
    for (int k = 1; k < (int)(blockDim.x >> 5); ++k) r = better(r, red[k]);
    am_val[(int64_t)row * vchunks + c] = r.v;
    am_idx[(int64_t)row * vchunks + c] = r.i;
  }
}

// ----------------------------------------------------------------- A4 + A5

// One block per sequence: finish the argmax, walk, then copy the accepted
// rows' K/V into the cache and advance prefix_len.
__global__ __launch_bounds__(256) void walk_commit_kernel(AcceptParams p) {
  __shared__ int s_am[kMaxNodes], s_par[kMaxNodes], s_draft[kMaxNodes], s_dep[kMaxNodes];
  __shared__ uint64_t s_anc[kMaxNodes];
  __shared__ unsigned long long s_match;
  __shared__ int s_bad_tree, s_key, s_commit_ok, s_P;
  __shared__ int s_path[kMaxNodes];

  const int b = blockIdx.x;
  const int tid = threadIdx.x;
  int o0, n;
  if (!seq_rows(p.node_offsets, b, p.R, p.max_nodes, p.status, &o0, &n)) {
    if (tid < p.max_nodes) {
      p.path[(int64_t)b * p.max_nodes + tid] = -1;
      p.tokens[(int64_t)b * p.max_nodes + tid] = -1;
    }
    if (tid == 0) p.accept_len[b] = -1;
    return;
  }
  if (tid == 0) {
    s_match = 0ull;
    s_bad_tree = 0;
    s_key = -1;
  }
  __syncthreads();

  // finish the argmax of each row from its chunk partials (ascending chunk
  // order keeps the smallest index on ties)
  if (tid < n) {
    Best bst{-FLT_MAX, -1};
    const int64_t r = o0 + tid;
    for (int c = 0; c < p.vchunks; ++c) {
      Best o{p.am_val[r * p.vchunks + c], p.am_idx[r * p.vchunks + c]};
      bst = better(bst, o);
    }
    const int am = bst.i < 0 ? 0 : bst.i;
    s_am[tid] = am;
    p.argmax[r] = am;
    s_par[tid] = p.parents[r];
    s_draft[tid] = p.draft[r];
  }
  __syncthreads();

  // ancestors and depth by walking parents; validate the tree
  if (tid < n) {
    uint64_t bits = 0;
    int dep = 0, j = tid;
    bool ok = true;
    while (true) {
      bits |= 1ull << j;
      const int q = s_par[j];
      if (j == 0) {
        ok = (q == -1);
        break;
      }
      if (q < 0 || q >= j) {
        ok = false;
        break;
      }
      j = q;
      ++dep;
    }
    if (!ok) {
      s_bad_tree = 1;
      bits = 1ull << tid;
      dep = 0;
    }
    s_anc[tid] = bits;
    s_dep[tid] = dep;
    // node matches when its draft equals the target argmax at its parent
    const bool m = (tid == 0) || (ok && s_draft[tid] == s_am[s_par[tid]]);
    if (m) atomicOr(&s_match, 1ull << tid);
  }
  __syncthreads();
  if (s_bad_tree && tid == 0) set_status(p.status, TV_DEV_BAD_TREE);
  // a node is reachable when every node on its root path matches; the best
  // end is the deepest reachable node, ties to the smallest index
  if (tid < n) {
    const bool ok = (s_anc[tid] & ~(uint64_t)s_match) == 0;
    if (ok) atomicMax(&s_key, (s_dep[tid] << 8) | (255 - tid));
  }
  __syncthreads();
  const int key = s_key;                 // >= 0: the root is always reachable
  const int end = 255 - (key & 255);
  const int k = key >> 8;
  if (tid < n && ((s_anc[end] >> tid) & 1ull)) s_path[s_dep[tid]] = tid;
  __syncthreads();
  if (tid < p.max_nodes) {
    const int64_t o = (int64_t)b * p.max_nodes + tid;
    p.path[o] = tid <= k ? s_path[tid] : -1;
    p.tokens[o] = tid < k ? s_draft[s_path[tid + 1]] : (tid == k ? s_am[end] : -1);
  }
  if (tid == 0) {
    p.accept_len[b] = k;
    const int P = p.prefix_len[b];
    s_P = P;
    int ok = 1;
    if (P < 0) {
      set_status(p.status, TV_DEV_BAD_PREFIX);
      ok = 0;
    } else if ((int64_t)P + k + 1 > p.capacity) {
      set_status(p.status, TV_DEV_CAPACITY);
      ok = 0;
    }
    s_commit_ok = ok;
  }
  __syncthreads();
  if (!s_commit_ok) return;
  const int P = s_P;
  if (p.paged) {
    // every page the commit writes must be valid before anything is written
    if (tid <= k) {
      const int64_t pos = (int64_t)P + tid;
      const int pid = p.page_table[(int64_t)b * p.max_pages + pos / kPageSize];
      if (pid < 0 || pid >= p.num_pages) s_commit_ok = 0;
    }
    __syncthreads();
    if (!s_commit_ok) {
      if (tid == 0) set_status(p.status, TV_DEV_BAD_PAGE);
      return;
    }
  }
  // copy k+1 rows x Hkv heads of K and of V in 16-byte units
  const int units_row = p.d * p.esize / 16;
  const int64_t total = 2LL * (k + 1) * p.Hkv * units_row;
  for (int64_t u = tid; u < total; u += blockDim.x) {
    int64_t x = u;
    const int cu = (int)(x % units_row); x /= units_row;
    const int g = (int)(x % p.Hkv); x /= p.Hkv;
    const int t = (int)(x % (k + 1)); x /= (k + 1);
    const int which = (int)x;                     // 0 = K, 1 = V
    const int node = s_path[t];
    const char* src = reinterpret_cast<const char*>(which ? p.v_tree : p.k_tree) +
                      (((int64_t)g * p.R + o0 + node) * p.d) * p.esize;
    const int64_t pos = (int64_t)P + t;
    int64_t drow;
    if (p.paged) {
      const int pid = p.page_table[(int64_t)b * p.max_pages + pos / kPageSize];
      drow = ((int64_t)pid * p.Hkv + g) * kPageSize + pos % kPageSize;
    } else {
      drow = ((int64_t)b * p.Hkv + g) * p.capacity + pos;
    }
    char* dst = reinterpret_cast<char*>(which ? p.v_cache : p.k_cache) + drow * p.d * p.esize;
    reinterpret_cast<uint4*>(dst)[cu] = reinterpret_cast<const uint4*>(src)[cu];
  }
  __syncthreads();
  if (tid == 0) p.prefix_len[b] = P + k + 1;
}

}  // namespace

cudaError_t launch_tree_mask(const int32_t* parents, const int32_t* offs, uint64_t* anc, int32_t* depth,
                             int32_t* status, int B, int R, int max_nodes, cudaStream_t s) {
  tree_mask_kernel<<<B, kMaxNodes, 0, s>>>(parents, offs, anc, depth, status, B, R, max_nodes);
  return cudaGetLastError();
}

cudaError_t launch_accept_commit(const AcceptParams& p, cudaStream_t s) {
  dim3 grid(p.vchunks, p.R);
  if (p.logits_bf16)
    argmax_partial_kernel<true><<<grid, 256, 0, s>>>(p.logits, p.V, p.vchunk_len, p.vchunks, p.am_val, p.am_idx);
  else
    argmax_partial_kernel<false><<<grid, 256, 0, s>>>(p.logits, p.V, p.vchunk_len, p.vchunks, p.am_val, p.am_idx);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  walk_commit_kernel<<<p.B, 256, 0, s>>>(p);
  return cudaGetLastError();
}

}  // namespace tv
