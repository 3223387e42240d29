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
#include "tv_accept.cuh"
#include "tc_ptx.cuh"

namespace tv {
namespace {

using namespace tc;

// ----------------------------------------------------------------- A0

// One block per sequence, one thread per node: the sequence's parents are
// read into shared memory in one step, then each thread walks its chain there.
__global__ void tree_mask_kernel(const int32_t* __restrict__ parents, const int32_t* __restrict__ offs,
                                 uint64_t* __restrict__ anc, int32_t* __restrict__ depth, int32_t* status,
                                 int B, int R, int max_nodes) {
  __shared__ int s_par[kMaxNodes];
  dep_wait();
  dep_launch();
  const int b = blockIdx.x;
  if (b == B - 1 && threadIdx.x == 0 && offs[B] != R) set_status(status, TV_DEV_BAD_OFFSETS);
  int o0, n;
  if (!seq_rows(offs, b, R, max_nodes, status, &o0, &n)) return;   // uniform over the block
  const int i = threadIdx.x;
  if (i < n) s_par[i] = parents[o0 + i];
  __syncthreads();
  if (i >= n) return;
  uint64_t bits = 0;
  int dep = 0, j = i;
  bool ok = true;
  while (true) {                       // terminates: the chain index strictly falls
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

template <bool BF16>
__device__ __forceinline__ float load_elem(const void* base, int64_t e) {
  if (BF16) return __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(base)[e]);
  return reinterpret_cast<const float*>(base)[e];
}

// In-order update: a thread sees its elements in increasing index order, so
// a strictly greater value is the only way to replace the current best (ties
// keep the earlier, smaller index); NaN never enters; the first non-NaN value
// is taken even when it is -inf.
__device__ __forceinline__ void take_in_order(Best& bst, float x, int idx) {
  const bool take = (x > bst.v) || (bst.i < 0 && x == x);
  bst.v = take ? x : bst.v;
  bst.i = take ? idx : bst.i;
}

// Largest of the 8 values in a 16-byte word (NaN ignored unless all are NaN).
template <bool BF16>
__device__ __forceinline__ float vec_max(const uint4& u) {
  if (BF16) {
    const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&u);
    const __nv_bfloat162 m = __hmax2(__hmax2(h[0], h[1]), __hmax2(h[2], h[3]));
    return fmaxf(__low2float(m), __high2float(m));
  }
  const float* f = reinterpret_cast<const float*>(&u);
  return fmaxf(fmaxf(f[0], f[1]), fmaxf(f[2], f[3]));
}

// First element of the word equal to `x` (x is a value the word holds).
template <bool BF16>
__device__ __forceinline__ int vec_first(const uint4& u, float x) {
  if (BF16) {
    const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
    for (int t = 0; t < 4; ++t) {
      if (__low2float(h[t]) == x) return 2 * t;
      if (__high2float(h[t]) == x) return 2 * t + 1;
    }
    return 7;
  }
  const float* f = reinterpret_cast<const float*>(&u);
#pragma unroll
  for (int t = 0; t < 3; ++t)
    if (f[t] == x) return t;
  return 3;
}

// L2 prefetches a pass block issues while the previous kernel runs (a
// prefetch does not read data before the wait, it only warms the cache):
// its slice of the logits and, from the blocks of chunk 0, the row's tree K
// and V (every KV head), which the commit may copy into the cache.
template <int ES>
__device__ __forceinline__ void prefetch_pass_t(const AcceptParams& p, int row, int v0, int v1) {
  if (v0 < v1) {
    const char* base = reinterpret_cast<const char*>(p.logits) + ((int64_t)row * p.V + v0) * ES;
    const int64_t bytes = (int64_t)(v1 - v0) * ES;
    for (int64_t off = (int64_t)threadIdx.x * 128; off < bytes; off += 128 * (int64_t)blockDim.x)
      prefetch_l2(base + off);
  }
  if (blockIdx.x == 0) {
    const int64_t row_bytes = (int64_t)p.d * p.esize;
    const int lines = (int)(row_bytes / 128);
    for (int e = threadIdx.x; e < 2 * p.Hkv * lines; e += blockDim.x) {
      const int kind = e / (p.Hkv * lines), g = (e / lines) % p.Hkv, ln = e % lines;
      const char* src = reinterpret_cast<const char*>(kind ? p.v_tree : p.k_tree);
      prefetch_l2(src + ((int64_t)g * p.R + row) * row_bytes + ln * 128);
    }
  }
}
#define prefetch_pass(p, row, v0, v1) prefetch_pass_t<ES>(p, row, v0, v1)

// grid (vchunks, R): one block reduces one vocab chunk of one row.  Each
// thread streams 16-byte words (four in flight) in increasing index order.
// A packed max over each batch of words is compared with the thread's best:
// only a strictly larger batch maximum triggers the index search (first
// word, then first element, holding it), so equal values keep the earlier
// index and NaN never wins.  Scalar loads cover the ragged chunk ends.
template <bool BF16>
__global__ __launch_bounds__(256) void argmax_partial_kernel(const AcceptParams p) {
  constexpr int ES = BF16 ? 2 : 4;
  constexpr int PER = 16 / ES;                       // elements per 16-byte load
  constexpr int UNROLL = 4;                          // words in flight per thread
  const void* __restrict__ logits = p.logits;
  const int V = p.V;
  const int row = blockIdx.y, c = blockIdx.x;
  const int v0 = c * p.vchunk_len;
  const int v1 = min(V, v0 + p.vchunk_len);
  const int64_t rbase = (int64_t)row * V;            // element index of the row start
  prefetch_pass(p, row, v0, v1);
  dep_wait();
  dep_launch();
  const uintptr_t addr0 = reinterpret_cast<uintptr_t>(logits) + (uintptr_t)((rbase + v0) * ES);
  int head = (int)(((16 - (addr0 & 15)) & 15) / ES);
  if ((addr0 & (ES - 1)) != 0) head = v1 - v0;       // cannot align: all scalar
  const int a0 = min(v0 + head, v1);
  const int nvec = (v1 - a0) / PER;
  const int a1 = a0 + nvec * PER;
  Best bst{-INFINITY, -1};
  // head (lowest indices) first, then the body, then the tail: in order
  for (int e = v0 + (int)threadIdx.x; e < a0; e += blockDim.x) take_in_order(bst, load_elem<BF16>(logits, rbase + e), e);
  const uint4* vp = reinterpret_cast<const uint4*>(reinterpret_cast<const char*>(logits) + (rbase + a0) * ES);
  const int step = (int)blockDim.x;
  for (int k0 = threadIdx.x; k0 < nvec; k0 += UNROLL * step) {
    uint4 u[UNROLL];
    float m[UNROLL];
#pragma unroll
    for (int q = 0; q < UNROLL; ++q) {
      const int k = k0 + q * step;
      u[q] = k < nvec ? __ldcs(vp + k) : make_uint4(0xffffffffu, 0xffffffffu, 0xffffffffu, 0xffffffffu);
    }
#pragma unroll
    for (int q = 0; q < UNROLL; ++q) m[q] = (k0 + q * step < nvec) ? vec_max<BF16>(u[q]) : __int_as_float(0x7fffffff);
    float mb = m[0];                                  // NaN only if all NaN
#pragma unroll
    for (int q = 1; q < UNROLL; ++q) mb = fmaxf(mb, m[q]);
    if (mb > bst.v || (bst.i < 0 && mb == mb)) {
      int qs = UNROLL - 1;                          // first word holding the batch maximum
#pragma unroll
      for (int q = UNROLL - 1; q >= 0; --q)
        if (m[q] == mb) qs = q;
      uint4 uq = u[0];
#pragma unroll
      for (int q = 1; q < UNROLL; ++q)
        if (q == qs) uq = u[q];
      bst.v = mb;
      bst.i = a0 + (k0 + qs * step) * PER + vec_first<BF16>(uq, mb);
    }
  }
  for (int e = a1 + (int)threadIdx.x; e < v1; e += blockDim.x) take_in_order(bst, load_elem<BF16>(logits, rbase + e), e);
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
    p.am_val[(int64_t)row * p.vchunks + c] = r.v;
    p.am_idx[(int64_t)row * p.vchunks + c] = r.i;
  }
}

// ----------------------------------------------------------------- A3, sampled

// Philox4x32 with 10 rounds (Salmon, Moraes, Dror, Shaw, "Parallel random
// numbers: as easy as 1, 2, 3", SC 2011): each round multiplies words 0 and
// 2 by the two multipliers; the new words are (hi1 ^ c1 ^ k0, lo1,
// hi0 ^ c3 ^ k1, lo0); the key grows by the Weyl constants between rounds.
__device__ __forceinline__ void philox4x32_10(uint32_t c[4], uint32_t k0, uint32_t k1) {
  constexpr uint32_t M0 = 0xD2511F53u, M1 = 0xCD9E8D57u, W0 = 0x9E3779B9u, W1 = 0xBB67AE85u;
#pragma unroll
  for (int r = 0; r < 10; ++r) {
    if (r) {
      k0 += W0;
      k1 += W1;
    }
    const uint32_t hi0 = __umulhi(M0, c[0]), lo0 = M0 * c[0];
    const uint32_t hi1 = __umulhi(M1, c[2]), lo1 = M1 * c[2];
    const uint32_t n0 = hi1 ^ c[1] ^ k0, n2 = hi0 ^ c[3] ^ k1;
    c[0] = n0;
    c[1] = lo1;
    c[2] = n2;
    c[3] = lo0;
  }
}

// Gumbel noise G = -log(E), E = -log U, from a Philox word: U = ((w >> 9) +
// 0.5) * 2^-23 and d = 1 - U are both exact in float32 and strictly inside
// (0, 1).  The largest possible G is -log(-log(1 - 2^-24)) = 16.636...
// E needs relative accuracy (G = -log E): for d < 1/16 it is the Mercator
// series d + d^2/2 + ... + d^6/6 (truncation below 1e-9 relative), else the
// hardware base-2 logarithm of U (U <= 15/16, where its absolute error is a
// small relative one); G's base-2 logarithm needs only absolute accuracy.
constexpr float kGumbelMax = 16.75f;
constexpr float kLn2 = 0.69314718f;
__device__ __forceinline__ float gumbel_of(uint32_t w) {
  const uint32_t m = w >> 9;
  const float d = ((float)(0x7FFFFFu - m) + 0.5f) * 0x1p-23f;     // 1 - U
  float e;
  if (d < 0.0625f)
    e = d * fmaf(d, fmaf(d, fmaf(d, fmaf(d, fmaf(d, 1.f / 6.f, 0.2f), 0.25f), 1.f / 3.f), 0.5f), 1.f);
  else
    e = -__log2f(((float)m + 0.5f) * 0x1p-23f) * kLn2;
  return -__log2f(e) * kLn2;
}

// Sampled verification's draw, one vocab chunk of one row per block (grid
// (vchunks, R)): y = argmax_v (logits[v] / T + G[v]) with G from Philox at
// counter (v / 4, row, offset) and key seed, word v % 4.  Each thread takes
// groups of four entries in increasing order and keeps the first strictly
// larger value, so the block reduction's smallest-index rule gives the first
// index of the maximum; NaN never enters.  A group whose entries cannot
// reach the thread's best even with the largest possible noise is skipped
// without drawing its noise (the skip is exact: the bound is never met).
template <bool BF16>
__global__ __launch_bounds__(256) void sample_partial_kernel(const AcceptParams p) {
  constexpr int ES = BF16 ? 2 : 4;
  const void* __restrict__ logits = p.logits;
  const int V = p.V;
  const float inv_t = p.inv_temp;
  const uint32_t k0 = p.seed_lo, k1 = p.seed_hi, off0 = p.off_lo, off1 = p.off_hi;
  const int row = blockIdx.y, c = blockIdx.x;
  const int v0 = c * p.vchunk_len;                   // a multiple of 8
  const int v1 = min(V, v0 + p.vchunk_len);
  const int64_t rbase = (int64_t)row * V;
  prefetch_pass(p, row, v0, v1);
  dep_wait();
  dep_launch();
  // four consecutive entries load as one word when the row keeps them aligned
  const bool vec = (V % 4 == 0) && ((reinterpret_cast<uintptr_t>(logits) & (4 * ES - 1)) == 0);
  Best bst{-INFINITY, -1};
  for (int g = (v0 >> 2) + (int)threadIdx.x; 4 * g < v1; g += blockDim.x) {
    float x[4];
    const int e = 4 * g;
    if (vec && e + 3 < v1) {
      if (BF16) {
        const uint2 u = *reinterpret_cast<const uint2*>(reinterpret_cast<const __nv_bfloat16*>(logits) + rbase + e);
        const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u.x));
        const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u.y));
        x[0] = a.x; x[1] = a.y; x[2] = b.x; x[3] = b.y;
      } else {
        const float4 f = *reinterpret_cast<const float4*>(reinterpret_cast<const float*>(logits) + rbase + e);
        x[0] = f.x; x[1] = f.y; x[2] = f.z; x[3] = f.w;
      }
    } else {
#pragma unroll
      for (int q = 0; q < 4; ++q) x[q] = e + q < v1 ? load_elem<BF16>(logits, rbase + e + q) : __int_as_float(0x7fffffff);
    }
    // no entry of the group can beat the best even with the largest noise:
    // skip it without drawing (false for NaN)
    bool may = bst.i < 0;
#pragma unroll
    for (int q = 0; q < 4; ++q) may |= fmaf(x[q], inv_t, kGumbelMax) > bst.v;
    if (!may) continue;
    uint32_t w[4] = {(uint32_t)g, (uint32_t)row, off0, off1};
    philox4x32_10(w, k0, k1);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      if (e + q >= v1) continue;
      const float xt = x[q] * inv_t;
      if (xt != xt) continue;                         // NaN is never drawn
      if (bst.i >= 0) {
        // E = -log(1 - d) >= d: when d > 1.001 e^-c (c = best - xt), G <=
        // c - 0.001 and this entry cannot beat the best (nor can it with
        // G's rounding); most entries leave here without a logarithm.
        // c = -inf (xt = +inf) never prunes, c = +inf always does.
        const float c = bst.v - xt;
        const float d = ((float)(0x7FFFFFu - (w[q] >> 9)) + 0.5f) * 0x1p-23f;
        if (d > 1.001f * __expf(-c)) continue;
      }
      take_in_order(bst, xt + gumbel_of(w[q]), e + q);
    }
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    Best o;
    o.v = __shfl_xor_sync(0xffffffffu, bst.v, off);
    o.i = __shfl_xor_sync(0xffffffffu, bst.i, off);
    bst = better(bst, o);
  }
  __shared__ Best red[8];
  const int w8 = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (lane == 0) red[w8] = bst;
  __syncthreads();
  if (threadIdx.x == 0) {
    Best r = red[0];
    for (int k = 1; k < (int)(blockDim.x >> 5); ++k) r = better(r, red[k]);
    p.am_val[(int64_t)row * p.vchunks + c] = r.v;
    p.am_idx[(int64_t)row * p.vchunks + c] = r.i;
  }
}

// ----------------------------------------------------------------- A4 + A5

// The walk and commit of one sequence, run by a cluster of C blocks of 256
// threads, C = min(8, 2 Hkv): the rows to commit fall into 2 Hkv sets (K or
// V, KV head), and block x of the cluster copies sets x, x + C, ...  Every
// block finishes the argmax of every node from its chunk partials (four
// threads per node) or takes the given one, and walks (warp 0: lane i owns
// nodes i and i + 32; ballots and shuffles, no shared atomics); the blocks
// reach the same path from the same inputs, and block 0 alone writes the
// outputs.  Where a block's sets fit in shared memory, it stages the
// sequence's tree rows of its sets there by bulk copies while the pass
// kernel still runs, so that after the walk the commit only stores.  Block 0
// advances prefix_len behind a cluster barrier that each block arrives on
// once it has read the old value.
constexpr int kCommitPages = kMaxNodes / kPageSize + 1;   // pages the k + 1 <= 64 rows can touch
constexpr int kWalkThreads = 256;
constexpr uint64_t kWalkWaitNs = 1000000000ull;           // bound on the staging copies' wait

struct WalkSmem {
  int par[kMaxNodes], draft[kMaxNodes], am[kMaxNodes], path[kMaxNodes];
  uint64_t anc[kMaxNodes];
  int pid[kCommitPages];
  int k, ok, abort_flag;
  alignas(8) uint64_t staged;                        // mbarrier: the staging copies have landed
};

__device__ __forceinline__ void cluster_arrive_release() {
  asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait_acquire() {
  asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// what warp 0 keeps of the tree (lane i: nodes i and i + 32)
struct WalkRegs {
  uint64_t anc[2];
  int dep[2];
  bool tree_ok[2];
};

// Part 1, which needs no argmax.  walk_stage: the sequence's parents,
// drafts and the page ids a commit may write (the positions P .. P + 63,
// paged cache only), into shared memory.
__device__ __forceinline__ void walk_stage_pages(const AcceptParams& p, int b, WalkSmem& s, int P) {
  const int tid = threadIdx.x;
  if (p.paged && tid >= 64 && tid < 64 + kCommitPages && P >= 0) {
    const int64_t pg = (int64_t)P / kPageSize + (tid - 64);
    s.pid[tid - 64] = pg < p.max_pages ? p.page_table[(int64_t)b * p.max_pages + pg] : -1;
  }
}

__device__ void walk_stage(const AcceptParams& p, int b, WalkSmem& s, int o0, int n, int P) {
  const int tid = threadIdx.x;
  if (tid < n) {
    s.par[tid] = p.parents[o0 + tid];
    s.draft[tid] = p.draft[o0 + tid];
  }
  walk_stage_pages(p, b, s, P);
}

// walk_tree: once the parents are staged, warp 0 builds each node's
// ancestor word and depth by walking the parent pointers.
__device__ void walk_tree(WalkSmem& s, WalkRegs& wr, int n) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
#pragma unroll
  for (int hlf = 0; hlf < 2; ++hlf) {
    wr.anc[hlf] = 0ull;
    wr.dep[hlf] = 0;
    wr.tree_ok[hlf] = true;
  }
  __syncthreads();                                  // parents staged
  if (warp == 0) {
#pragma unroll
    for (int hlf = 0; hlf < 2; ++hlf) {
      const int i = lane + 32 * hlf;
      if (i < n) {
        uint64_t bits = 0;
        int d = 0, j = i;
        bool ok = true;
        while (true) {                              // terminates: the chain index strictly falls
          bits |= 1ull << j;
          const int q = s.par[j];
          if (j == 0) {
            ok = (q == -1);
            break;
          }
          if (q < 0 || q >= j) {
            ok = false;
            break;
          }
          j = q;
          ++d;
        }
        if (!ok) {
          bits = 1ull << i;
          d = 0;
        }
        wr.anc[hlf] = bits;
        wr.dep[hlf] = d;
        wr.tree_ok[hlf] = ok;
        s.anc[i] = bits;
      }
    }
  }
}

// The outputs of a sequence whose node offsets are invalid.
__device__ void walk_invalid(const AcceptParams& p, int b) {
  const int tid = threadIdx.x;
  if (tid == 0) set_status(p.status, TV_DEV_BAD_OFFSETS);
  if (tid < p.max_nodes) {
    p.path[(int64_t)b * p.max_nodes + tid] = -1;
    p.tokens[(int64_t)b * p.max_nodes + tid] = -1;
  }
  if (tid == 0) p.accept_len[b] = -1;
}

// Thread 0 starts the bulk copies of this block's sets of sequence b: set j
// = (K or V, KV head g) holds the sequence's n tree rows contiguously (rows
// o0 .. o0 + n - 1 of head g), staged at slot m = (j - x) / C, max_nodes rows
// per slot.  Addresses and sizes are multiples of 16 bytes (the host checks
// the buffers' alignment; a row is d * esize bytes, a multiple of 16).
__device__ void walk_stage_rows(const AcceptParams& p, WalkSmem& s, char* stage, int o0, int n) {
  if (threadIdx.x != 0) return;
  const int C = (int)gridDim.x;
  const int64_t row_bytes = (int64_t)p.d * p.esize;
  const uint32_t bar = smem_u32(&s.staged);
  uint32_t total = 0;
  for (int j = blockIdx.x; j < 2 * p.Hkv; j += C) total += (uint32_t)(n * row_bytes);
  mbar_expect_tx(bar, total);
  for (int j = blockIdx.x, m = 0; j < 2 * p.Hkv; j += C, ++m) {
    const int kind = j / p.Hkv, g = j - kind * p.Hkv;
    const char* src = reinterpret_cast<const char*>(kind ? p.v_tree : p.k_tree) + ((int64_t)g * p.R + o0) * row_bytes;
    if (n > 0) bulk_load(smem_u32(stage + (int64_t)m * p.max_nodes * row_bytes), src, (uint32_t)(n * row_bytes), bar);
  }
}

// The commit: rows t = 0 .. k of this block's sets, from the staged rows or
// (sets too large to stage) from the tree buffers, into cache positions
// P + t.  16-byte units (unit u: row u / units_row), up to 8 loads in flight
// per thread, all issued before the stores.
__device__ void walk_commit_rows(const AcceptParams& p, int b, const WalkSmem& s, const char* stage, int o0, int P,
                                 int k) {
  const int C = (int)gridDim.x, tid = threadIdx.x;
  const int64_t row_bytes = (int64_t)p.d * p.esize;
  const int units_row = (int)(row_bytes / 16);      // a power of two (16 .. 128)
  const int ushift = __ffs(units_row) - 1;
  const int sets = (2 * p.Hkv - (int)blockIdx.x + C - 1) / C;
  const int total = sets * (k + 1) * units_row;
  constexpr int U = 8;
  for (int base = 0; base < total; base += U * (int)blockDim.x) {
    uint4 v[U];
    uint4* dst[U];
#pragma unroll
    for (int q = 0; q < U; ++q) {
      const int u = base + q * (int)blockDim.x + tid;
      dst[q] = nullptr;
      if (u < total) {
        const int rr = u >> ushift, w = u & (units_row - 1);
        const int m = rr / (k + 1), t = rr - m * (k + 1);
        const int j = (int)blockIdx.x + m * C, kind = j / p.Hkv, g = j - kind * p.Hkv;
        const int node = s.path[t];
        const int64_t pos = (int64_t)P + t;
        int64_t drow;
        if (p.paged) {
          const int pid = s.pid[(P + t) / kPageSize - P / kPageSize];
          drow = ((int64_t)pid * p.Hkv + g) * kPageSize + pos % kPageSize;
        } else {
          drow = ((int64_t)b * p.Hkv + g) * p.capacity + pos;
        }
        if (stage) {
          v[q] = reinterpret_cast<const uint4*>(stage + ((int64_t)m * p.max_nodes + node) * row_bytes)[w];
        } else {
          const char* src = reinterpret_cast<const char*>(kind ? p.v_tree : p.k_tree) +
                            ((int64_t)g * p.R + o0 + node) * row_bytes;
          v[q] = __ldcg(reinterpret_cast<const uint4*>(src) + w);
        }
        dst[q] = reinterpret_cast<uint4*>(reinterpret_cast<char*>(kind ? p.v_cache : p.k_cache) + drow * row_bytes) + w;
      }
    }
#pragma unroll
    for (int q = 0; q < U; ++q)
      if (dst[q]) *dst[q] = v[q];
  }
}

// Part 2: each node's argmax (the caller's, or finished from the chunk
// partials, which other blocks of the pass grid wrote: read through L2), the
// walk, the outputs (block 0) and the commit of this block's sets.
__device__ void walk_finish(const AcceptParams& p, int b, WalkSmem& s, const WalkRegs& wr, const char* stage, int o0,
                            int n, int P) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const bool lead = blockIdx.x == 0;
  if (p.given_argmax) {
    if (tid < n) s.am[tid] = p.argmax[o0 + tid];
  } else {
    // argmax of node tid / 4 from chunks c = tid % 4, + 4, ...; max value,
    // smallest index (better() is order-free), NaN never enters.  All of a
    // thread's partials are loaded before the first comparison: one L2
    // round instead of one per chunk.
    constexpr int kPer = kMaxVChunks / 4;
    static_assert(kMaxVChunks % 4 == 0, "four threads per node share the chunks");
    const int vc = p.vchunks;
    const int i = tid >> 2;
    const bool live = i < n;
    const int64_t pbase = (int64_t)(o0 + (live ? i : 0)) * vc;
    float pv[kPer];
    int pi[kPer];
#pragma unroll
    for (int q = 0; q < kPer; ++q) {
      const int c = (tid & 3) + 4 * q;
      const bool use = live && c < vc;
      pv[q] = use ? __ldcg(p.am_val + pbase + c) : 0.f;
      pi[q] = use ? __ldcg(p.am_idx + pbase + c) : -1;
    }
    Best bst{-FLT_MAX, -1};
#pragma unroll
    for (int q = 0; q < kPer; ++q) bst = better(bst, Best{pv[q], pi[q]});
#pragma unroll
    for (int off = 1; off < 4; off <<= 1) {
      Best o;
      o.v = __shfl_xor_sync(0xffffffffu, bst.v, off);
      o.i = __shfl_xor_sync(0xffffffffu, bst.i, off);
      bst = better(bst, o);
    }
    if (i < n && (tid & 3) == 0) {
      const int am = bst.i < 0 ? 0 : bst.i;
      s.am[i] = am;
      if (lead) p.argmax[o0 + i] = am;
    }
  }
  __syncthreads();

  if (warp == 0) {
    const unsigned all = 0xffffffffu;
    // match against the parent's argmax
    bool mt[2] = {false, false}, bad = false;
#pragma unroll
    for (int hlf = 0; hlf < 2; ++hlf) {
      const int i = lane + 32 * hlf;
      if (i < n) {
        bad |= !wr.tree_ok[hlf];
        mt[hlf] = (i == 0) || (wr.tree_ok[hlf] && s.draft[i] == s.am[s.par[i]]);
      }
    }
    if (__any_sync(all, bad) && lane == 0 && lead) set_status(p.status, TV_DEV_BAD_TREE);
    const uint64_t match = (uint64_t)__ballot_sync(all, mt[0]) | ((uint64_t)__ballot_sync(all, mt[1]) << 32);
    // reachable = every node on the root path matches; best = deepest, then
    // smallest index
    int key = -1;
#pragma unroll
    for (int hlf = 0; hlf < 2; ++hlf) {
      const int i = lane + 32 * hlf;
      if (i < n && (wr.anc[hlf] & ~match) == 0) key = max(key, (wr.dep[hlf] << 8) | (255 - i));
    }
    key = __reduce_max_sync(all, key);              // >= 0: the root is always reachable
    const int end = 255 - (key & 255), k = key >> 8;
    __syncwarp();
    const uint64_t end_anc = s.anc[end];
#pragma unroll
    for (int hlf = 0; hlf < 2; ++hlf) {
      const int i = lane + 32 * hlf;
      if (i < n && ((end_anc >> i) & 1ull)) s.path[wr.dep[hlf]] = i;
    }
    __syncwarp();
#pragma unroll
    for (int hlf = 0; hlf < 2; ++hlf) {
      const int t = lane + 32 * hlf;
      if (t < p.max_nodes && lead) {
        const int64_t o = (int64_t)b * p.max_nodes + t;
        p.path[o] = t <= k ? s.path[t] : -1;
        p.tokens[o] = t < k ? s.draft[s.path[t + 1]] : (t == k ? s.am[end] : -1);
      }
    }
    // can the k+1 rows be committed?
    bool ok = true;
    if (P < 0) {
      ok = false;
      if (lane == 0 && lead) set_status(p.status, TV_DEV_BAD_PREFIX);
    } else if ((int64_t)P + k + 1 > p.capacity) {
      ok = false;
      if (lane == 0 && lead) set_status(p.status, TV_DEV_CAPACITY);
    } else if (p.paged) {
      bool page_bad = false;
#pragma unroll
      for (int hlf = 0; hlf < 2; ++hlf) {
        const int t = lane + 32 * hlf;
        if (t <= k) {
          const int pid = s.pid[(P + t) / kPageSize - P / kPageSize];
          page_bad |= (pid < 0 || pid >= p.num_pages);
        }
      }
      if (__any_sync(all, page_bad)) {
        ok = false;
        if (lane == 0 && lead) set_status(p.status, TV_DEV_BAD_PAGE);
      }
    }
    if (lane == 0) {
      if (lead) p.accept_len[b] = k;
      s.k = k;
      s.ok = ok ? 1 : 0;
    }
  }
  __syncthreads();
  if (!s.ok) return;
  if (stage) {
    // the staging copies have landed (bounded: on a timeout nothing is committed)
    const bool in = mbar_wait(smem_u32(&s.staged), 0, &s.abort_flag, kWalkWaitNs);
    if (!__syncthreads_and(in)) {
      if (tid == 0) set_status(p.status, TV_DEV_TIMEOUT);
      s.ok = 0;                                     // read only after the cluster barrier's wait below
      return;
    }
  }
  walk_commit_rows(p, b, s, stage, o0, P, s.k);
}

// Walk and commit: grid (C, B), clusters of C blocks (one cluster per
// sequence).  After the pass kernel of the same call (which writes only the
// chunk partials and waited for its own predecessor before letting this
// kernel start), the sequence's lengths, parents, drafts, page ids and tree
// rows are read and the ancestors built before the dependency wait; on a
// given argmax (no pass kernel), everything it reads may come from the
// kernel just before it, so it waits first.
__global__ __launch_bounds__(kWalkThreads) void walk_commit_kernel(AcceptParams p) {
  __shared__ WalkSmem s;
  extern __shared__ __align__(128) char stage_mem[];
  char* stage = p.stage_bytes > 0 ? stage_mem : nullptr;
  if (p.given_argmax) {
    dep_wait();
    dep_launch();
  }
  const int b = blockIdx.y, tid = threadIdx.x;
  const bool lead = blockIdx.x == 0;
  int o0 = 0, n = 0;
  const bool valid = seq_rows(p.node_offsets, b, p.R, p.max_nodes, nullptr, &o0, &n);
  const int P = valid ? p.prefix_len[b] : 0;
  if (tid == 0) {
    s.abort_flag = 0;
    s.ok = 0;
    if (stage) {
      mbar_init(smem_u32(&s.staged), 1);
      fence_barrier_init();
    }
  }
  if (valid) {
    walk_stage(p, b, s, o0, n, P);
    if (stage) walk_stage_rows(p, s, stage, o0, n);
  }
  WalkRegs wr;
  walk_tree(s, wr, valid ? n : 0);
  cluster_arrive_release();                         // this block has read prefix_len[b]
  if (!p.given_argmax) {
    dep_wait();
    dep_launch();
  }
  if (!valid) {
    if (lead) walk_invalid(p, b);
  } else {
    walk_finish(p, b, s, wr, stage, o0, n, P);
  }
  // no block exits with its staging copies in flight (they completed before
  // any commit; this covers the sequences that commit nothing, and a wait
  // that gave up: its own flag is raised, so this wait has a fresh one)
  if (stage && valid && tid == 0) {
    int spare = 0;
    mbar_wait(smem_u32(&s.staged), 0, &spare, kWalkWaitNs);
  }
  cluster_wait_acquire();                           // every block has read prefix_len[b]
  if (lead && tid == 0 && valid && s.ok) p.prefix_len[b] = P + s.k + 1;
}

}  // namespace

cudaError_t launch_tree_mask(const int32_t* parents, const int32_t* offs, uint64_t* anc, int32_t* depth,
                             int32_t* status, int B, int R, int max_nodes, cudaStream_t s) {
  return launch_dep(tree_mask_kernel, dim3(B), dim3(kMaxNodes), 0, s, parents, offs, anc, depth, status, B, R,
                    max_nodes);
}

cudaError_t launch_accept_commit(const AcceptParams& p, cudaStream_t s) {
  if (!p.given_argmax) {
    dim3 grid(p.vchunks, p.R);
    cudaError_t e = launch_dep(p.sampled ? (p.logits_bf16 ? sample_partial_kernel<true> : sample_partial_kernel<false>)
                                         : (p.logits_bf16 ? argmax_partial_kernel<true> : argmax_partial_kernel<false>),
                               grid, dim3(256), 0, s, p);
    if (e != cudaSuccess) return e;
  }
  const int C = walk_cluster(p.Hkv);
  if (p.stage_bytes > 48 * 1024) {
    const cudaError_t e = ensure_max_dynamic_smem<walk_commit_kernel>(p.stage_bytes);
    if (e != cudaSuccess) return e;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(C, p.B);
  cfg.blockDim = dim3(kWalkThreads);
  cfg.dynamicSmemBytes = (size_t)p.stage_bytes;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = C;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, walk_commit_kernel, p);
}

}  // namespace tv
