// Dynamic draft-tree expansion ("ADR-037 — EAGLE-3 with dynamic tree port",
// phase rows E4a and E4b.10a, §4 Phase E4), one step per call:
//
//   draft_topk_kernel   grid (vocabulary chunks, expanded rows): each CTA
//                       reads one chunk of one row of draft logits once and
//                       leaves its top-K entries (largest first, smaller
//                       index on ties) and its log-sum-exp partial (running
//                       maximum, sum of exponentials).
//   expand_step_kernel  one CTA per tree: merges the chunks of each expanded
//                       row into its top-K children with float64 cumulative
//                       log-probabilities, ranks them together with the
//                       pending pool, moves the best W into the tree and
//                       keeps the pool sorted in the workspace.
//
// The pool never holds more than N - size entries: an entry ranked below
// that many others can never enter the tree, since every later candidate is
// inserted, never removed, ahead of it.  So one tree's whole state is a few
// hundred bytes and a step is one pass of ranks (binary searches in sorted
// runs) instead of a heap.
#include <cmath>
#include <cstdint>

#include "tree_expand.h"
#include "tv_internal.cuh"

namespace tv {
namespace {

constexpr int kXK = 16;          // largest top_k
constexpr int kXW = 16;          // largest width
constexpr int kXN = 64;          // largest max_nodes
constexpr int kXChunks = 64;     // largest number of vocabulary chunks per row
constexpr int kXThreads = 256;
constexpr int kXMaxBatch = 4095; // rows of one step (batch x width) fit a grid's y dimension
constexpr int32_t kXMagic = 0x54455850;
constexpr float kLog2e = 1.4426950408889634f;

// One tree's state between steps (in the workspace).
struct XState {
  int32_t magic, step, n_nodes, pool_n;
  int32_t gen, exp_count, done, pad;
  int32_t exp_node[kXW];                 // nodes the next step expands (row j = exp_node[j])
  double pool_cum[kXN];                  // pending candidates, sorted: best first
  int32_t pool_parent[kXN], pool_token[kXN], pool_depth[kXN], pool_order[kXN];
};

// An entry of a top-K list: logit and vocabulary index (i < 0: empty).
struct Ent {
  float v;
  int i;
};

// a comes before b: a valid entry before an empty one, the larger logit
// first, equal logits in increasing index order (NaN never enters a list).
__device__ __forceinline__ bool ent_before(Ent a, Ent b) {
  if (a.i < 0) return false;
  if (b.i < 0) return true;
  if (a.v != b.v) return a.v > b.v;
  return a.i < b.i;
}

__device__ __forceinline__ Ent warp_first(Ent e) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    Ent o{__shfl_xor_sync(0xffffffffu, e.v, off), __shfl_xor_sync(0xffffffffu, e.i, off)};
    if (ent_before(o, e)) e = o;
  }
  return e;
}

// A thread's KT best entries, sorted.  Entries arrive in increasing index
// order, so a new entry equal to the last one held loses the tie.
template <int KT>
struct TopList {
  Ent e[KT];
  __device__ __forceinline__ void init() {
#pragma unroll
    for (int q = 0; q < KT; ++q) e[q] = Ent{-INFINITY, -1};
  }
  __device__ __forceinline__ void push(float x, int idx) {
    if (!(e[KT - 1].i < 0 || x > e[KT - 1].v)) return;
    e[KT - 1] = Ent{x, idx};
#pragma unroll
    for (int q = KT - 1; q > 0; --q) {
      if (ent_before(e[q], e[q - 1])) {
        const Ent t = e[q];
        e[q] = e[q - 1];
        e[q - 1] = t;
      }
    }
  }
  __device__ __forceinline__ void pop() {
#pragma unroll
    for (int q = 0; q + 1 < KT; ++q) e[q] = e[q + 1];
    e[KT - 1] = Ent{-INFINITY, -1};
  }
};

template <bool BF16>
__device__ __forceinline__ float load_logit(const void* base, int64_t e) {
  if (BF16) return __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(base)[e]);
  return reinterpret_cast<const float*>(base)[e];
}

// (m, s) pairs of a log-sum-exp: s = sum of exp(x - m); m = -inf means empty.
__device__ __forceinline__ void lse_combine(float& m, double& s, float m2, double s2) {
  const float M = fmaxf(m, m2);
  double r = 0.0;
  if (m > -INFINITY) r += s * (double)exp2f((m - M) * kLog2e);
  if (m2 > -INFINITY) r += s2 * (double)exp2f((m2 - M) * kLog2e);
  m = M;
  s = r;
}

// grid (vchunks, B * R).  Row j of tree b starts at element b * seq_stride +
// j * V.  Leaves, per (row, chunk): the chunk's top-K in pv / pi (stride
// kXK), its maximum in pm (+inf when the chunk holds +inf) and its sum of
// exponentials in ps.
template <bool BF16, int KT>
__global__ __launch_bounds__(kXThreads) void draft_topk_kernel(const void* __restrict__ logits, int64_t seq_stride,
                                                               int V, int R, int vlen, int vchunks, int K, int vec,
                                                               float* __restrict__ pv, int32_t* __restrict__ pi,
                                                               float* __restrict__ pm, double* __restrict__ ps) {
  constexpr int ES = BF16 ? 2 : 4;
  const int row = blockIdx.y, c = blockIdx.x;
  const int b = row / R, j = row - b * R;
  const int64_t rbase = (int64_t)b * seq_stride + (int64_t)j * V;
  const int v0 = c * vlen;                       // a multiple of 8
  const int v1 = min(V, v0 + vlen);
  {
    const char* base = reinterpret_cast<const char*>(logits) + (rbase + v0) * ES;
    const int64_t bytes = (int64_t)(v1 - v0) * ES;
    for (int64_t off = (int64_t)threadIdx.x * 128; off < bytes; off += 128 * (int64_t)blockDim.x)
      prefetch_l2(base + off);
  }
  dep_wait();
  dep_launch();

  TopList<KT> L;
  L.init();
  float m = -INFINITY, s = 0.f;
  bool bad = false;
  auto take = [&](float x, int idx) {
    if (x != x) return;                          // NaN: never a child, not in the sum
    if (x == INFINITY) {
      bad = true;
      return;
    }
    if (x > m) {
      s = s * exp2f((m - x) * kLog2e) + 1.f;
      m = x;
    } else if (x > -INFINITY) {
      s += exp2f((x - m) * kLog2e);
    }
    L.push(x, idx);
  };
  if (vec) {
    constexpr int VE = 16 / ES;                  // elements per 16-byte load
    for (int e = v0 + (int)threadIdx.x * VE; e < v1; e += (int)blockDim.x * VE) {
      if (e + VE <= v1) {
        const uint4 u = *reinterpret_cast<const uint4*>(reinterpret_cast<const char*>(logits) + (rbase + e) * ES);
        float x[VE];
        if (BF16) {
          const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w[q]));
            x[2 * q] = f.x;
            x[2 * q + 1] = f.y;
          }
        } else {
          x[0] = __uint_as_float(u.x);
          x[1] = __uint_as_float(u.y);
          x[2] = __uint_as_float(u.z);
          x[3] = __uint_as_float(u.w);
        }
#pragma unroll
        for (int q = 0; q < VE; ++q) take(x[q], e + q);
      } else {
        for (int q = 0; e + q < v1; ++q) take(load_logit<BF16>(logits, rbase + e + q), e + q);
      }
    }
  } else {
    for (int e = v0 + (int)threadIdx.x; e < v1; e += blockDim.x) take(load_logit<BF16>(logits, rbase + e), e);
  }

  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  constexpr int NW = kXThreads / 32;
  __shared__ Ent wtop[NW][KT];
  __shared__ float red_m[NW];
  __shared__ double red_s[NW];

  // log-sum-exp partial
  double sd = s;
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    const float m2 = __shfl_xor_sync(0xffffffffu, m, off);
    const double s2 = __shfl_xor_sync(0xffffffffu, sd, off);
    lse_combine(m, sd, m2, s2);
  }
  if (lane == 0) {
    red_m[warp] = m;
    red_s[warp] = sd;
  }
  // top-K of each warp: K rounds of the warp's first head
  for (int r = 0; r < K; ++r) {
    const Ent best = warp_first(L.e[0]);
    if (best.i >= 0 && L.e[0].i == best.i) L.pop();
    if (lane == 0) wtop[warp][r] = best;
  }
  const int any_bad = __syncthreads_or(bad);
  const int64_t slot = (int64_t)row * vchunks + c;
  if (warp == 0) {
    int pos = 0;
    for (int r = 0; r < K; ++r) {
      const Ent h = (lane < NW && pos < K) ? wtop[lane][pos] : Ent{-INFINITY, -1};
      const Ent best = warp_first(h);
      if (lane < NW && h.i >= 0 && h.i == best.i) ++pos;
      if (lane == 0) {
        pv[slot * kXK + r] = best.v;
        pi[slot * kXK + r] = best.i;
      }
    }
    if (lane == 0) {
      float M = red_m[0];
      double S = red_s[0];
      for (int w = 1; w < NW; ++w) lse_combine(M, S, red_m[w], red_s[w]);
      pm[slot] = any_bad ? INFINITY : M;
      ps[slot] = S;
    }
  }
}

struct XParams {
  const float* pv;
  const int32_t* pi;
  const float* pm;
  const double* ps;
  const int32_t* root_tokens;
  const int32_t* token_map;
  int32_t* tokens;
  int32_t* parents;
  int32_t* depths;
  double* cum;
  int32_t* n_nodes;
  int32_t* expand_count;
  XState* state;
  int32_t* status;
  int step, R, vchunks, K, W, N, max_depth;
};

// a precedes b in the pool order: larger cumulative log-probability first,
// equal values to the candidate generated first (orders are unique).
__device__ __forceinline__ bool cand_before(double ca, int oa, double cb, int ob) {
  return ca > cb || (ca == cb && oa < ob);
}

// Entries of the sorted run (cum[0..n), order[0..n)) that precede (c, o).
__device__ __forceinline__ int count_before(const double* cum, const int* order, int n, double c, int o) {
  int lo = 0, hi = n;
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    if (cand_before(cum[mid], order[mid], c, o)) lo = mid + 1;
    else hi = mid;
  }
  return lo;
}

// grid (B): one CTA per tree.
__global__ __launch_bounds__(kXThreads) void expand_step_kernel(XParams p) {
  const int b = blockIdx.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  constexpr int NW = kXThreads / 32;
  XState* st = p.state + b;
  int32_t* tok = p.tokens + (int64_t)b * p.N;
  int32_t* par = p.parents + (int64_t)b * p.N;
  int32_t* dep = p.depths + (int64_t)b * p.N;
  double* cum = p.cum + (int64_t)b * p.N;

  __shared__ int s_ok, s_n, s_pool_n, s_gen, s_exp_count, s_done;
  __shared__ int s_exp_node[kXW], s_exp_depth[kXW], s_count[kXW];
  __shared__ double s_exp_cum[kXW];
  __shared__ double c_cum[kXW * kXK];            // new candidates, row j at [j * K, j * K + count_j)
  __shared__ int c_parent[kXW * kXK], c_token[kXW * kXK], c_depth[kXW * kXK], c_order[kXW * kXK];
  __shared__ double q_cum[kXN];                   // pending pool (sorted)
  __shared__ int q_parent[kXN], q_token[kXN], q_depth[kXN], q_order[kXN];

  dep_wait();
  dep_launch();

  if (tid == 0) {
    if (p.step == 0) {
      s_ok = 1;
      s_n = 1;
      s_pool_n = 0;
      s_gen = 0;
      s_exp_count = 1;
      s_done = 0;
      s_exp_node[0] = 0;
    } else {
      // the state must be the one step - 1 left for this descriptor
      // (anything else, e.g. a workspace of another expansion, is refused)
      const int n = st->n_nodes, pn = st->pool_n, ec = st->exp_count;
      int ok = st->magic == kXMagic && st->step == p.step - 1 && n >= 1 && n <= p.N && pn >= 0 &&
               pn <= p.N - n && ec >= 0 && ec <= p.R && ec < n;
      for (int j = 0; ok && j < ec; ++j) {
        const int u = st->exp_node[j];
        ok = u >= 1 && u < n;
        s_exp_node[j] = u;
      }
      s_ok = ok;
      if (!ok) {
        set_status(p.status, TV_DEV_BAD_STEP);
      } else {
        s_n = n;
        s_pool_n = pn;
        s_gen = st->gen;
        s_exp_count = ec;
        s_done = st->done;
      }
    }
  }
  __syncthreads();
  if (!s_ok) return;
  if (p.step == 0) {
    for (int i = tid; i < p.N; i += blockDim.x) {
      tok[i] = i ? -1 : p.root_tokens[b];
      par[i] = -1;
      dep[i] = i ? -1 : 0;
      cum[i] = i ? -INFINITY : 0.0;
    }
  }
  if (s_done) {
    if (tid == 0) {
      st->step = p.step;
      p.n_nodes[b] = s_n;
      p.expand_count[b] = 0;
    }
    return;
  }
  const int E = s_exp_count, K = p.K, P = s_pool_n;
  if (tid < kXW) s_count[tid] = 0;
  if (tid < E) {
    const int u = s_exp_node[tid];
    s_exp_depth[tid] = p.step == 0 ? 0 : dep[u];
    s_exp_cum[tid] = p.step == 0 ? 0.0 : cum[u];
  }
  if (tid < P) {
    q_cum[tid] = st->pool_cum[tid];
    q_parent[tid] = st->pool_parent[tid];
    q_token[tid] = st->pool_token[tid];
    q_depth[tid] = st->pool_depth[tid];
    q_order[tid] = st->pool_order[tid];
  }
  __syncthreads();

  // children of each expanded row: warp j % NW merges row j's chunks
  const int vc = p.vchunks;
  for (int j = warp; j < E; j += NW) {
    if (s_exp_depth[j] >= p.max_depth) continue;   // at the depth limit: no children
    const int64_t row = (int64_t)b * p.R + j;
    const float* pm = p.pm + row * vc;
    const double* ps = p.ps + row * vc;
    float M = -INFINITY;
    bool bad = false;
    for (int c = lane; c < vc; c += 32) {
      const float mc = pm[c];
      if (mc == INFINITY) bad = true;
      else M = fmaxf(M, mc);
    }
    if (__any_sync(0xffffffffu, bad)) {
      if (lane == 0) set_status(p.status, TV_DEV_BAD_LOGITS);
      continue;
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
    double S = 0.0;
    for (int c = lane; c < vc; c += 32) {
      const float mc = pm[c];
      if (mc > -INFINITY) S += ps[c] * (double)exp2f((mc - M) * kLog2e);
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) S += __shfl_xor_sync(0xffffffffu, S, off);
    const bool all_ninf = !(M > -INFINITY);
    const double lse = all_ninf ? -INFINITY : (double)M + log(S);
    const float* pv = p.pv + row * vc * kXK;
    const int32_t* pi = p.pi + row * vc * kXK;
    int p0 = 0, p1 = 0;                            // heads of chunks lane and lane + 32
    int cnt = 0;
    for (int r = 0; r < K; ++r) {
      const int c0 = lane, c1 = lane + 32;
      const Ent h0 = (c0 < vc && p0 < K) ? Ent{pv[(int64_t)c0 * kXK + p0], pi[(int64_t)c0 * kXK + p0]}
                                         : Ent{-INFINITY, -1};
      const Ent h1 = (c1 < vc && p1 < K) ? Ent{pv[(int64_t)c1 * kXK + p1], pi[(int64_t)c1 * kXK + p1]}
                                         : Ent{-INFINITY, -1};
      const Ent h = ent_before(h1, h0) ? h1 : h0;
      const Ent best = warp_first(h);
      if (best.i < 0) break;                       // the row has no more valid entries
      if (h0.i == best.i) ++p0;
      else if (h1.i == best.i) ++p1;
      if (lane == 0) {
        const int sl = j * K + r;
        c_cum[sl] = all_ninf ? -INFINITY : s_exp_cum[j] + ((double)best.v - lse);
        c_token[sl] = p.token_map ? p.token_map[best.i] : best.i;
        c_parent[sl] = s_exp_node[j];
        c_depth[sl] = s_exp_depth[j] + 1;
        c_order[sl] = s_gen + sl;
      }
      cnt = r + 1;
    }
    if (lane == 0) s_count[j] = cnt;
  }
  __syncthreads();

  // rank every pending and new candidate in the union; the first `pops`
  // enter the tree, the next up to N - size - pops stay pending
  int total = P;
  for (int j = 0; j < E; ++j) total += s_count[j];
  const int keep = p.N - s_n;
  int pops = p.W < keep ? p.W : keep;
  if (pops > total) pops = total;
  __shared__ double n_cum[kXN];
  __shared__ int n_parent[kXN], n_token[kXN], n_depth[kXN], n_order[kXN];
  for (int t = tid; t < P + E * K; t += blockDim.x) {
    double c;
    int o, pa, tk, dp, rank;
    if (t < P) {
      c = q_cum[t];
      o = q_order[t];
      pa = q_parent[t];
      tk = q_token[t];
      dp = q_depth[t];
      rank = t;
      for (int j = 0; j < E; ++j) rank += count_before(c_cum + j * K, c_order + j * K, s_count[j], c, o);
    } else {
      const int sl = t - P, j = sl / K, r = sl - j * K;
      if (r >= s_count[j]) continue;
      c = c_cum[sl];
      o = c_order[sl];
      pa = c_parent[sl];
      tk = c_token[sl];
      dp = c_depth[sl];
      rank = r + count_before(q_cum, q_order, P, c, o);
      for (int j2 = 0; j2 < E; ++j2)
        if (j2 != j) rank += count_before(c_cum + j2 * K, c_order + j2 * K, s_count[j2], c, o);
    }
    if (rank < pops) {
      const int i = s_n + rank;
      tok[i] = tk;
      par[i] = pa;
      dep[i] = dp;
      cum[i] = c;
    } else if (rank < keep) {
      const int q = rank - pops;
      n_cum[q] = c;
      n_parent[q] = pa;
      n_token[q] = tk;
      n_depth[q] = dp;
      n_order[q] = o;
    }
  }
  __syncthreads();
  const int remain = (total < keep ? total : keep) - pops;
  if (tid < remain) {
    st->pool_cum[tid] = n_cum[tid];
    st->pool_parent[tid] = n_parent[tid];
    st->pool_token[tid] = n_token[tid];
    st->pool_depth[tid] = n_depth[tid];
    st->pool_order[tid] = n_order[tid];
  }
  if (tid < pops) st->exp_node[tid] = s_n + tid;
  if (tid == 0) {
    const int n = s_n + pops;
    const int done = n >= p.N || pops == 0;
    st->magic = kXMagic;
    st->step = p.step;
    st->n_nodes = n;
    st->pool_n = remain;
    st->gen = s_gen + E * K;
    st->exp_count = pops;
    st->done = done;
    p.n_nodes[b] = n;
    p.expand_count[b] = done ? 0 : pops;
  }
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int64_t align_up(int64_t x, int64_t a) { return (x + a - 1) / a * a; }

int x_validate(const tv_expand_desc* d) {
  if (!d) return TV_ERR_NULL;
  if (d->logits_dtype != TV_F32 && d->logits_dtype != TV_BF16) return TV_ERR_DTYPE;
  if (d->batch < 1 || d->batch > kXMaxBatch || d->vocab < 1 || d->vocab > (1 << 30) || d->top_k < 1 ||
      d->top_k > kXK || d->width < 1 || d->width > kXW || d->max_nodes < 1 || d->max_nodes > kXN ||
      d->max_depth < 1)
    return TV_ERR_SHAPE;
  return TV_OK;
}

// Vocabulary chunks per row: about two CTAs per SM over all rows, at least
// 1024 entries per chunk, at most kXChunks chunks; chunk lengths are
// multiples of 8 so 16-byte loads stay aligned.
void x_chunks(int64_t rows, int V, int* vchunks, int* vlen) {
  int64_t want = (2 * (int64_t)num_sms() + rows - 1) / rows;
  int64_t maxc = ((int64_t)V + 1023) / 1024;
  if (maxc > kXChunks) maxc = kXChunks;
  if (maxc < 1) maxc = 1;
  if (want > maxc) want = maxc;
  if (want < 1) want = 1;
  int64_t len = ((int64_t)V + want - 1) / want;
  len = (len + 7) / 8 * 8;
  *vlen = (int)len;
  *vchunks = (int)(((int64_t)V + len - 1) / len);
}

struct XLayout {
  int64_t state, pv, pi, pm, ps, total;
};

XLayout x_layout(const tv_expand_desc* d) {
  const int64_t rows = (int64_t)d->batch * d->width;
  XLayout l;
  int64_t off = 0;
  l.state = off;
  off = align_up(off + (int64_t)d->batch * (int64_t)sizeof(XState), 256);
  l.pv = off;
  off = align_up(off + rows * kXChunks * kXK * 4, 256);
  l.pi = off;
  off = align_up(off + rows * kXChunks * kXK * 4, 256);
  l.pm = off;
  off = align_up(off + rows * kXChunks * 4, 256);
  l.ps = off;
  off = align_up(off + rows * kXChunks * 8, 256);
  l.total = off;
  return l;
}

template <bool BF16>
cudaError_t launch_topk(int KT, dim3 grid, cudaStream_t s, const void* logits, int64_t stride, int V, int R, int vlen,
                        int vc, int K, int vec, float* pv, int32_t* pi, float* pm, double* ps) {
  switch (KT) {
    case 1: return launch_dep(draft_topk_kernel<BF16, 1>, grid, dim3(kXThreads), 0, s, logits, stride, V, R, vlen, vc, K, vec, pv, pi, pm, ps);
    case 2: return launch_dep(draft_topk_kernel<BF16, 2>, grid, dim3(kXThreads), 0, s, logits, stride, V, R, vlen, vc, K, vec, pv, pi, pm, ps);
    case 4: return launch_dep(draft_topk_kernel<BF16, 4>, grid, dim3(kXThreads), 0, s, logits, stride, V, R, vlen, vc, K, vec, pv, pi, pm, ps);
    case 8: return launch_dep(draft_topk_kernel<BF16, 8>, grid, dim3(kXThreads), 0, s, logits, stride, V, R, vlen, vc, K, vec, pv, pi, pm, ps);
    default: return launch_dep(draft_topk_kernel<BF16, 16>, grid, dim3(kXThreads), 0, s, logits, stride, V, R, vlen, vc, K, vec, pv, pi, pm, ps);
  }
}

}  // namespace
}  // namespace tv

using namespace tv;

extern "C" {

int tv_expand_workspace_size(const tv_expand_desc* desc, size_t* bytes) {
  const int rc = x_validate(desc);
  if (rc) return rc;
  if (!bytes) return TV_ERR_NULL;
  *bytes = (size_t)x_layout(desc).total;
  return TV_OK;
}

int tv_expand_steps(const tv_expand_desc* desc, int32_t* steps) {
  const int rc = x_validate(desc);
  if (rc) return rc;
  if (!steps) return TV_ERR_NULL;
  const int64_t kids = desc->top_k < desc->vocab ? desc->top_k : desc->vocab;
  const int64_t N = desc->max_nodes, W = desc->width;
  int64_t size = 1, pending = kids, n = 0;
  for (;;) {
    int64_t pops = W < pending ? W : pending;
    if (pops > N - size) pops = N - size;
    size += pops;
    pending -= pops;
    ++n;
    if (size >= N || pops == 0) break;
    pending += pops * kids;
  }
  *steps = (int32_t)n;
  return TV_OK;
}

int tv_tree_expand_step(const tv_expand_desc* desc, int32_t step, const void* d_logits, int64_t seq_stride,
                        const int32_t* d_root_tokens, const int32_t* d_token_map, int32_t* d_tokens,
                        int32_t* d_parents, int32_t* d_depths, double* d_cum, int32_t* d_n_nodes,
                        int32_t* d_expand_count, void* d_workspace, size_t workspace_bytes,
                        int32_t* d_status, void* stream) {
  int rc = x_validate(desc);
  if (rc) return rc;
  if (!d_logits || !d_tokens || !d_parents || !d_depths || !d_cum || !d_n_nodes || !d_expand_count ||
      !d_workspace || !d_status || (step == 0 && !d_root_tokens))
    return TV_ERR_NULL;
  const int V = desc->vocab;
  const int R = step == 0 ? 1 : desc->width;
  int64_t min_stride = 0;
  if (step < 0 || __builtin_mul_overflow((int64_t)R, (int64_t)V, &min_stride) || seq_stride < min_stride)
    return TV_ERR_SHAPE;
  const int ES = desc->logits_dtype == TV_BF16 ? 2 : 4;
  int64_t span = 0;
  if (__builtin_mul_overflow(seq_stride, (int64_t)desc->batch, &span) || __builtin_mul_overflow(span, (int64_t)ES, &span))
    return TV_ERR_OVERFLOW;
  const void* ptrs[] = {d_logits, d_tokens, d_parents, d_depths, d_cum, d_n_nodes, d_expand_count, d_workspace, d_status};
  for (const void* q : ptrs)
    if (!aligned16(q)) return TV_ERR_ALIGN;
  if ((d_root_tokens && !aligned16(d_root_tokens)) || (d_token_map && !aligned16(d_token_map))) return TV_ERR_ALIGN;
  const XLayout l = x_layout(desc);
  if ((int64_t)workspace_bytes < l.total) return TV_ERR_WORKSPACE;

  char* ws = static_cast<char*>(d_workspace);
  float* pv = reinterpret_cast<float*>(ws + l.pv);
  int32_t* pi = reinterpret_cast<int32_t*>(ws + l.pi);
  float* pm = reinterpret_cast<float*>(ws + l.pm);
  double* ps = reinterpret_cast<double*>(ws + l.ps);
  const int64_t rows = (int64_t)desc->batch * R;
  int vc = 1, vlen = V;
  x_chunks(rows, V, &vc, &vlen);
  const int K = desc->top_k;
  const int KT = K <= 1 ? 1 : K <= 2 ? 2 : K <= 4 ? 4 : K <= 8 ? 8 : 16;
  const int vec = ((int64_t)V * ES) % 16 == 0 && (seq_stride * ES) % 16 == 0;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const dim3 grid(vc, (unsigned)rows);
  cudaError_t e = desc->logits_dtype == TV_BF16
                      ? launch_topk<true>(KT, grid, s, d_logits, seq_stride, V, R, vlen, vc, K, vec, pv, pi, pm, ps)
                      : launch_topk<false>(KT, grid, s, d_logits, seq_stride, V, R, vlen, vc, K, vec, pv, pi, pm, ps);
  if (e != cudaSuccess) return TV_ERR_CUDA;
  XParams xp;
  xp.pv = pv;
  xp.pi = pi;
  xp.pm = pm;
  xp.ps = ps;
  xp.root_tokens = d_root_tokens;
  xp.token_map = d_token_map;
  xp.tokens = d_tokens;
  xp.parents = d_parents;
  xp.depths = d_depths;
  xp.cum = d_cum;
  xp.n_nodes = d_n_nodes;
  xp.expand_count = d_expand_count;
  xp.state = reinterpret_cast<XState*>(ws + l.state);
  xp.status = d_status;
  xp.step = step;
  xp.R = R;
  xp.vchunks = vc;
  xp.K = K;
  xp.W = desc->width;
  xp.N = desc->max_nodes;
  xp.max_depth = desc->max_depth;
  e = launch_dep(expand_step_kernel, dim3(desc->batch), dim3(kXThreads), 0, s, xp);
  return e == cudaSuccess ? TV_OK : TV_ERR_CUDA;
}

}  // extern "C"
