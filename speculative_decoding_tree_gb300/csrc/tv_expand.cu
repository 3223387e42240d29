// Dynamic draft-tree expansion ("ADR-037 — EAGLE-3 with dynamic tree port",
// phase rows E4a and E4b.10a, §4 Phase E4), one step per call:
//
//   draft_topk_kernel   grid (vocabulary chunks, expanded rows): each
//                       CTA reads one chunk of one row of draft logits and
//                       leaves its top-K entries (largest first, smaller
//                       index on ties) and its log-sum-exp partial (maximum,
//                       sum of exponentials).
//   expand_step_kernel  one CTA per tree: merges the chunks of each expanded
//                       row into its top-K children with float64 cumulative
//                       log-probabilities, ranks them together with the
//                       pending pool, moves the best W into the tree and
//                       keeps the pool sorted in the workspace.
//
// The pool never holds more than N - size entries: an entry ranked below
// that many others can never enter the tree, since every later candidate is
// inserted, never removed, ahead of it.  So one tree's whole state is a few
// hundred bytes and a step is one pass of ranks (each entry counts the
// entries of the union that precede it) instead of a heap.
#include <cmath>
#include <cstdint>

#include "tree_expand.h"
#include "tv_internal.cuh"
#include "tv_select.cuh"

namespace tv {
namespace {

constexpr int kXK = 16;          // largest top_k
constexpr int kXW = 16;          // largest width
constexpr int kXN = 64;          // largest max_nodes
constexpr int kXThreads = 256;
constexpr int kXMaxBatch = 4095; // rows of one step (batch x width) fit a grid's y dimension
constexpr int32_t kXMagic = 0x54455850;
constexpr float kLog2e = 1.4426950408889634f;

// One tree's state between steps (in the workspace).  Cumulative
// log-probabilities are float pairs (hi + lo, see DF below).
struct XState {
  int32_t magic, step, n_nodes, pool_n;
  int32_t gen, exp_count, done, pad;
  int32_t exp_node[kXW];                 // nodes the next step expands (row j = exp_node[j])
  float pool_hi[kXN], pool_lo[kXN];      // pending candidates, sorted: best first
  int32_t pool_parent[kXN], pool_token[kXN], pool_depth[kXN], pool_order[kXN];
  float node_hi[kXN], node_lo[kXN];      // the tree's nodes
  int32_t node_depth[kXN];
};


static_assert(sizeof(XState) % 16 == 0, "the state is copied in 16-byte units");
static_assert(kXN == 64, "");

// Double-float arithmetic.  A value is hi + lo with |lo| <= ulp(hi) / 2
// (about 48 significant bits), computed with float32 error-free
// transformations (Knuth's two-sum, Dekker's fast two-sum).  Float64
// arithmetic on this part has a dependent latency of about 30-70 ns per
// operation (against about 2 ns in float32), and the step is a chain of
// dependent operations, so the cumulative log-probabilities are carried as
// float pairs and converted to float64 only when written out.
struct DF {
  float hi, lo;
};

__device__ __forceinline__ DF df_norm(float s, float e) {   // |e| small against s
  if (!(fabsf(s) < INFINITY)) return DF{s, 0.f};
  const float h = __fadd_rn(s, e);
  return DF{h, __fsub_rn(e, __fsub_rn(h, s))};
}

__device__ __forceinline__ DF df_add(DF a, DF b) {
  const float s = __fadd_rn(a.hi, b.hi);
  if (!(fabsf(s) < INFINITY)) return DF{s, 0.f};
  const float bb = __fsub_rn(s, a.hi);
  const float e = __fadd_rn(__fsub_rn(a.hi, __fsub_rn(s, bb)), __fsub_rn(b.hi, bb));
  return df_norm(s, __fadd_rn(e, __fadd_rn(a.lo, b.lo)));
}

__device__ __forceinline__ DF df_neg(DF a) { return DF{-a.hi, -a.lo}; }

// a * f for a float f >= 0 (the product's rounding error recovered by an fma)
__device__ __forceinline__ DF df_mulf(DF a, float f) {
  const float p = __fmul_rn(a.hi, f);
  if (!(fabsf(p) < INFINITY)) return DF{p, 0.f};
  const float e = __fmaf_rn(a.hi, f, -p);
  return df_norm(p, __fmaf_rn(a.lo, f, e));
}

// log(S) for 1 <= S < 2^30: S = m * 2^e with m in [1, 2), e * ln2 with ln2
// split so that e * ln2_hi is exact, plus logf(m) (at most 1 ulp of a value
// below 0.7): within about 1e-7.
__device__ __forceinline__ DF df_log_ge1(DF S) {
  int e;
  const float m2 = frexpf(S.hi, &e);                      // S.hi = m2 * 2^e, m2 in [0.5, 1)
  const float m = 2.f * m2;
  const float le = (float)(e - 1);
  const DF a = df_add(DF{le * 0.693145751953125f, 0.f}, DF{le * 1.428606765330187e-06f, 0.f});
  // log(S.hi + S.lo) = log(S.hi) + S.lo / S.hi to first order
  return df_add(a, DF{logf(m), __fdiv_rn(S.lo, S.hi)});
}

// An integer with the order of the double-float value (hi, then lo): the
// pool compares these instead of floating-point values.
__device__ __forceinline__ uint64_t df_key(DF a) { return ((uint64_t)val_key(a.hi) << 32) | val_key(a.lo); }

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

// The top-K pass: CTAs of kXTopkThreads threads, each reading one chunk of
// one row in tiles of kXTopkThreads * PT entries (thread t holds PT entries of
// a tile, in increasing index order; PT = 16, or 32 when a step has so many
// rows that 16 would take more than two waves of CTAs).
constexpr int kXTopkThreads = 512;
constexpr int kXRowEntries = 512;                    // chunks x K per row (the step stages them in shared memory)
constexpr int kXCand = 1024;                         // candidates a CTA ranks directly

// Vocabulary index of entry k of the thread's share of the tile at t0.
template <bool BF16>
__device__ __forceinline__ int tile_index(int t0, int k, int vec) {
  constexpr int VE = 16 / (BF16 ? 2 : 4);
  if (vec) return t0 + ((k / VE) * kXTopkThreads + (int)threadIdx.x) * VE + (k % VE);
  return t0 + k * kXTopkThreads + (int)threadIdx.x;
}

// Loads the thread's PT entries of one tile (NaN where the chunk ends).
// vec: 16-byte loads (rows 16-byte aligned).
template <bool BF16, int PT>
__device__ __forceinline__ void load_tile(const void* logits, int64_t rbase, int t0, int v1, int vec, float x[PT]) {
  constexpr int ES = BF16 ? 2 : 4;
  constexpr int VE = 16 / ES;
  if (vec) {
#pragma unroll
    for (int g = 0; g < PT / VE; ++g) {
      const int e = t0 + (g * kXTopkThreads + (int)threadIdx.x) * VE;
      if (e + VE <= v1) {
        const uint4 u = *reinterpret_cast<const uint4*>(reinterpret_cast<const char*>(logits) + (rbase + e) * ES);
        const uint32_t w[4] = {u.x, u.y, u.z, u.w};
        if (BF16) {
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w[q]));
            x[g * VE + 2 * q] = f.x;
            x[g * VE + 2 * q + 1] = f.y;
          }
        } else {
#pragma unroll
          for (int q = 0; q < 4; ++q) x[g * VE + q] = __uint_as_float(w[q]);
        }
      } else {
#pragma unroll
        for (int q = 0; q < VE; ++q) x[g * VE + q] = e + q < v1 ? load_logit<BF16>(logits, rbase + e + q) : __int_as_float(0x7fffffff);
      }
    }
  } else {
#pragma unroll
    for (int g = 0; g < PT; ++g) {
      const int e = t0 + g * kXTopkThreads + (int)threadIdx.x;
      x[g] = e < v1 ? load_logit<BF16>(logits, rbase + e) : __int_as_float(0x7fffffff);
    }
  }
}

// grid (vchunks, B * R), kXTopkThreads threads.  Row j of tree b starts at
// element b * seq_stride + j * V; CTA c reads entries [c * vlen, (c+1) * vlen).
//
// Pass 1: each thread's first maximum; the CTA's maximum M, and a threshold T
// no larger than the CTA's K-th largest entry: the smallest of the warps'
// maxima (16 warps, K <= 16, so 16 distinct entries are >= T).  Pass 2: the
// sum of exp(x - M), and every entry >= T as a candidate; the candidates'
// first K by rank are the CTA's top-K.  (More than kXCand candidates, e.g. a
// chunk of equal logits: per-thread sorted lists and K rounds of warp
// merges instead.)  Leaves, per (row, chunk): the top-K in pv / pi at
// ((row * vchunks + chunk) * K, -1 indices after the valid entries), the
// maximum in pm (+inf when the chunk holds +inf) and the sum of
// exponentials in ps (a double-float: float32 per thread, pairs above).
template <bool BF16, int KT, int PT>
__global__ __launch_bounds__(kXTopkThreads) void draft_topk_kernel(const void* __restrict__ logits, int64_t seq_stride,
                                                                   int V, int R, int vlen, int vchunks, int K, int vec,
                                                                   float* __restrict__ pv, int32_t* __restrict__ pi,
                                                                   float* __restrict__ pm, float2* __restrict__ ps) {
  constexpr int ES = BF16 ? 2 : 4;
  constexpr int NW = kXTopkThreads / 32;
  const int row = blockIdx.y, c = blockIdx.x;
  const int b = row / R, j = row - b * R;
  const int64_t rbase = (int64_t)b * seq_stride + (int64_t)j * V;
  const int v0 = c * vlen;                       // a multiple of 8
  const int v1 = min(V, v0 + vlen);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  {
    const char* base = reinterpret_cast<const char*>(logits) + (rbase + v0) * ES;
    const int64_t bytes = (int64_t)(v1 - v0) * ES;
    for (int64_t off = (int64_t)threadIdx.x * 128; off < bytes; off += 128 * (int64_t)blockDim.x)
      prefetch_l2(base + off);
  }
  __shared__ float s_wmax[NW];
  __shared__ int s_wi[NW];
  __shared__ float s_sum[NW], s_sum_lo[NW];
  __shared__ int s_cnt;
  __shared__ uint64_t ck[kXCand];                // candidates as entry keys
  __shared__ Ent wtop[NW][KT];
  if (threadIdx.x == 0) s_cnt = 0;
  dep_wait();
  dep_launch();

  // pass 1: the thread's first maximum (NaN and +inf excluded); the first
  // tile stays in registers for pass 2
  constexpr int kTileElems = kXTopkThreads * PT;
  float x[PT];
  float tmax = -INFINITY;
  int tidx = -1;
  bool bad = false;
  const bool one_tile = v1 - v0 <= kTileElems;
  for (int t0 = v0; t0 < v1; t0 += kTileElems) {
    load_tile<BF16, PT>(logits, rbase, t0, v1, vec, x);
#pragma unroll
    for (int k = 0; k < PT; ++k) {
      const float xv = x[k];
      if (xv != xv) continue;
      if (xv == INFINITY) {
        bad = true;
        continue;
      }
      if (tidx < 0 || xv > tmax) {
        tmax = xv;
        tidx = tile_index<BF16>(t0, k, vec);
      }
    }
  }
  const Ent wm = warp_first(Ent{tmax, tidx});
  if (lane == 0) {
    s_wmax[warp] = wm.i >= 0 ? wm.v : -INFINITY;
    s_wi[warp] = wm.i;
  }
  const int any_bad = __syncthreads_or(bad);
  float M = -INFINITY, T = INFINITY;
  bool no_thr = false;
#pragma unroll
  for (int w = 0; w < NW; ++w) {
    M = fmaxf(M, s_wmax[w]);
    T = fminf(T, s_wmax[w]);
    no_thr |= s_wi[w] < 0;
  }
  if (no_thr) T = -INFINITY;                     // a warp without entries: every entry is a candidate

  // pass 2: sum of exponentials and candidates
  float s = 0.f;
  auto scan = [&](int t0) {
#pragma unroll
    for (int k = 0; k < PT; ++k) {
      const float xv = x[k];
      if (!(xv < INFINITY)) continue;            // NaN, +inf
      if (xv > -INFINITY) s += exp2f((xv - M) * kLog2e);
    }
    // candidates (>= T, not NaN, not +inf), appended with one shared
    // atomic per warp and tile (ballots counted first, then recomputed)
    int tot = 0;
#pragma unroll
    for (int k = 0; k < PT; ++k) tot += __popc(__ballot_sync(0xffffffffu, x[k] < INFINITY && x[k] >= T));
    if (tot == 0) return;                        // warp-uniform
    int base = 0;
    if (lane == 0) base = atomicAdd(&s_cnt, tot);
    base = __shfl_sync(0xffffffffu, base, 0);
    const uint32_t below = (1u << lane) - 1u;
#pragma unroll
    for (int k = 0; k < PT; ++k) {
      const bool cand = x[k] < INFINITY && x[k] >= T;
      const uint32_t m = __ballot_sync(0xffffffffu, cand);
      const int pos = base + __popc(m & below);
      if (cand && pos < kXCand) ck[pos] = ent_key(x[k], tile_index<BF16>(t0, k, vec));
      base += __popc(m);
    }
  };
  if (one_tile) {
    scan(v0);                                    // the tile pass 1 left in registers
  } else {
    for (int t0 = v0; t0 < v1; t0 += kTileElems) {
      load_tile<BF16, PT>(logits, rbase, t0, v1, vec, x);
      scan(t0);
    }
  }
  DF sw{s, 0.f};
#pragma unroll
  for (int off = 16; off > 0; off >>= 1)
    sw = df_add(sw, DF{__shfl_xor_sync(0xffffffffu, sw.hi, off), __shfl_xor_sync(0xffffffffu, sw.lo, off)});
  if (lane == 0) {
    s_sum[warp] = sw.hi;
    s_sum_lo[warp] = sw.lo;
  }
  __syncthreads();
  const int64_t slot = (int64_t)row * vchunks + c;
  const int n = s_cnt;
  float* ov = pv + slot * K;
  int32_t* oi = pi + slot * K;
  if (n <= kXCand) {
    // warp 0: K rounds, round r taking the largest key below round r - 1's
    // (keys are distinct; every lane scans the same number of slots, with
    // no branch on the data)
    if (warp == 0) {
      uint64_t prev = ~0ull;
      int r = 0;
      for (; r < K; ++r) {
        uint64_t mine = 0ull;
        for (int u0 = 0; u0 < n; u0 += 32) {
          const uint64_t k2 = u0 + lane < n ? ck[u0 + lane] : 0ull;
          mine = (k2 < prev && k2 > mine) ? k2 : mine;
        }
        const uint64_t w = warp_max_key(mine);
        if (w == 0ull) break;                      // fewer than K candidates
        prev = w;
        if (lane == 0) {
          const Ent best = key_ent(w);
          ov[r] = best.v;
          oi[r] = best.i;
        }
      }
      for (int r2 = r + lane; r2 < K; r2 += 32) {
        ov[r2] = -INFINITY;
        oi[r2] = -1;
      }
    }
  } else {
    // many equal entries: per-thread sorted lists, then K rounds of merges
    TopList<KT> L;
    L.init();
    for (int t0 = v0; t0 < v1; t0 += kTileElems) {
      load_tile<BF16, PT>(logits, rbase, t0, v1, vec, x);
#pragma unroll
      for (int k = 0; k < PT; ++k)
        if (x[k] < INFINITY) L.push(x[k], tile_index<BF16>(t0, k, vec));
    }
    for (int r = 0; r < K; ++r) {
      const Ent best = warp_first(L.e[0]);
      if (best.i >= 0 && L.e[0].i == best.i) L.pop();
      if (lane == 0) wtop[warp][r] = best;
    }
    __syncthreads();
    if (warp == 0) {
      int pos = 0;
      for (int r = 0; r < K; ++r) {
        const Ent h = (lane < NW && pos < K) ? wtop[lane][pos] : Ent{-INFINITY, -1};
        const Ent best = warp_first(h);
        if (lane < NW && h.i >= 0 && h.i == best.i) ++pos;
        if (lane == 0) {
          ov[r] = best.v;
          oi[r] = best.i;
        }
      }
    }
  }
  if (warp == 1) {                               // beside warp 0's rounds
    DF S = lane < NW ? DF{s_sum[lane], s_sum_lo[lane]} : DF{0.f, 0.f};
#pragma unroll
    for (int off = 16; off > 0; off >>= 1)
      S = df_add(S, DF{__shfl_xor_sync(0xffffffffu, S.hi, off), __shfl_xor_sync(0xffffffffu, S.lo, off)});
    if (lane == 0) {
      pm[slot] = any_bad ? INFINITY : M;
      ps[slot] = make_float2(S.hi, S.lo);
    }
  }
}

struct XParams {
  const float* pv;           // [B * R, vchunks, K] each chunk's top-K logits, largest first
  const int32_t* pi;         // their vocabulary indices (-1 after the valid entries)
  const float* pm;           // [B * R, vchunks] chunk maximum (+inf: the chunk holds +inf)
  const float2* ps;          // [B * R, vchunks] sum of exp(x - chunk maximum), double-float
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
__device__ __forceinline__ bool cand_before(uint64_t ka, int oa, uint64_t kb, int ob) {
  return ka > kb || (ka == kb && oa < ob);
}

// Order of an empty candidate slot: such a slot (key 0) precedes nothing.
constexpr int kXNoOrder = 0x7fffffff;

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
  __shared__ DF s_exp_cum[kXW];
  __shared__ DF c_cum[kXW * kXK];                // new candidates, row j at [j * K, j * K + count_j)
  __shared__ int c_parent[kXW * kXK], c_token[kXW * kXK], c_depth[kXW * kXK];
  __shared__ DF q_cum[kXN];                      // pending pool (sorted)
  __shared__ int q_parent[kXN], q_token[kXN], q_depth[kXN];
  // keys and orders of the union: pool entry t at slot t, new candidate
  // sl at slot P + sl (empty slots hold key 0, order kXNoOrder)
  __shared__ uint64_t u_key[kXN + kXW * kXK];
  __shared__ int u_ord[kXN + kXW * kXK];
  __shared__ __align__(16) XState s_st;

  // The state step - 1 left.  That grid completed before the top-K grid of
  // this step passed its own dependency wait, which comes before the moment
  // this grid may start, so it is read here, before this grid's wait, from
  // L2 (the top-K grid does not touch it).
  if (p.step > 0) {
    const uint4* src = reinterpret_cast<const uint4*>(st);
    uint4* dst = reinterpret_cast<uint4*>(&s_st);
    for (int i = tid; i < (int)(sizeof(XState) / 16); i += blockDim.x) dst[i] = __ldcg(src + i);
  }
  __syncthreads();
  if (tid == 0) {
    if (p.step == 0) {
      s_ok = 1;
      s_n = 1;
      s_pool_n = 0;
      s_gen = 0;
      s_exp_count = 1;
      s_done = 0;
      s_exp_node[0] = 0;
      s_st.node_hi[0] = 0.f;
      s_st.node_lo[0] = 0.f;
      s_st.node_depth[0] = 0;
    } else {
      // the state must be the one step - 1 left for this descriptor
      // (anything else, e.g. a workspace of another expansion, is refused)
      const int n = s_st.n_nodes, pn = s_st.pool_n, ec = s_st.exp_count;
      int ok = s_st.magic == kXMagic && s_st.step == p.step - 1 && n >= 1 && n <= p.N && pn >= 0 &&
               pn <= p.N - n && ec >= 0 && ec <= p.R && ec < n;
      for (int j = 0; ok && j < ec; ++j) {
        const int u = s_st.exp_node[j];
        ok = u >= 1 && u < n;
        s_exp_node[j] = u;
      }
      s_ok = ok;
      if (!ok) {
        set_status(p.status, TV_DEV_BAD_STEP);
      } else {
        s_n = n;
        s_pool_n = pn;
        s_gen = s_st.gen;
        s_exp_count = ec;
        s_done = s_st.done;
      }
    }
  }
  __syncthreads();
  if (!s_ok) {
    dep_wait();
    dep_launch();
    return;
  }
  const int E = s_exp_count, K = p.K, P = s_pool_n;
  if (tid < kXW) s_count[tid] = 0;
  if (tid < E) {
    const int u = s_exp_node[tid];
    s_exp_depth[tid] = s_st.node_depth[u];
    s_exp_cum[tid] = DF{s_st.node_hi[u], s_st.node_lo[u]};
  }
  if (tid < P) {
    q_cum[tid] = DF{s_st.pool_hi[tid], s_st.pool_lo[tid]};
    u_key[tid] = df_key(q_cum[tid]);
    u_ord[tid] = s_st.pool_order[tid];
    q_parent[tid] = s_st.pool_parent[tid];
    q_token[tid] = s_st.pool_token[tid];
    q_depth[tid] = s_st.pool_depth[tid];
  }
  for (int sl = tid; sl < E * K; sl += blockDim.x) {
    u_key[P + sl] = 0;
    u_ord[P + sl] = kXNoOrder;
  }
  dep_wait();
  dep_launch();
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
  __syncthreads();

  // children of each expanded row (warp j % NW): the row's log-sum-exp from
  // its chunks, and its top-K by K rounds over the heads of the chunks'
  // sorted lists (staged in shared memory as entry keys)
  constexpr int RE = kXRowEntries / 32;
  __shared__ uint64_t w_k[NW][kXRowEntries];
  const int vc = p.vchunks, nE = vc * K;
  for (int j = warp; j < E; j += NW) {
    if (s_exp_depth[j] >= p.max_depth) continue;   // at the depth limit: no children
    const int64_t row = (int64_t)b * p.R + j;
    const float* rv = p.pv + row * nE;
    const int32_t* ri = p.pi + row * nE;
    // every load of the row in one round: the lists, then the chunks'
    // maxima and sums (chunks lane and lane + 32)
    float lv[RE];
    int li[RE];
#pragma unroll
    for (int q = 0; q < RE; ++q) {
      const int t = lane + 32 * q;
      lv[q] = t < nE ? __ldcg(rv + t) : -INFINITY;
      li[q] = t < nE ? __ldcg(ri + t) : -1;
    }
    const float mc0 = lane < vc ? __ldcg(p.pm + row * vc + lane) : -INFINITY;
    const float mc1 = lane + 32 < vc ? __ldcg(p.pm + row * vc + lane + 32) : -INFINITY;
    const float2 sc0 = lane < vc ? __ldcg(p.ps + row * vc + lane) : make_float2(0.f, 0.f);
    const float2 sc1 = lane + 32 < vc ? __ldcg(p.ps + row * vc + lane + 32) : make_float2(0.f, 0.f);
#pragma unroll
    for (int q = 0; q < RE; ++q) {
      const int t = lane + 32 * q;
      if (t < nE) w_k[warp][t] = li[q] < 0 ? 0ull : ent_key(lv[q], li[q]);
    }
    if (__any_sync(0xffffffffu, mc0 == INFINITY || mc1 == INFINITY)) {
      if (lane == 0) set_status(p.status, TV_DEV_BAD_LOGITS);
      continue;
    }
    float M = fmaxf(mc0, mc1);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
    DF S{0.f, 0.f};
    if (mc0 > -INFINITY) S = df_add(S, df_mulf(DF{sc0.x, sc0.y}, exp2f((mc0 - M) * kLog2e)));
    if (mc1 > -INFINITY) S = df_add(S, df_mulf(DF{sc1.x, sc1.y}, exp2f((mc1 - M) * kLog2e)));
#pragma unroll
    for (int off = 16; off > 0; off >>= 1)
      S = df_add(S, DF{__shfl_xor_sync(0xffffffffu, S.hi, off), __shfl_xor_sync(0xffffffffu, S.lo, off)});
    // S >= 1: the chunk holding M contributes at least exp(0)
    const bool all_ninf = !(M > -INFINITY);
    const DF lse = all_ninf ? DF{-INFINITY, 0.f} : df_add(DF{M, 0.f}, df_log_ge1(S));
    __syncwarp();
    // lane l walks the lists of chunks l and l + 32 (head h, next entry n,
    // loaded a round ahead); lane r keeps the r-th winner
    const bool has0 = lane < vc, has1 = lane + 32 < vc;
    const uint64_t* L0 = &w_k[warp][has0 ? lane * K : 0];
    const uint64_t* L1 = &w_k[warp][has1 ? (lane + 32) * K : 0];
    uint64_t h0 = has0 ? L0[0] : 0ull, n0 = has0 && K > 1 ? L0[1] : 0ull;
    uint64_t h1 = has1 ? L1[0] : 0ull, n1 = has1 && K > 1 ? L1[1] : 0ull;
    int q0 = 1, q1 = 1;                            // index of the next entry
    int nvalid = 0;
    uint64_t won = 0ull;
    for (int r = 0; r < K; ++r) {
      const uint64_t w = warp_max_key(h0 > h1 ? h0 : h1);
      if (w == 0ull) break;                        // warp-uniform: the row has no more valid entries
      won = lane == r ? w : won;
      nvalid = r + 1;
      // the lane holding w advances that list (selects, no branch; the
      // loads read a clamped, always valid slot)
      const bool a0 = h0 == w, a1 = !a0 && h1 == w;
      q0 += a0;
      q1 += a1;
      const uint64_t f0 = L0[q0 < K ? q0 : K - 1], f1 = L1[q1 < K ? q1 : K - 1];
      h0 = a0 ? n0 : h0;
      h1 = a1 ? n1 : h1;
      n0 = a0 ? (q0 < K ? f0 : 0ull) : n0;
      n1 = a1 ? (q1 < K ? f1 : 0ull) : n1;
    }
    // the children, one per lane: cumulative log-probability = parent's +
    // (logit - lse); -inf when the row (or the logit, or the parent) has
    // probability 0
    if (lane < nvalid) {
      const Ent e = key_ent(won);
      const int sl = j * K + lane;
      DF cv;
      if (all_ninf || e.v == -INFINITY || s_exp_cum[j].hi == -INFINITY) cv = DF{-INFINITY, 0.f};
      else cv = df_add(s_exp_cum[j], df_add(DF{e.v, 0.f}, df_neg(lse)));
      c_cum[sl] = cv;
      u_key[P + sl] = df_key(cv);
      c_token[sl] = p.token_map ? p.token_map[e.i] : e.i;
      c_parent[sl] = s_exp_node[j];
      c_depth[sl] = s_exp_depth[j] + 1;
      u_ord[P + sl] = s_gen + sl;
    }
    if (lane == 0) s_count[j] = nvalid;
    __syncwarp();
  }
  __syncthreads();

  // rank every pending and new candidate in the union; the first `pops`
  // enter the tree, the next up to N - size - pops stay pending
  int total = P;
  for (int j = 0; j < E; ++j) total += s_count[j];
  const int keep = p.N - s_n;
  int pops = p.W < keep ? p.W : keep;
  if (pops > total) pops = total;
  __shared__ DF n_cum[kXN];
  __shared__ int n_parent[kXN], n_token[kXN], n_depth[kXN], n_order[kXN];
  // rank of slot u = the valid slots that precede it, counted by S threads
  // of one warp that scan every S-th slot (all threads of a warp read the
  // same or neighbouring slots: broadcasts, no dependent load chains)
  const int nslot = P + E * K;
  int S = 1;
  while (S < 32 && 2 * S * nslot <= kXThreads) S <<= 1;
  const int per = kXThreads / S, sub = tid & (S - 1);
  for (int base = 0; base < nslot; base += per) {   // uniform trip count: the shuffles below see whole warps
    const int u = base + tid / S;
    const bool live = u < nslot;
    const uint64_t kk = live ? u_key[u] : 0;
    const int o = live ? u_ord[u] : kXNoOrder;
    int rank = 0;
    if (o != kXNoOrder)
      for (int v = sub; v < nslot; v += S) rank += cand_before(u_key[v], u_ord[v], kk, o);
    for (int off = 1; off < S; off <<= 1) rank += __shfl_xor_sync(0xffffffffu, rank, off);
    if (o == kXNoOrder || sub != 0) continue;
    DF c;
    int pa, tk, dp;
    if (u < P) {
      c = q_cum[u];
      pa = q_parent[u];
      tk = q_token[u];
      dp = q_depth[u];
    } else {
      c = c_cum[u - P];
      pa = c_parent[u - P];
      tk = c_token[u - P];
      dp = c_depth[u - P];
    }
    if (rank < pops) {
      const int i = s_n + rank;
      tok[i] = tk;
      par[i] = pa;
      dep[i] = dp;
      cum[i] = (double)c.hi + (double)c.lo;
      st->node_hi[i] = c.hi;
      st->node_lo[i] = c.lo;
      st->node_depth[i] = dp;
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
    st->pool_hi[tid] = n_cum[tid].hi;
    st->pool_lo[tid] = n_cum[tid].lo;
    st->pool_parent[tid] = n_parent[tid];
    st->pool_token[tid] = n_token[tid];
    st->pool_depth[tid] = n_depth[tid];
    st->pool_order[tid] = n_order[tid];
  }
  if (tid < pops) st->exp_node[tid] = s_n + tid;
  if (tid == 0) {
    const int n = s_n + pops;
    const int done = n >= p.N || pops == 0;
    if (p.step == 0) {
      st->node_hi[0] = 0.f;
      st->node_lo[0] = 0.f;
      st->node_depth[0] = 0;
    }
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

// Vocabulary chunks per row: one tile (8192 entries) per CTA, so each
// thread issues all its loads at once and keeps them in registers for both
// passes; at most min(64, kXRowEntries / K) chunks (the step stages the
// row's lists in shared memory and each lane walks two of them), larger
// chunks looping over tiles beyond that.  The row
// is spread evenly over its chunks (lengths a multiple of 8: 16-byte loads
// stay aligned), so every warp of a CTA holds entries.
void x_chunks(int K, int V, int tile_elems, int* vchunks, int* vlen) {
  int64_t want = ((int64_t)V + tile_elems - 1) / tile_elems;
  if (want > kXRowEntries / K) want = kXRowEntries / K;
  if (want > 64) want = 64;                    // the step's lanes walk two lists each
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
  auto take = [&](int64_t bytes) {
    const int64_t at = off;
    off = align_up(off + bytes, 256);
    return at;
  };
  l.state = take((int64_t)d->batch * (int64_t)sizeof(XState));
  l.pv = take(rows * kXRowEntries * 4);
  l.pi = take(rows * kXRowEntries * 4);
  l.pm = take(rows * kXRowEntries * 4);
  l.ps = take(rows * kXRowEntries * 8);
  l.total = off;
  return l;
}

struct TopkArgs {
  const void* logits;
  int64_t stride;
  int V, R, vlen, vc, K, vec;
  float* pv;
  int32_t* pi;
  float* pm;
  float2* ps;
};

template <bool BF16, int KT, int PT>
cudaError_t launch_topk_kt(dim3 grid, cudaStream_t s, const TopkArgs& a) {
  return launch_dep(draft_topk_kernel<BF16, KT, PT>, grid, dim3(kXTopkThreads), 0, s, a.logits, a.stride, a.V, a.R,
                    a.vlen, a.vc, a.K, a.vec, a.pv, a.pi, a.pm, a.ps);
}

template <bool BF16, int PT>
cudaError_t launch_topk_pt(int KT, dim3 grid, cudaStream_t s, const TopkArgs& a) {
  switch (KT) {
    case 1: return launch_topk_kt<BF16, 1, PT>(grid, s, a);
    case 2: return launch_topk_kt<BF16, 2, PT>(grid, s, a);
    case 4: return launch_topk_kt<BF16, 4, PT>(grid, s, a);
    case 8: return launch_topk_kt<BF16, 8, PT>(grid, s, a);
    default: return launch_topk_kt<BF16, 16, PT>(grid, s, a);
  }
}

template <bool BF16>
cudaError_t launch_topk(int KT, int PT, dim3 grid, cudaStream_t s, const TopkArgs& a) {
  return PT == 32 ? launch_topk_pt<BF16, 32>(KT, grid, s, a) : launch_topk_pt<BF16, 16>(KT, grid, s, a);
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
  const int64_t rows = (int64_t)desc->batch * R;
  TopkArgs ta = {};
  ta.logits = d_logits;
  ta.stride = seq_stride;
  ta.V = V;
  ta.R = R;
  // 16 entries per thread, or 32 when 16 would take more than two waves of
  // CTAs (two resident per SM)
  int PT = 16;
  x_chunks(desc->top_k, V, kXTopkThreads * 16, &ta.vc, &ta.vlen);
  if (rows * ta.vc > 4 * (int64_t)num_sms()) {
    PT = 32;
    x_chunks(desc->top_k, V, kXTopkThreads * 32, &ta.vc, &ta.vlen);
  }
  ta.K = desc->top_k;
  // 16-byte loads when rows stay aligned and every thread gets a vector of
  // the first tile (else one entry per thread and step, which spreads short
  // chunks over all warps)
  ta.vec = ((int64_t)V * ES) % 16 == 0 && (seq_stride * ES) % 16 == 0 && ta.vlen >= kXTopkThreads * (16 / ES);
  ta.pv = reinterpret_cast<float*>(ws + l.pv);
  ta.pi = reinterpret_cast<int32_t*>(ws + l.pi);
  ta.pm = reinterpret_cast<float*>(ws + l.pm);
  ta.ps = reinterpret_cast<float2*>(ws + l.ps);
  const int K = desc->top_k;
  const int KT = K <= 1 ? 1 : K <= 2 ? 2 : K <= 4 ? 4 : K <= 8 ? 8 : 16;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const dim3 grid(ta.vc, (unsigned)rows);
  cudaError_t e = desc->logits_dtype == TV_BF16 ? launch_topk<true>(KT, PT, grid, s, ta)
                                                : launch_topk<false>(KT, PT, grid, s, ta);
  if (e != cudaSuccess) return TV_ERR_CUDA;
  XParams xp;
  xp.pv = ta.pv;
  xp.pi = ta.pi;
  xp.pm = ta.pm;
  xp.ps = ta.ps;
  xp.vchunks = ta.vc;
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
  xp.K = K;
  xp.W = desc->width;
  xp.N = desc->max_nodes;
  xp.max_depth = desc->max_depth;
  e = launch_dep(expand_step_kernel, dim3(desc->batch), dim3(kXThreads), 0, s, xp);
  return e == cudaSuccess ? TV_OK : TV_ERR_CUDA;
}

}  // extern "C"
