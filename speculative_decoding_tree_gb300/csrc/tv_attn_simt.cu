// CUDA-core split-KV tree-verify attention (fp32 inputs, and bf16 where the
// query rows per KV head are too few for a tensor-core tile or head_dim is
// 512), plus the log-sum-exp merge kernel shared with the tensor-core path.
//
// The method is flash-decode with a tree mask ("ADR-037 — EAGLE-3 with
// dynamic tree port", phase rows E1.1-E1.5 and E4b.6): each split walks a
// range of keys with an online softmax (running maximum m, running sum l,
// unnormalised output O) and the merge combines the splits:
//   M = max_s m_s,  L = sum_s l_s 2^(m_s - M),  O = sum_s O_s 2^(m_s - M) / L.
// Scores are kept in base-2 units (score * scale * log2 e) so exp2 applies.
//
// Work split: CTA (row tile, KV head g, split s, sequence b).  Four warps;
// warp w owns RPW query rows (row m = node * G + group head).  Keys stream
// through shared memory 32 at a time; for QK each lane owns one key, for PV
// each lane owns d/32 output columns of every row.
#include <cfloat>

#include "tv_internal.cuh"

namespace tv {
namespace {

constexpr int kKeyTile = 32;

template <typename T>
__device__ __forceinline__ void load8(const T* src, float* dst);

template <>
__device__ __forceinline__ void load8<float>(const float* src, float* dst) {
  const float4* s = reinterpret_cast<const float4*>(src);
  float4 a = s[0], b = s[1];
  dst[0] = a.x; dst[1] = a.y; dst[2] = a.z; dst[3] = a.w;
  dst[4] = b.x; dst[5] = b.y; dst[6] = b.z; dst[7] = b.w;
}

template <>
__device__ __forceinline__ void load8<__nv_bfloat16>(const __nv_bfloat16* src, float* dst) {
  uint4 u = *reinterpret_cast<const uint4*>(src);
  const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
  for (int t = 0; t < 4; ++t) {
    float2 f = __bfloat1622float2(h[t]);
    dst[2 * t] = f.x;
    dst[2 * t + 1] = f.y;
  }
}

template <typename T, int D>
__global__ __launch_bounds__(128) void attn_simt_kernel(AttnParams p) {
  constexpr int RPW = 1024 / D;          // rows per warp
  constexpr int ROWS = 4 * RPW;          // rows per CTA
  constexpr int KS = D + 4;              // padded K row (conflict-free float4 reads by key)
  constexpr int CPL = D / 128;           // float4 output chunks per lane
  extern __shared__ float4 smem_f4[];
  float* qs = reinterpret_cast<float*>(smem_f4);          // [ROWS][D]
  float* ks = qs + ROWS * D;                              // [32][KS]
  float* vs = ks + kKeyTile * KS;                         // [32][D]
  float* ps = vs + kKeyTile * D;                          // [4 warps][RPW][32]
  __shared__ uint64_t s_anc[ROWS];
  dep_wait();
  dep_launch();

  const int b = blockIdx.z;
  const int s = blockIdx.y;
  const int g = blockIdx.x / p.row_tiles;
  const int rt = blockIdx.x % p.row_tiles;
  int o0, n;
  if (!seq_rows(p.node_offsets, b, p.R, p.max_nodes, p.status, &o0, &n)) return;
  const int nrows = n * p.G;
  const int m0 = rt * ROWS;
  if (m0 >= nrows) return;
  const int64_t Praw = p.prefix_len[b];
  const int64_t P = clamp_prefix(Praw, p.max_prefix, p.capacity);
  if (P != Praw && threadIdx.x == 0 && rt == 0 && s == 0 && g == 0) set_status(p.status, TV_DEV_BAD_PREFIX);
  const int nch = num_chunks(P, p.chunk, p.tree_tile);
  if (s >= nch) return;
  const int64_t k_begin = (int64_t)s * p.chunk;
  const int64_t k_end = min(P, k_begin + p.chunk);
  const bool has_tree = (s == nch - 1);

  const T* q = reinterpret_cast<const T*>(p.q);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  // stage the CTA's query rows (fp32) and their ancestor masks
  for (int e = tid; e < ROWS * (D / 8); e += blockDim.x) {
    const int r = e / (D / 8), c8 = e % (D / 8);
    const int m = m0 + r;
    float tmp[8];
    if (m < nrows) {
      const int i = m / p.G, hh = m % p.G;
      load8<T>(q + (((int64_t)(o0 + i) * p.Hq + g * p.G + hh) * D + c8 * 8), tmp);
    } else {
#pragma unroll
      for (int t = 0; t < 8; ++t) tmp[t] = 0.f;
    }
    float4* dst = reinterpret_cast<float4*>(qs + r * D + c8 * 8);
    dst[0] = make_float4(tmp[0], tmp[1], tmp[2], tmp[3]);
    dst[1] = make_float4(tmp[4], tmp[5], tmp[6], tmp[7]);
  }
  for (int r = tid; r < ROWS; r += blockDim.x) {
    const int m = m0 + r;
    s_anc[r] = m < nrows ? p.anc[o0 + m / p.G] : 0ull;
  }

  float m_run[RPW], l_run[RPW];
  float4 acc[RPW][CPL];
#pragma unroll
  for (int r = 0; r < RPW; ++r) {
    m_run[r] = -INFINITY;
    l_run[r] = 0.f;
#pragma unroll
    for (int c = 0; c < CPL; ++c) acc[r][c] = make_float4(0.f, 0.f, 0.f, 0.f);
  }

  const T* kc = reinterpret_cast<const T*>(p.k_cache);
  const T* vc = reinterpret_cast<const T*>(p.v_cache);
  const T* kt = reinterpret_cast<const T*>(p.k_tree);
  const T* vt = reinterpret_cast<const T*>(p.v_tree);
  const int64_t n_prefix_tiles = (k_end - k_begin + kKeyTile - 1) / kKeyTile;
  const int n_tree_tiles = has_tree ? (n + kKeyTile - 1) / kKeyTile : 0;

  for (int64_t tile = 0; tile < n_prefix_tiles + n_tree_tiles; ++tile) {
    const bool tree_tile = tile >= n_prefix_tiles;
    const int64_t t0 = tree_tile ? (tile - n_prefix_tiles) * kKeyTile : k_begin + tile * kKeyTile;
    const int64_t t1 = tree_tile ? (int64_t)n : k_end;
    __syncthreads();   // previous tile fully consumed (and query rows staged)
    // cooperative load of 32 keys x D of K and V, converted to fp32
    for (int e = tid; e < kKeyTile * (D / 8); e += blockDim.x) {
      const int j = e / (D / 8), c8 = e % (D / 8);
      const int64_t pos = t0 + j;
      float tk[8], tv[8];
      const T* ksrc = nullptr;
      const T* vsrc = nullptr;
      if (pos < t1) {
        if (tree_tile) {
          const int64_t row = (int64_t)g * p.R + o0 + pos;
          ksrc = kt + row * D;
          vsrc = vt + row * D;
        } else if (p.paged) {
          const int pid = p.page_table[(int64_t)b * p.max_pages + pos / kPageSize];
          if (pid >= 0 && pid < p.num_pages) {
            const int64_t row = ((int64_t)pid * p.Hkv + g) * kPageSize + pos % kPageSize;
            ksrc = kc + row * D;
            vsrc = vc + row * D;
          } else if (c8 == 0) {
            set_status(p.status, TV_DEV_BAD_PAGE);
          }
        } else {
          const int64_t row = ((int64_t)b * p.Hkv + g) * p.capacity + pos;
          ksrc = kc + row * D;
          vsrc = vc + row * D;
        }
      }
      if (ksrc) {
        load8<T>(ksrc + c8 * 8, tk);
        load8<T>(vsrc + c8 * 8, tv);
      } else {
#pragma unroll
        for (int t = 0; t < 8; ++t) tk[t] = tv[t] = 0.f;
      }
      float4* kd = reinterpret_cast<float4*>(ks + j * KS + c8 * 8);
      kd[0] = make_float4(tk[0], tk[1], tk[2], tk[3]);
      kd[1] = make_float4(tk[4], tk[5], tk[6], tk[7]);
      float4* vd = reinterpret_cast<float4*>(vs + j * D + c8 * 8);
      vd[0] = make_float4(tv[0], tv[1], tv[2], tv[3]);
      vd[1] = make_float4(tv[4], tv[5], tv[6], tv[7]);
    }
    __syncthreads();

    // scores: lane = key
    float sc[RPW];
#pragma unroll
    for (int r = 0; r < RPW; ++r) sc[r] = 0.f;
    const float4* krow = reinterpret_cast<const float4*>(ks + lane * KS);
#pragma unroll 4
    for (int c = 0; c < D / 4; ++c) {
      const float4 kv = krow[c];
#pragma unroll
      for (int r = 0; r < RPW; ++r) {
        const float4 qv = reinterpret_cast<const float4*>(qs + (warp * RPW + r) * D)[c];
        sc[r] = fmaf(qv.x, kv.x, sc[r]);
        sc[r] = fmaf(qv.y, kv.y, sc[r]);
        sc[r] = fmaf(qv.z, kv.z, sc[r]);
        sc[r] = fmaf(qv.w, kv.w, sc[r]);
      }
    }
    const int64_t pos = t0 + lane;
    const bool in_range = pos < t1;
    float* pw = ps + warp * RPW * kKeyTile;
#pragma unroll
    for (int r = 0; r < RPW; ++r) {
      bool vis = in_range;
      if (tree_tile) vis = vis && ((s_anc[warp * RPW + r] >> pos) & 1ull);
      float x = vis ? sc[r] * p.scale_log2 : -INFINITY;
      float mx = x;
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
      const float m_new = fmaxf(m_run[r], mx);
      float pr = 0.f, alpha = 1.f;
      if (m_new != -INFINITY) {
        pr = vis ? exp2f(x - m_new) : 0.f;
        alpha = exp2f(m_run[r] - m_new);     // 0 when m_run was -inf
      }
      float sum = pr;
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, off);
      l_run[r] = l_run[r] * alpha + sum;
      m_run[r] = m_new;
#pragma unroll
      for (int c = 0; c < CPL; ++c) {
        acc[r][c].x *= alpha; acc[r][c].y *= alpha; acc[r][c].z *= alpha; acc[r][c].w *= alpha;
      }
      pw[r * kKeyTile + lane] = pr;
    }
    __syncwarp();
    // PV: lane owns columns lane*4 + 128*c
#pragma unroll 4
    for (int j = 0; j < kKeyTile; ++j) {
      float4 vv[CPL];
#pragma unroll
      for (int c = 0; c < CPL; ++c) vv[c] = reinterpret_cast<const float4*>(vs + j * D)[lane + 32 * c];
#pragma unroll
      for (int r = 0; r < RPW; ++r) {
        const float pj = pw[r * kKeyTile + j];
#pragma unroll
        for (int c = 0; c < CPL; ++c) {
          acc[r][c].x = fmaf(pj, vv[c].x, acc[r][c].x);
          acc[r][c].y = fmaf(pj, vv[c].y, acc[r][c].y);
          acc[r][c].z = fmaf(pj, vv[c].z, acc[r][c].z);
          acc[r][c].w = fmaf(pj, vv[c].w, acc[r][c].w);
        }
      }
    }
    __syncwarp();
  }

  // partial outputs of this split; a sequence with one chunk writes its
  // normalised rows directly (the merge's arithmetic for one split)
  const bool direct = p.out != nullptr && nch == 1;
#pragma unroll
  for (int r = 0; r < RPW; ++r) {
    const int m = m0 + warp * RPW + r;
    if (m >= nrows) continue;
    const int64_t rowg = o0 + m / p.G;
    const int h = g * p.G + m % p.G;
    const int64_t idx = partial_slot(s, b, g, rt, m - m0, p.Hkv, p.row_tiles, p.tile_stride, p.splits);
    if (direct) {
      const float inv = l_run[r] > 0.f ? 1.f / l_run[r] : 0.f;
      const int64_t obase = (rowg * p.Hq + h) * D;
#pragma unroll
      for (int c = 0; c < CPL; ++c) {
        const float4 v = make_float4(acc[r][c].x * inv, acc[r][c].y * inv, acc[r][c].z * inv, acc[r][c].w * inv);
        const int64_t e = obase + (lane + 32 * c) * 4;
        if (p.out_bf16) {
          __nv_bfloat162 a = __floats2bfloat162_rn(v.x, v.y), bb = __floats2bfloat162_rn(v.z, v.w);
          uint2 u;
          u.x = *reinterpret_cast<uint32_t*>(&a);
          u.y = *reinterpret_cast<uint32_t*>(&bb);
          *reinterpret_cast<uint2*>(reinterpret_cast<__nv_bfloat16*>(p.out) + e) = u;
        } else {
          *reinterpret_cast<float4*>(reinterpret_cast<float*>(p.out) + e) = v;
        }
      }
      continue;
    }
    // partial O_s / l_s (fp32) with the split's running max and sum
    const float inv = l_run[r] > 0.f ? 1.f / l_run[r] : 0.f;
    float4* dst = reinterpret_cast<float4*>(p.o_part + idx * D);
#pragma unroll
    for (int c = 0; c < CPL; ++c)
      dst[lane + 32 * c] = make_float4(acc[r][c].x * inv, acc[r][c].y * inv, acc[r][c].z * inv, acc[r][c].w * inv);
    if (lane == 0) p.ml_part[idx] = make_float2(m_run[r], l_run[r]);
  }
}

template <typename T, int D>
cudaError_t launch_simt_t(const AttnParams& p, cudaStream_t s) {
  constexpr int RPW = 1024 / D;
  constexpr int ROWS = 4 * RPW;
  const size_t smem = sizeof(float) * (ROWS * D + kKeyTile * (D + 4) + kKeyTile * D + 4 * RPW * kKeyTile);
  cudaError_t e = ensure_max_dynamic_smem<attn_simt_kernel<T, D>>((int)smem);
  if (e != cudaSuccess) return e;
  dim3 grid(p.row_tiles * p.Hkv, p.splits, p.B);
  return launch_dep(attn_simt_kernel<T, D>, grid, dim3(128), smem, s, p);
}

}  // namespace

cudaError_t launch_attn_simt(const AttnParams& p, int dtype, cudaStream_t s) {
  if (dtype == TV_F32) {
    if (p.d == 128) return launch_simt_t<float, 128>(p, s);
    if (p.d == 256) return launch_simt_t<float, 256>(p, s);
    return launch_simt_t<float, 512>(p, s);
  }
  if (p.d == 128) return launch_simt_t<__nv_bfloat16, 128>(p, s);
  if (p.d == 256) return launch_simt_t<__nv_bfloat16, 256>(p, s);
  return launch_simt_t<__nv_bfloat16, 512>(p, s);
}


}  // namespace tv
