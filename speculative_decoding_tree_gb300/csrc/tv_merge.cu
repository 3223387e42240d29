// Log-sum-exp merge of the split-KV partials ("ADR-037 — EAGLE-3 with dynamic
// tree port", phase row E1.3: the reduce kernel of the split pass).
//
// For every query row (node, head) with splits s = 0 .. nch-1 holding a
// normalised output Y_s = O_s / l_s, a running maximum m_s (log2 units) and
// a sum l_s:
//   M = max_s m_s,  c_s = 2^(m_s - M) l_s,  out = sum_s c_s Y_s / sum_s c_s.
// Y_s is fp32, or bf16 when the output is bf16 (tensor-core kernels).
//
// The partials sit at partial_slot(): the splits of a row are adjacent and
// the rows of a row tile follow each other, so the partials of a slab of
// slab_rows rows of one (sequence b, KV head g, row tile rt) are one
// contiguous block.  One CTA takes one slab: right after the dependency wait
// it starts a single bulk copy of the block into shared memory (one per row
// when the splits come in several batches), reads the (m, l) pairs and the
// sequence's lengths with plain loads meanwhile, reduces in shared memory and
// writes the output rows.  More splits than fit in shared memory are taken in
// batches with a running maximum.
#include "tc_ptx.cuh"
#include "tv_internal.cuh"

namespace tv {
namespace {

using namespace tc;

constexpr int kMergeThreads = 256;
// most rows one merge CTA takes: 32 at head_dim 128 (a batch's many small
// tiles: fewer CTAs), 16 otherwise
__host__ __device__ constexpr int max_slab_rows(int d) { return d <= 128 ? 32 : 16; }
constexpr uint64_t kMergeWaitNs = 1000000000ull;

__device__ __forceinline__ float4 load4(const float* row, int c) {
  return reinterpret_cast<const float4*>(row)[c];
}
__device__ __forceinline__ float4 load4(const __nv_bfloat16* row, int c) {
  const uint2 u = reinterpret_cast<const uint2*>(row)[c];
  const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u.x));
  const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u.y));
  return make_float4(a.x, a.y, b.x, b.y);
}

template <int D, typename PT>
__global__ __launch_bounds__(kMergeThreads) void merge_slab_kernel(MergeParams p) {
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  __shared__ float s_m[max_slab_rows(D)], s_l[max_slab_rows(D)], s_keep[max_slab_rows(D)];
  const int tid = threadIdx.x;
  const int RS = p.slab_rows, SB = p.batch_splits, S = p.splits;
  PT* so = reinterpret_cast<PT*>(smem);                                              // [RS][SB][D]
  float2* sml = reinterpret_cast<float2*>(smem + (size_t)RS * SB * D * sizeof(PT));  // [RS][SB]
  float* s_w = reinterpret_cast<float*>(sml + (size_t)RS * SB);                      // [RS][SB]
  if (tid == 0) {
    mbar_init(smem_u32(&bar), 1);
    abort_flag = 0;
    fence_barrier_init();
  }
  __syncthreads();

  const int b = blockIdx.z;
  const int g = blockIdx.y / p.row_tiles, rt = blockIdx.y % p.row_tiles;
  const int r0 = blockIdx.x * RS;                   // first row of the slab inside the tile
  // Launched right after the split pass of the same call (early_reads), the
  // sequence's lengths are read before the dependency wait: the split pass
  // does not write them and waited for its own predecessor before letting
  // this kernel start.  Only the partials wait for it.
  if (!p.early_reads) dep_wait();
  const int64_t Praw = p.prefix_len[b];
  int o0 = 0, n = 1;
  const bool valid = seq_rows(p.node_offsets, b, p.R, p.max_nodes, nullptr, &o0, &n);
  const int nrows = n * p.G;
  const int m_first = rt * p.rows_per_tile + r0;
  const int64_t P = clamp_prefix(Praw, p.max_prefix, p.capacity);
  const int nch = num_chunks(P, p.chunk, p.tree_tile);
  // rows this CTA writes (none: empty slab, or the split pass wrote them)
  const bool live = valid && r0 < p.rows_per_tile && m_first < nrows && !(p.skip_single && nch == 1);
  const int rows = live ? min(RS, min(p.rows_per_tile - r0, nrows - m_first)) : 0;
  dep_wait();
  dep_launch();
  if (!valid && tid == 0) set_status(p.status, TV_DEV_BAD_OFFSETS);
  if (!live) return;

  const int crow = min(RS, p.tile_stride - r0);     // rows gathered (inside the tile)
  const int64_t slot0 = partial_slot(0, b, g, rt, r0, p.Hkv, p.row_tiles, p.tile_stride, S);
  const PT* src = reinterpret_cast<const PT*>(p.o_part);
  const uint32_t bar_a = smem_u32(&bar);
  // batch of splits [s0, s0 + nb) of the slab's rows into shared memory: one
  // copy when the batch holds every split (the slab is contiguous), else one
  // per row
  auto gather = [&](int s0, int nb) {
    if (tid == 0) {
      mbar_expect_tx(bar_a, (uint32_t)(crow * nb * D * sizeof(PT)));
      if (nb == S)
        bulk_load(smem_u32(so), src + slot0 * D, (uint32_t)(crow * S * D * sizeof(PT)), bar_a);
      else
        for (int r = 0; r < crow; ++r)
          bulk_load(smem_u32(so + (size_t)r * SB * D), src + (slot0 + (int64_t)r * S + s0) * D,
                    (uint32_t)(nb * D * sizeof(PT)), bar_a);
    }
  };
  gather(0, min(SB, S));

  constexpr int C4 = D / 4;                         // float4 columns per row
  const int items = rows * C4;
  constexpr int kMaxItems = max_slab_rows(D) * C4 / kMergeThreads + 1;
  float4 acc[kMaxItems];
#pragma unroll
  for (int k = 0; k < kMaxItems; ++k) acc[k] = make_float4(0.f, 0.f, 0.f, 0.f);
  if (tid < rows) {
    s_m[tid] = -INFINITY;
    s_l[tid] = 0.f;
  }
  bool ok = true;
  int phase = 0;
  for (int s0 = 0; s0 < nch && ok; s0 += SB, ++phase) {
    const int nb = min(SB, nch - s0);
    if (s0 > 0) gather(s0, min(SB, S - s0));
    for (int e = tid; e < rows * nb; e += kMergeThreads) {   // (m, l) of the batch, plain loads
      const int r = e / nb, j = e % nb;
      sml[r * SB + j] = p.ml_part[slot0 + (int64_t)r * S + s0 + j];
    }
    ok = __syncthreads_and(mbar_wait(bar_a, phase & 1, &abort_flag, kMergeWaitNs));
    if (!ok) break;
    // per row (one warp per row, lanes over the splits): M' = max(M, m_s);
    // earlier sums and outputs scale by 2^(M - M'); split s weighs
    // 2^(m_s - M') l_s (0 for a split whose keys were all masked)
    for (int r = tid >> 5; r < rows; r += kMergeThreads / 32) {
      const int lane = tid & 31;
      const float M = s_m[r];
      float Mn = M;
      for (int j = lane; j < nb; j += 32) Mn = fmaxf(Mn, sml[r * SB + j].x);
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) Mn = fmaxf(Mn, __shfl_xor_sync(0xffffffffu, Mn, off));
      float part = 0.f;
      for (int j = lane; j < nb; j += 32) {
        const float2 ml = sml[r * SB + j];
        const float w = (ml.x == -INFINITY) ? 0.f : exp2f(ml.x - Mn) * ml.y;
        s_w[r * SB + j] = w;
        part += w;
      }
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) part += __shfl_xor_sync(0xffffffffu, part, off);
      if (lane == 0) {
        const float keep = (M == -INFINITY) ? 0.f : exp2f(M - Mn);
        s_m[r] = Mn;
        s_l[r] = s_l[r] * keep + part;
        s_keep[r] = keep;
      }
    }
    __syncthreads();
#pragma unroll
    for (int k = 0; k < kMaxItems; ++k) {
      const int it = tid + k * kMergeThreads;
      if (it >= items) break;
      const int r = it / C4, c = it % C4;
      const float keep = s_keep[r];
      float4 a = make_float4(acc[k].x * keep, acc[k].y * keep, acc[k].z * keep, acc[k].w * keep);
#pragma unroll 4
      for (int j = 0; j < nb; ++j) {
        const float w = s_w[r * SB + j];
        const float4 v = load4(so + ((size_t)r * SB + j) * D, c);
        a.x = fmaf(w, v.x, a.x);
        a.y = fmaf(w, v.y, a.y);
        a.z = fmaf(w, v.z, a.z);
        a.w = fmaf(w, v.w, a.w);
      }
      acc[k] = a;
    }
    __syncthreads();                                // the next batch overwrites the buffers
  }
  if (!ok) {
    // a copy that never landed: flag it, and give the copies in flight a
    // bounded time to finish before the CTA (and its shared memory) ends
    if (tid == 0) set_status(p.status, TV_DEV_TIMEOUT);
    int spare = 0;
    mbar_wait(bar_a, phase & 1, &spare, kMergeWaitNs);
    return;
  }
#pragma unroll
  for (int k = 0; k < kMaxItems; ++k) {
    const int it = tid + k * kMergeThreads;
    if (it >= items) break;
    const int r = it / C4, c = it % C4;
    const int m = m_first + r;                      // query row of the KV head: node m / G, head g G + m % G
    const int64_t e = ((int64_t)(o0 + m / p.G) * p.Hq + g * p.G + m % p.G) * D + c * 4;
    const float L = s_l[r];
    const float inv = L > 0.f ? 1.f / L : 0.f;
    const float4 v = make_float4(acc[k].x * inv, acc[k].y * inv, acc[k].z * inv, acc[k].w * inv);
    if (p.out_bf16) {
      __nv_bfloat162 lo = __floats2bfloat162_rn(v.x, v.y), hi = __floats2bfloat162_rn(v.z, v.w);
      uint2 u;
      u.x = *reinterpret_cast<uint32_t*>(&lo);
      u.y = *reinterpret_cast<uint32_t*>(&hi);
      *reinterpret_cast<uint2*>(reinterpret_cast<__nv_bfloat16*>(p.out) + e) = u;
    } else {
      *reinterpret_cast<float4*>(reinterpret_cast<float*>(p.out) + e) = v;
    }
  }
}

template <int D, typename PT>
cudaError_t launch_merge_t(const MergeParams& p, cudaStream_t s) {
  const size_t smem = (size_t)p.batch_splits * p.slab_rows * (D * sizeof(PT) + 8 + 4);
  cudaError_t e = ensure_max_dynamic_smem<merge_slab_kernel<D, PT>>((int)smem);
  if (e != cudaSuccess) return e;
  dim3 grid((p.tile_stride + p.slab_rows - 1) / p.slab_rows, p.Hkv * p.row_tiles, p.B);
  return launch_dep(merge_slab_kernel<D, PT>, grid, dim3(kMergeThreads), smem, s, p);
}

}  // namespace

cudaError_t launch_merge(const MergeParams& p, cudaStream_t s) {
  if (p.part_bf16) {
    if (p.d == 128) return launch_merge_t<128, __nv_bfloat16>(p, s);
    if (p.d == 256) return launch_merge_t<256, __nv_bfloat16>(p, s);
    return launch_merge_t<512, __nv_bfloat16>(p, s);
  }
  if (p.d == 128) return launch_merge_t<128, float>(p, s);
  if (p.d == 256) return launch_merge_t<256, float>(p, s);
  return launch_merge_t<512, float>(p, s);
}

void merge_shape(int tiles, int tile_stride, int d, int esize, int splits, int sms, int* slab_rows,
                 int* batch_splits) {
  // the largest slab (32 rows at head_dim 128, else 16; then 8, 4, 2) that
  // still gives every SM a CTA,
  // then as many splits per batch as about 100 KB of shared memory holds
  int rs = max_slab_rows(d);
  while (rs > 2 && (rs > tile_stride || (int64_t)tiles * ((tile_stride + rs - 1) / rs) < sms)) rs >>= 1;
  const int per_split = rs * (d * esize + 8 + 4);
  int sb = (100 * 1024) / per_split;
  if (sb < 1) sb = 1;
  if (sb > splits) sb = splits;
  *slab_rows = rs;
  *batch_splits = sb;
}

}  // namespace tv
