// Fused lm_head + argmax ("ADR-037 — EAGLE-3 with dynamic tree port", phase
// rows E4b.9, E5a and E4b.10a): argmax over the vocabulary of hidden . weight
// for every tree row, without writing the logits.
//
// lmhead_argmax_kernel: persistent, one CTA per SM.  A unit is 256
// vocabulary rows of the weight against one tile of 128 hidden rows; CTA c
// takes units c, c + grid, ... (increasing vocabulary within each row tile).
// For each unit the tensor cores compute D[row, v] = sum_k H[row, k] W[v, k]
// (tcgen05.mma kind::f16, M = 128 hidden rows, N = 256 vocabulary rows,
// K = 16 per instruction, fp32 accumulators in tensor memory), fed by a
// four-stage TMA ring of 64-wide k-chunks of W and H (128-byte swizzle).
// With the hidden rows on the M side each epilogue thread owns one row (one
// TMEM lane), so the argmax over the unit's 256 vocabulary columns is a
// thread-local scan; two accumulators alternate so the scan of one unit
// overlaps the MMAs of the next.  The weight is read from HBM once; at 64
// rows a unit's arithmetic intensity is 64 flop per weight byte, far below
// the bf16 ridge, so the kernel is bound by the weight stream.
//
// lmhead_finish_kernel: one warp per row picks the first maximum over the
// CTAs' partial maxima.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cudaTypedefs.h>

#include <cmath>
#include <cstdint>
#include <mutex>

#include "tc_ptx.cuh"
#include "tree_lm_head.h"
#include "tv_internal.cuh"
#include "tv_select.cuh"

namespace tv {
namespace {

using namespace tc;

constexpr int LM = 128;                          // hidden rows per tile (MMA M)
constexpr int LV = 256;                          // vocabulary rows per unit (MMA N)
constexpr int LKC = 64;                          // k per chunk (one 128-byte swizzle row)
constexpr int LNS = 4;                           // ring stages
constexpr uint32_t W_BYTES = LV * 128;           // 32 KB
constexpr uint32_t H_BYTES = LM * 128;           // 16 KB
constexpr uint32_t STAGE_BYTES = W_BYTES + H_BYTES;
constexpr int kLThreads = 256;                   // warp 0 TMA, 1 MMA, 2 TMEM, 4-7 epilogue
constexpr int kMaxRowTiles = 16;                 // rows <= 2048
constexpr uint32_t kLHeader = 1024;              // barriers, TMEM address, abort flag
constexpr uint32_t kLSmem = kLHeader + LNS * STAGE_BYTES + kMaxRowTiles * LM * 8;
constexpr uint64_t kLWaitNs = 1000000000ull;
static_assert(kLSmem + 1024 <= 232448, "shared memory over the per-block limit");

struct LmParams {
  float* part_v;             // [grid, R] each CTA's largest logit per row
  int32_t* part_i;           // [grid, R] its vocabulary index (-1: none)
  int32_t* status;
  int R, Hd, V, RT, units, KCH;
};

__global__ void __launch_bounds__(kLThreads, 1)
lmhead_argmax_kernel(const __grid_constant__ LmParams p, const __grid_constant__ CUtensorMap tm_w,
                     const __grid_constant__ CUtensorMap tm_h) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* base = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);   // 1 KB aligned
  uint64_t* bars = reinterpret_cast<uint64_t*>(base);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(base + 256);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(base + 260);
  uint8_t* ring = base + kLHeader;
  float* best_v = reinterpret_cast<float*>(ring + LNS * STAGE_BYTES);       // [row tile][128]
  int32_t* best_i = reinterpret_cast<int32_t*>(best_v + kMaxRowTiles * LM);
  auto bar = [&](int i) { return smem_u32(&bars[i]); };
  auto FULL = [&](int i) { return bar(i); };
  auto EMPTY = [&](int i) { return bar(LNS + i); };
  auto ACC_FULL = [&](int i) { return bar(2 * LNS + i); };
  auto ACC_EMPTY = [&](int i) { return bar(2 * LNS + 2 + i); };
  const uint32_t FIN = bar(2 * LNS + 4);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  constexpr unsigned kAll = 0xffffffffu;
  if (tid == 0) {
    for (int i = 0; i < LNS; ++i) {
      mbar_init(FULL(i), 1);
      mbar_init(EMPTY(i), 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(ACC_FULL(i), 1);
      mbar_init(ACC_EMPTY(i), 4);                 // one arrive per epilogue warp
    }
    mbar_init(FIN, 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 2) {
    tmem_alloc(smem_u32(tmem_slot), 512);
    tmem_relinquish();
  }
  if (warp >= 4) {
    const int rl = tid - 128;
    for (int t = 0; t < kMaxRowTiles; ++t) {
      best_v[t * LM + rl] = -INFINITY;
      best_i[t * LM + rl] = -1;
    }
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tm_w);
    tma_prefetch_desc(&tm_h);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  dep_wait();
  dep_launch();

  if (warp == 0) {
    // ============================================================ TMA producer
    if (lane == 0) {
      int it = 0;
      bool ok = true;
      for (int u = blockIdx.x; u < p.units && ok; u += gridDim.x) {
        const int vb = u / p.RT, rt = u - vb * p.RT;
        for (int kc = 0; kc < p.KCH; ++kc, ++it) {
          const int slot = it % LNS, use = it / LNS;
          if (use > 0 && !mbar_wait(EMPTY(slot), (use - 1) & 1, abort_flag, kLWaitNs)) {
            ok = false;
            break;
          }
          uint8_t* st = ring + slot * STAGE_BYTES;
          mbar_expect_tx(FULL(slot), STAGE_BYTES);
          tma_load_2d(smem_u32(st), &tm_w, FULL(slot), kc * LKC, vb * LV);
          tma_load_2d(smem_u32(st + W_BYTES), &tm_h, FULL(slot), kc * LKC, rt * LM);
        }
      }
      // every copy started has landed before the CTA exits
      for (int j = (it > LNS ? it - LNS : 0); j < it; ++j)
        mbar_wait(FULL(j % LNS), (j / LNS) & 1, abort_flag, kLWaitNs);
    }
  } else if (warp == 1) {
    // ============================================================ MMA issuer
    if (lane == 0) {
      constexpr uint32_t IDESC = idesc_bf16_f32(LM, LV, 0, 0);
      const uint32_t ring_addr = smem_u32(ring);
      int it = 0, acc = 0;
      bool ok = true;
      for (int u = blockIdx.x; u < p.units && ok; u += gridDim.x, ++acc) {
        const int ab = acc & 1;
        if (acc >= 2 && !mbar_wait(ACC_EMPTY(ab), ((acc >> 1) - 1) & 1, abort_flag, kLWaitNs)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d = tmem + (uint32_t)(ab * LV);
        for (int kc = 0; kc < p.KCH; ++kc, ++it) {
          const int slot = it % LNS;
          if (!mbar_wait(FULL(slot), (it / LNS) & 1, abort_flag, kLWaitNs)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t w_addr = ring_addr + slot * STAGE_BYTES;
          const uint32_t h_addr = w_addr + W_BYTES;
#pragma unroll
          for (int kk = 0; kk < LKC / 16; ++kk) {
            const uint64_t a = smem_desc(h_addr + kk * 32, 16, 1024, 2);
            const uint64_t b = smem_desc(w_addr + kk * 32, 16, 1024, 2);
            mma_ss(d, a, b, IDESC, (kc > 0 || kk > 0) ? 1u : 0u);
          }
          mma_commit(EMPTY(slot));
        }
        if (!ok) break;
        mma_commit(ACC_FULL(ab));
      }
      // every MMA issued has finished before tensor memory is freed
      mma_commit(FIN);
      mbar_wait(FIN, 0, abort_flag, kLWaitNs);
    }
  } else if (warp >= 4) {
    // ============================================================ epilogue
    // thread = hidden row rl of the tile = TMEM lane; tcgen05.ld is
    // warp-collective, so control flow around it stays warp-uniform
    const int q = warp & 3, rl = q * 32 + lane;
    const uint32_t lane_base = (uint32_t)(q * 32) << 16;
    int acc = 0;
    for (int u = blockIdx.x; u < p.units; u += gridDim.x, ++acc) {
      const int vb = u / p.RT, rt = u - vb * p.RT, ab = acc & 1;
      if (!__all_sync(kAll, mbar_wait(ACC_FULL(ab), (acc >> 1) & 1, abort_flag, kLWaitNs))) break;
      tc_fence_after();
      float bv = best_v[rt * LM + rl];
      int bi = best_i[rt * LM + rl];
      const int v0 = vb * LV;
#pragma unroll 1
      for (int c = 0; c < LV / 64; ++c) {
        uint32_t rr[64];
        tmem_ld_x64(tmem + lane_base + (uint32_t)(ab * LV + c * 64), rr);
#pragma unroll
        for (int e = 0; e < 64; ++e) {
          const float x = __uint_as_float(rr[e]);
          const int v = v0 + c * 64 + e;
          // columns in increasing order: a strictly larger value replaces the
          // best, so the first index of the maximum stays; NaN never wins
          if (v < p.V && x == x && (bi < 0 || x > bv)) {
            bv = x;
            bi = v;
          }
        }
      }
      best_v[rt * LM + rl] = bv;
      best_i[rt * LM + rl] = bi;
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(ACC_EMPTY(ab));
    }
    for (int rt = 0; rt < p.RT; ++rt) {
      const int r = rt * LM + rl;
      if (r < p.R) {
        p.part_v[(int64_t)blockIdx.x * p.R + r] = best_v[rt * LM + rl];
        p.part_i[(int64_t)blockIdx.x * p.R + r] = best_i[rt * LM + rl];
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (tid == 0 && *abort_flag) set_status(p.status, TV_DEV_TIMEOUT);
  if (warp == 2) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// grid (ceil(R / 8)), 256 threads: warp w of CTA b takes row 8b + w.
__global__ void __launch_bounds__(256) lmhead_finish_kernel(const float* __restrict__ part_v,
                                                            const int32_t* __restrict__ part_i, int nparts, int R,
                                                            int32_t* __restrict__ argmax,
                                                            float* __restrict__ max_logit) {
  dep_wait();
  dep_launch();
  const int r = blockIdx.x * 8 + (threadIdx.x >> 5), lane = threadIdx.x & 31;
  if (r >= R) return;
  Ent best{-INFINITY, -1};
  for (int c = lane; c < nparts; c += 32) {
    const Ent e{part_v[(int64_t)c * R + r], part_i[(int64_t)c * R + r]};
    if (ent_before(e, best)) best = e;
  }
  best = warp_first(best);
  if (lane == 0) {
    argmax[r] = best.i < 0 ? 0 : best.i;
    if (max_logit) max_logit[r] = best.i < 0 ? __int_as_float(0x7fffffff) : best.v;
  }
}

// ---------------------------------------------------------------- host

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn_lm() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(f);
    else
      cudaGetLastError();
  });
  return fn;
}

// 2D bf16 map over [rows, cols] row-major, box [box_rows, 64], 128-byte
// swizzle; reads past the last row fill zeros
bool encode_rows(CUtensorMap* m, const void* ptr, int64_t rows, int64_t cols, uint32_t box_rows) {
  EncodeTiledFn fn = encode_fn_lm();
  if (!fn) return false;
  cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)cols * 2};
  cuuint32_t box[2] = {64, box_rows};
  cuuint32_t es[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int lm_validate(const tv_lmhead_desc* d) {
  if (!d) return TV_ERR_NULL;
  if (d->rows < 1 || d->rows > kMaxRowTiles * LM || d->hidden < 64 || d->hidden > 65536 || d->hidden % 64 ||
      d->vocab < 1)
    return TV_ERR_SHAPE;
  return TV_OK;
}

int lm_grid(const tv_lmhead_desc* d) {
  const int64_t RT = (d->rows + LM - 1) / LM;
  const int64_t units = ((int64_t)d->vocab + LV - 1) / LV * RT;
  const int64_t sms = num_sms();
  return (int)(units < sms ? units : sms);
}

}  // namespace
}  // namespace tv

using namespace tv;

extern "C" {

int tv_lm_head_workspace_size(const tv_lmhead_desc* desc, size_t* bytes) {
  const int rc = lm_validate(desc);
  if (rc) return rc;
  if (!bytes) return TV_ERR_NULL;
  const int64_t parts = (int64_t)lm_grid(desc) * desc->rows;
  *bytes = (size_t)((parts * 4 + 255) / 256 * 256 + (parts * 4 + 255) / 256 * 256);
  return TV_OK;
}

int tv_lm_head_argmax(const tv_lmhead_desc* desc, const void* d_hidden, const void* d_weight, int32_t* d_argmax,
                      float* d_max_logit, void* d_workspace, size_t workspace_bytes, int32_t* d_status,
                      void* stream) {
  int rc = lm_validate(desc);
  if (rc) return rc;
  if (!d_hidden || !d_weight || !d_argmax || !d_workspace || !d_status) return TV_ERR_NULL;
  int64_t wbytes = 0;
  if (__builtin_mul_overflow((int64_t)desc->vocab, (int64_t)desc->hidden * 2, &wbytes)) return TV_ERR_OVERFLOW;
  if (!aligned16(d_hidden) || !aligned16(d_weight) || !aligned16(d_argmax) || !aligned16(d_workspace) ||
      !aligned16(d_status) || (d_max_logit && !aligned16(d_max_logit)))
    return TV_ERR_ALIGN;
  size_t need = 0;
  tv_lm_head_workspace_size(desc, &need);
  if (workspace_bytes < need) return TV_ERR_WORKSPACE;

  CUtensorMap tm_w, tm_h;
  if (!encode_rows(&tm_w, d_weight, desc->vocab, desc->hidden, LV) ||
      !encode_rows(&tm_h, d_hidden, desc->rows, desc->hidden, LM))
    return TV_ERR_CUDA;
  const int grid = lm_grid(desc);
  const int64_t parts = (int64_t)grid * desc->rows;
  LmParams p;
  p.part_v = static_cast<float*>(d_workspace);
  p.part_i = reinterpret_cast<int32_t*>(static_cast<char*>(d_workspace) + (parts * 4 + 255) / 256 * 256);
  p.status = d_status;
  p.R = desc->rows;
  p.Hd = desc->hidden;
  p.V = desc->vocab;
  p.RT = (desc->rows + LM - 1) / LM;
  p.units = (int)(((int64_t)desc->vocab + LV - 1) / LV * p.RT);
  p.KCH = desc->hidden / LKC;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = ensure_max_dynamic_smem<lmhead_argmax_kernel>((int)(kLSmem + 1024));
  if (e != cudaSuccess) return TV_ERR_CUDA;
  e = launch_dep(lmhead_argmax_kernel, dim3(grid), dim3(kLThreads), kLSmem + 1024, s, p, tm_w, tm_h);
  if (e != cudaSuccess) return TV_ERR_CUDA;
  e = launch_dep(lmhead_finish_kernel, dim3((desc->rows + 7) / 8), dim3(256), 0, s, (const float*)p.part_v,
                 (const int32_t*)p.part_i, grid, desc->rows, d_argmax, d_max_logit);
  return e == cudaSuccess ? TV_OK : TV_ERR_CUDA;
}

}  // extern "C"
