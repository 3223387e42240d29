// tcgen05 split-KV tree-verify attention on CTA pairs (bf16, head_dim 128 or
// 256), for KV heads whose query rows fill two or more 128-row tiles.
//
// Same method as the one-CTA kernel (flash-decode with a tree mask, "ADR-037
// — EAGLE-3 with dynamic tree port", phase rows E1.1-E1.5 and E4b.6), run by
// two CTAs of a cluster on two query-row tiles of the same KV head and key
// chunk, with M = 256 tcgen05.mma (cta_group::2):
//   S = Q K^T: each CTA holds its own 128 query rows and HALF of the keys of
//              every K tile (64 keys x d); the leader's MMA reads both halves.
//   O += P V:  P from each CTA's tensor memory; each CTA holds all 128 keys of
//              the V tile but only half of its columns (d/2).
// So each CTA stages 64 KB per 128-key tile (d = 256) instead of 128 KB: the
// ring of K/V slots holds twice as many tiles in flight, and every K/V byte
// crosses from L2 to the SMs once instead of twice.
//
//   warp 0     TMA producer (both CTAs): its Q tile, then its K half and V
//              half of each tile in MMA consumption order; completion is
//              counted on the leader's FULL barrier (expect_tx for both
//              halves by the leader, a plain arrive by the peer).
//   warp 1     owns the pair's tensor memory; lane 0 of the leader issues the
//              MMAs and multicasts every commit to both CTAs.
//   warps 4-11 softmax on the CTA's own rows, as in the one-CTA kernel;
//              P_FULL lives in the leader (512 arrivals).
// Every wait is bounded; the pair meets at a cluster barrier before freeing
// tensor memory.
#include <cuda.h>

#include <climits>
#include <mutex>

#include "tc_ptx.cuh"
#include "tv_internal.cuh"

namespace tv {
namespace {

using namespace tc;

constexpr int BM = 128;                         // query rows per CTA
constexpr int BN = 128;                         // keys per tile
constexpr int KH = 64;                          // keys per CTA in a K half
// key tiles of the chunk warmed in L2 before the dependency wait (measured on
// the 4K, 32K and batched workloads: 2 beats 1, 4 and 8 by up to 7%; warming
// further tiles while streaming was slower, up to 35% on the batched one)
constexpr int kPrefetchTiles = 2;
static_assert(kPrefetchTiles >= 0 && kPrefetchTiles <= 32, "one lane per prefetched tile");
constexpr uint64_t kWaitNs = 1000000000ull;
constexpr float kRescaleThreshold = 8.0f;       // rescale O when the max grows by > 2^8
constexpr int kThreads = 384;
constexpr int kSoftmax = 256;
constexpr int kSoftmaxWarps = kSoftmax / 32;   // barriers count warps: lane 0 arrives after __syncwarp
constexpr uint32_t kHeader = 3072;
constexpr uint32_t kSmemMax = 232448;

template <int D>
struct Cfg2 {
  static constexpr uint32_t SLOT = D * 128;      // K half (64 keys x D) == V half (128 keys x D/2)
  static constexpr uint32_t Q_BYTES = BM * D * 2;
  static constexpr int NS = (kSmemMax - kHeader - Q_BYTES) / SLOT;
  static constexpr uint32_t RING_BYTES = NS * SLOT;
  static constexpr int NBARS = 2 * NS + 13 + D / 32;   // ring, pipeline, epilogue boxes
  static constexpr uint32_t SMEM = kHeader + Q_BYTES + RING_BYTES;
  static_assert(NBARS * 8 + 8 <= 512, "barriers overflow the header");
  static_assert(SMEM <= kSmemMax, "shared memory over the per-block limit");
  static_assert(BM * D * 4 <= RING_BYTES, "the fp32 O tile must fit the ring for the epilogue");
};

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ uint32_t pack_bf16(float a, float b) {
  __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&h);
}

template <int D>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
tv_attn_tc2_kernel(const __grid_constant__ AttnParams p, const __grid_constant__ CUtensorMap tm_q,
                   const __grid_constant__ CUtensorMap tm_kc, const __grid_constant__ CUtensorMap tm_vc,
                   const __grid_constant__ CUtensorMap tm_kt, const __grid_constant__ CUtensorMap tm_vt,
                   const __grid_constant__ CUtensorMap tm_op) {
  using C = Cfg2<D>;
  constexpr int NS = C::NS;
  constexpr uint32_t SLOT = C::SLOT;
  constexpr unsigned kAll = 0xffffffffu;
  extern __shared__ __align__(1024) uint8_t smem_raw[];

  // ------------------------------------------------------- smem
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem_raw);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem_raw + C::NBARS * 8);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  float* xch = reinterpret_cast<float*>(smem_raw + 512);          // [2 parity][2 half][128 rows]
  uint8_t* sQ = smem_raw + kHeader;
  uint8_t* ring = sQ + C::Q_BYTES;
  auto bar = [&](int i) { return smem_u32(&bars[i]); };
  auto FULL = [&](int i) { return bar(i); };                      // used in the leader
  auto EMPTY = [&](int i) { return bar(NS + i); };
  const int bq = 2 * NS;
  const uint32_t Q_FULL = bar(bq), TAIL = bar(bq + 7), FIN = bar(bq + 8), XL = bar(bq + 11);
  auto BOX = [&](int i) { return bar(bq + 12 + i); };            // epilogue box i staged (D / 32 boxes)
  auto S_FULL = [&](int i) { return bar(bq + 1 + i); };
  auto P_FULL = [&](int i) { return bar(bq + 3 + i); };           // used in the leader
  auto O_DONE = [&](int i) { return bar(bq + 5 + i); };
  auto XCH = [&](int i) { return bar(bq + 9 + i); };

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (smem_u32(smem_raw) & 1023u) {                 // same for both CTAs of the pair
    dep_wait();
    if (tid == 0) set_status(p.status, TV_DEV_TIMEOUT);
    return;
  }
  // on-chip setup before the dependency wait: it overlaps the previous
  // kernel's tail when the launch is programmatic
  if (tid == 0) {
    for (int i = 0; i < NS; ++i) {
      mbar_init(FULL(i), 2);                        // leader's expect_tx arrive + peer's arrive
      mbar_init(EMPTY(i), 1);
    }
    mbar_init(Q_FULL, 2);
    for (int i = 0; i < 2; ++i) {
      mbar_init(S_FULL(i), 1);
      mbar_init(P_FULL(i), 2 * kSoftmaxWarps);     // one arrive per softmax warp of both CTAs
      mbar_init(O_DONE(i), 1);
      mbar_init(XCH(i), kSoftmaxWarps);
    }
    mbar_init(TAIL, 1);
    mbar_init(FIN, 1);
    mbar_init(XL, kSoftmaxWarps);
    // box i: the 4 warps of one half, once each
    for (int i = 0; i < D / 32; ++i) mbar_init(BOX(i), kSoftmaxWarps / 2);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (p.rows_per_tile < BM) {
    const int pad = BM - p.rows_per_tile;
    for (int e = tid; e < (D / 64) * pad * 8; e += blockDim.x) {
      const int kb = e / (pad * 8), r = p.rows_per_tile + (e / 8) % pad, c = e % 8;
      *reinterpret_cast<uint4*>(sQ + kb * (BM * 128) + r * 128 + c * 16) = make_uint4(0, 0, 0, 0);
    }
    fence_proxy_async_smem();
  }
  if (warp == 1) {
    tmem_alloc_pair(smem_u32(tmem_slot), 512);
    tmem_relinquish_pair();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tm_q);
    tma_prefetch_desc(&tm_kc);
    tma_prefetch_desc(&tm_vc);
    tma_prefetch_desc(&tm_kt);
    tma_prefetch_desc(&tm_vt);
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync_all();                               // both CTAs' barriers exist before any remote use
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  if (warp == 3) {
    // an idle warp warms L2 (and the TLB) for what the first steps read,
    // while the previous kernel may still run: the sequence's lengths, this
    // CTA's halves of the first kPrefetchTiles K and V tiles its chunk can
    // hold (bounded by the host's max_prefix, since the length itself is
    // not read yet) and, for the first sequence (rows start at 0), its query
    // tile.  These are hints: a prefetch has no effect on memory ordering,
    // so a line the previous kernel writes later is still read fresh, and a
    // page id read here only picks which lines to warm (a stale or invalid
    // id costs a wasted prefetch, never a wrong value).
    const int b = blockIdx.z, g = blockIdx.y / p.splits, s = blockIdx.y % p.splits;
    const uint32_t rank = cluster_ctarank();
    const int64_t c0 = (int64_t)s * p.chunk;
    const int64_t c1 = min(p.max_prefix, c0 + p.chunk);
    const int npf = c1 > c0 ? (int)min((int64_t)kPrefetchTiles, (c1 - c0 + BN - 1) / BN) : 0;
    if (lane == 0) {
      prefetch_l2(p.prefix_len + b);
      prefetch_l2(p.node_offsets + b);
      if (b == 0)
        for (int kb = 0; kb < D / 64; ++kb) tma_prefetch_3d(&tm_q, kb * 64, g * p.G, blockIdx.x * p.rows_per_tile / p.G);
    }
    if (!p.paged) {
      const int64_t row = ((int64_t)b * p.Hkv + g) * p.capacity + c0 + (int64_t)lane * BN;   // lane = tile
      if (lane < npf && row + BN <= (int64_t)INT_MAX) {
        for (int bx = 0; bx < D / 64; ++bx) tma_prefetch_2d(&tm_kc, bx * 64, (int)row + KH * (int)rank);
        for (int bx = 0; bx < D / 128; ++bx) tma_prefetch_2d(&tm_vc, (D / 2) * (int)rank + bx * 64, (int)row);
      }
    } else {
      // pages of the first tiles that hold keys below c1 (c1 <= capacity, so every index
      // stays inside the sequence's row of the page table)
      const int npg = (int)min((int64_t)npf * (BN / kPageSize), (c1 - c0 + kPageSize - 1) / kPageSize);
      for (int pg = lane; pg < npg; pg += 32) {
        const int64_t pos = c0 + (int64_t)pg * kPageSize;
        const int pid = p.page_table[(int64_t)b * p.max_pages + pos / kPageSize];
        if (pid >= 0 && pid < p.num_pages) {
          const int row = (int)(((int64_t)pid * p.Hkv + g) * kPageSize);
          if ((pg % (BN / kPageSize)) / (KH / kPageSize) == (int)rank)   // a page of this CTA's K half
            for (int bx = 0; bx < D / 64; ++bx) tma_prefetch_2d(&tm_kc, bx * 64, row);
          for (int bx = 0; bx < D / 128; ++bx) tma_prefetch_2d(&tm_vc, (D / 2) * (int)rank + bx * 64, row);
        }
      }
    }
  }
  dep_wait();
  dep_launch();

  // Speculative first copies, issued before the sequence's lengths are known
  // (a dependent round trip they then overlap): the query tile when its rows
  // start at 0 (the first sequence) and this CTA's half of the chunk's first
  // K tile on a contiguous cache (its position needs no length).  If the
  // chunk turns out to hold no prefix tile, slot 0's first fill is junk: the
  // MMA issuer releases it unused and the ring starts at slot 1.  A pair with
  // nothing to do waits for these copies before it leaves.
  const bool spec_q = blockIdx.z == 0;
  const bool spec_k = !p.paged && (int64_t)(blockIdx.y % p.splits) * p.chunk < p.max_prefix;
  if (warp == 0 && lane == 0) {
    const uint32_t rk = cluster_ctarank();
    const int gg = blockIdx.y / p.splits, ss = blockIdx.y % p.splits;
    if (spec_q) {
      const uint32_t qf = map_to_cta(Q_FULL, 0);
      if (rk == 0) mbar_expect_tx(Q_FULL, 2u * (uint32_t)p.rows_per_tile * 128u * (D / 64));
      for (int kb = 0; kb < D / 64; ++kb)
        tma2_load_3d(smem_u32(sQ + kb * (BM * 128)), &tm_q, qf, kb * 64, gg * p.G,
                     (int)blockIdx.x * p.rows_per_tile / p.G);
      if (rk != 0) mbar_arrive_cluster_relaxed(qf);
    }
    if (spec_k) {
      const uint32_t fl = map_to_cta(FULL(0), 0);
      if (rk == 0) mbar_expect_tx(FULL(0), 2 * SLOT);
      const int64_t row = ((int64_t)blockIdx.z * p.Hkv + gg) * p.capacity + (int64_t)ss * p.chunk + KH * rk;
      for (int bx = 0; bx < D / 64; ++bx) tma2_load_2d(smem_u32(ring + bx * (KH * 128)), &tm_kc, fl, bx * 64, (int)row);
      if (rk != 0) mbar_arrive_cluster_relaxed(fl);
    }
  }

  // ------------------------------------------------------- work (pair-uniform)
  const uint32_t rank = cluster_ctarank();          // 0 = leader
  const int rt = blockIdx.x;                        // row tile (pair = rt / 2)
  const int g = blockIdx.y / p.splits;
  const int s = blockIdx.y % p.splits;
  const int b = blockIdx.z;
  const int64_t Praw = p.prefix_len[b];
  int o0 = 0, n = 1;
  bool active = seq_rows(p.node_offsets, b, p.R, p.max_nodes, p.status, &o0, &n);
  const int G = p.G;
  const int nrows = n * G;
  const int m0 = rt * p.rows_per_tile;
  active = active && (rt & ~1) * p.rows_per_tile < nrows;   // the pair's first tile has rows
  const int64_t P = clamp_prefix(Praw, p.max_prefix, p.capacity);
  if (active && P != Praw && tid == 0 && rt == 0 && s == 0 && g == 0) set_status(p.status, TV_DEV_BAD_PREFIX);
  const int nch = num_chunks(P, p.chunk, p.tree_tile);
  active = active && s < nch;
  const int64_t k_begin = (int64_t)s * p.chunk;
  const int64_t k_end = min(P, k_begin + p.chunk);
  const bool has_tree = (s == nch - 1);
  const int npt = (int)((k_end - k_begin + BN - 1) / BN);
  const int T = npt + (has_tree ? 1 : 0);
  const int tail_valid = npt > 0 ? (int)(k_end - (k_begin + (int64_t)(npt - 1) * BN)) : BN;
  const bool rows_here = m0 < nrows;                // the peer of a one-tile pair only helps

  const bool junk0 = spec_k && npt == 0;           // slot 0's first fill is not this chunk's
  if (!active) {
    // nothing for this pair: wait for the speculative copies (the leader's
    // barriers count both CTAs' bytes), then teardown
    if (warp == 0 && lane == 0 && rank == 0) {
      if (spec_k) mbar_wait(FULL(0), 0, abort_flag, kWaitNs);
      if (spec_q) mbar_wait(Q_FULL, 0, abort_flag, kWaitNs);
    }
  } else if (warp == 0) {
    // ============================================================ producer
    const bool leader = rank == 0;
    const uint32_t qbytes = (uint32_t)p.rows_per_tile * 128u * (D / 64);
    if (lane == 0 && !spec_q) {
      const uint32_t qf = map_to_cta(Q_FULL, 0);
      if (leader) mbar_expect_tx(Q_FULL, 2 * qbytes);
      for (int kb = 0; kb < D / 64; ++kb)
        tma2_load_3d(smem_u32(sQ + kb * (BM * 128)), &tm_q, qf, kb * 64, g * G, o0 + m0 / G);
      if (!leader) mbar_arrive_cluster_relaxed(qf);
    }
    int j = junk0 ? 1 : 0, tail_uses = 0;
    bool ok = true;
    const int oob_row = p.paged ? (int)(p.num_pages * p.Hkv * kPageSize) : 0;
    auto page_id = [&](int tile) -> int {           // raw page id of this lane's page (lanes 0-7), or INT_MIN
      if (!p.paged || tile >= npt || lane >= BN / kPageSize) return INT_MIN;
      const int64_t pos = k_begin + (int64_t)tile * BN + lane * kPageSize;
      if (pos >= k_end) return INT_MIN;
      return p.page_table[(int64_t)b * p.max_pages + pos / kPageSize];
    };
    auto page_row = [&](int pid) -> int {
      if (pid == INT_MIN) return -1;
      if (pid >= 0 && pid < p.num_pages) return (int)(((int64_t)pid * p.Hkv + g) * kPageSize);
      set_status(p.status, TV_DEV_BAD_PAGE);
      return oob_row;
    };
    // pages of [a, a + len) that hold keys below k_end
    auto pages_in = [&](int64_t a, int len) -> int {
      const int64_t e = min(a + len, k_end);
      return e > a ? (int)((e - a + kPageSize - 1) / kPageSize) : 0;
    };
    int pid_a = page_id(0), pid_b = page_id(1), pid_c = page_id(2), pid_d = page_id(3);
    int row_k = -1, row_v = -1;
    for (int t = 0; t <= T && ok; ++t) {
      row_v = row_k;
      row_k = page_row(pid_a);
      pid_a = pid_b;
      pid_b = pid_c;
      pid_c = pid_d;
      pid_d = page_id(t + 4);
      for (int kind = 0; kind < 2 && ok; ++kind, ++j) {      // 0: K(t) half, 1: V(t-1) half
        const int tile = kind == 0 ? t : t - 1;
        if ((kind == 0 && t >= T) || (kind == 1 && t < 1)) { --j; continue; }
        if (spec_k && !junk0 && t == 0 && kind == 0) continue;   // K(0) is in slot 0 already
        const bool tree = (tile == npt);
        const bool tail_fix = (kind == 1) && !tree && tile == npt - 1 && tail_valid < BN;
        const int slot = j % NS, use = j / NS;
        if (use > 0 && !__all_sync(kAll, mbar_wait(EMPTY(slot), (use - 1) & 1, abort_flag, kWaitNs))) {
          ok = false;
          break;
        }
        uint8_t* dst = ring + slot * SLOT;
        const uint32_t full_l = map_to_cta(FULL(slot), 0);
        const uint32_t fb = tail_fix ? map_to_cta(TAIL, rank) : full_l;
        const int64_t t0 = k_begin + (int64_t)tile * BN;
        // bytes both halves of this slot bring (the leader expects them all)
        uint32_t total = 2 * SLOT;
        if (p.paged && !tree) {
          if (kind == 0) total = (uint32_t)(pages_in(t0, KH) + pages_in(t0 + KH, KH)) * (D / 64) * (kPageSize * 128u);
          else total = 2u * (uint32_t)pages_in(t0, BN) * (D / 128) * (kPageSize * 128u);
        }
        const uint32_t mine = tail_fix ? (total / 2) : 0;   // a tail slot's own bytes go to TAIL
        if (lane == 0) {
          if (tail_fix) mbar_expect_tx(TAIL, mine);
          else if (leader) mbar_expect_tx(FULL(slot), total);
        }
        __syncwarp();
        if (tree || !p.paged) {
          if (lane == 0) {
            if (kind == 0) {                         // K half: keys [64 rank, +64) x all D columns
              const int64_t row = tree ? (int64_t)g * p.R + o0 + KH * rank
                                       : ((int64_t)b * p.Hkv + g) * p.capacity + t0 + KH * rank;
              for (int bx = 0; bx < D / 64; ++bx)
                tma2_load_2d(smem_u32(dst + bx * (KH * 128)), tree ? &tm_kt : &tm_kc, fb, bx * 64, (int)row);
            } else {                                 // V half: all 128 keys x columns [D/2 rank, +D/2)
              const int64_t row = tree ? (int64_t)g * p.R + o0 : ((int64_t)b * p.Hkv + g) * p.capacity + t0;
              for (int bx = 0; bx < D / 128; ++bx)
                tma2_load_2d(smem_u32(dst + bx * (BN * 128)), tree ? &tm_vt : &tm_vc, fb,
                             (D / 2) * (int)rank + bx * 64, (int)row);
            }
          }
        } else {
          const int my_row = kind == 0 ? row_k : row_v;
          if (kind == 0) {
            // lanes 4 rank .. 4 rank + 3 own the pages of this CTA's 64 keys
            const int pg = lane - 4 * (int)rank;
            if (pg >= 0 && pg < 4 && my_row >= 0)
              for (int bx = 0; bx < D / 64; ++bx)
                tma2_load_2d(smem_u32(dst + bx * (KH * 128) + pg * kPageSize * 128), &tm_kc, fb, bx * 64, my_row);
          } else if (my_row >= 0) {
            for (int bx = 0; bx < D / 128; ++bx)
              tma2_load_2d(smem_u32(dst + bx * (BN * 128) + lane * kPageSize * 128), &tm_vc, fb,
                           (D / 2) * (int)rank + bx * 64, my_row);
          }
        }
        __syncwarp();
        if (tail_fix) {
          // this CTA's rows past the prefix end become zeros before any MMA reads them
          if (!__all_sync(kAll, mbar_wait(TAIL, tail_uses & 1, abort_flag, kWaitNs))) {
            ok = false;
            break;
          }
          ++tail_uses;
          const int nz = BN - tail_valid;
          for (int e = lane; e < (D / 128) * nz * 8; e += 32) {
            const int bx = e / (nz * 8), r = tail_valid + (e / 8) % nz, q16 = e % 8;
            *reinterpret_cast<uint4*>(dst + bx * (BN * 128) + r * 128 + q16 * 16) = make_uint4(0, 0, 0, 0);
          }
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) mbar_arrive_cluster_release(full_l);   // the zeros must reach the pair's MMA
        } else if (!leader && lane == 0) {
          mbar_arrive_cluster_relaxed(full_l);     // the bytes themselves are counted by complete_tx
        }
      }
    }
  } else if (warp == 1) {
    // ============================================================ MMA issuer (leader)
    if (lane == 0 && rank == 0) {
      constexpr uint32_t ID_QK = idesc_bf16_f32(2 * BM, BN, 0, 0);
      constexpr uint32_t ID_PV = idesc_bf16_f32(2 * BM, D, 0, 1);
      bool ok = mbar_wait(Q_FULL, 0, abort_flag, kWaitNs);
      tc_fence_after();
      const uint32_t q_addr = smem_u32(sQ);
      const uint32_t ring_addr = smem_u32(ring);
      int j = 0;
      if (ok && junk0) {                            // release slot 0's speculative fill unused
        ok = mbar_wait(FULL(0), 0, abort_flag, kWaitNs);
        mma_commit_pair(EMPTY(0));
        j = 1;
      }
      for (int t = 0; t <= T && ok; ++t) {
        if (t < T) {
          const uint32_t sbuf = tmem + (uint32_t)((t & 1) * 128);
          const int slot = j % NS;
          if (!mbar_wait(FULL(slot), (j / NS) & 1, abort_flag, kWaitNs)) { ok = false; break; }
          tc_fence_after();
          const uint32_t kaddr = ring_addr + slot * SLOT;
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {      // 16-column steps over d
            const uint64_t a = smem_desc(q_addr + (kk >> 2) * (BM * 128) + (kk & 3) * 32, 16, 1024, 2);
            const uint64_t bd = smem_desc(kaddr + (kk >> 2) * (KH * 128) + (kk & 3) * 32, 16, 1024, 2);
            mma_pair_ss(sbuf, a, bd, ID_QK, kk > 0 ? 1u : 0u);
          }
          mma_commit_pair(EMPTY(slot));
          mma_commit_pair(S_FULL(t & 1));
          ++j;
        }
        if (t >= 1) {
          const int u = t - 1;
          const uint32_t pbuf = tmem + (uint32_t)((u & 1) * 128);
          if (!mbar_wait(P_FULL(u & 1), (u >> 1) & 1, abort_flag, kWaitNs)) { ok = false; break; }
          tc_fence_after();
          const int slot = j % NS;
          if (!mbar_wait(FULL(slot), (j / NS) & 1, abort_flag, kWaitNs)) { ok = false; break; }
          tc_fence_after();
          const uint32_t vaddr = ring_addr + slot * SLOT;
#pragma unroll
          for (int kk = 0; kk < BN / 16; ++kk) {     // 16 keys per step
            const uint64_t bd = smem_desc(vaddr + kk * (16 * 128), BN * 128, 1024, 2);
            mma_pair_ts(tmem + 256, pbuf + kk * 8, bd, ID_PV, (u > 0 || kk > 0) ? 1u : 0u);
          }
          mma_commit_pair(EMPTY(slot));
          mma_commit_pair(O_DONE(u & 1));
          ++j;
        }
      }
      mma_commit_pair(FIN);
      mbar_wait(FIN, 0, abort_flag, kWaitNs);
    }
  } else if (warp == 2) {
    // ============================================================ partials store
    // one 128-byte-wide box of the partial tile at a time (32 fp32 or 64 bf16
    // columns), as soon as the softmax warps of its half have staged it;
    // every box barrier is arrived in all paths, so the waits here end
    if (lane == 0) {
      const bool store = !(p.out != nullptr && nch == 1) && rows_here;
      const int row0 = (int)(((int64_t)b * p.Hkv + g) * p.row_tiles + rt) * BM;   // first row of the tile
      const int cols = p.part_bf16 ? 64 : 32;     // columns per box
      const int per_half = (D / 2) / cols;
      bool issued = false;
      for (int j = 0; j < per_half; ++j) {
        for (int hf = 0; hf < 2; ++hf) {
          const int bx = hf * per_half + j;
          const bool in = mbar_wait(BOX(bx), 0, abort_flag, kWaitNs);
          if (in && store && !*abort_flag) {
            tma_store_3d(&tm_op, smem_u32(ring + bx * (BM * 128)), hf * (D / 2) + j * cols, s, row0);
            bulk_commit_group();
            issued = true;
          }
        }
      }
      if (issued) bulk_wait_read_all();
    }
  } else if (warp >= 4) {
    // ============================================================ softmax (own rows)
    const int half = (tid - 128) >> 7;
    const int r = (tid - 128) & 127;
    const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
    const bool row_ok = r < p.rows_per_tile && (m0 + r) < nrows;
    const int node = (m0 + r) / G;
    const uint64_t anc = row_ok ? p.anc[o0 + node] : 0ull;
    const float c2 = p.scale_log2;
    const int kofs = half * (BN / 2);
    float m_ref = -INFINITY, l = 0.f;
    bool ok = true;
    for (int t = 0; t < T && ok; ++t) {
      if (!__all_sync(kAll, mbar_wait(S_FULL(t & 1), (t >> 1) & 1, abort_flag, kWaitNs))) { ok = false; break; }
      tc_fence_after();
      const uint32_t sbuf = tmem + lane_base + (uint32_t)((t & 1) * 128);
      float sv[BN / 2];
      {
        uint32_t rr[64];
        tmem_ld_x64(sbuf + kofs, rr);
#pragma unroll
        for (int e = 0; e < 64; ++e) sv[e] = __uint_as_float(rr[e]);
      }
      const bool tree = (t == npt);
      const bool partial = tree || (t == npt - 1 && tail_valid < BN);
      if (partial) {
        const int lim = tree ? min(n, 64) : tail_valid;
#pragma unroll
        for (int e = 0; e < 64; ++e) {
          const int key = kofs + e;
          bool vis = key < lim;
          if (tree) vis = vis && ((anc >> (key & 63)) & 1ull);
          sv[e] = vis ? sv[e] : -INFINITY;
        }
      }
      float mx8[8];
#pragma unroll
      for (int a = 0; a < 8; ++a) mx8[a] = sv[a];
#pragma unroll
      for (int e = 8; e < 64; ++e) mx8[e & 7] = fmaxf(mx8[e & 7], sv[e]);
      float mx = fmaxf(fmaxf(fmaxf(mx8[0], mx8[1]), fmaxf(mx8[2], mx8[3])),
                       fmaxf(fmaxf(mx8[4], mx8[5]), fmaxf(mx8[6], mx8[7])));
      float* xb = xch + (t & 1) * 256;
      xb[half * 128 + r] = mx;
      __syncwarp();
      if (lane == 0) mbar_arrive(XCH(t & 1));
      if (!__all_sync(kAll, mbar_wait(XCH(t & 1), (t >> 1) & 1, abort_flag, kWaitNs))) { ok = false; break; }
      mx = fmaxf(mx, xb[(half ^ 1) * 128 + r]);
      const float m_tile = mx == -INFINITY ? -INFINITY : mx * c2;
      const float m_new = fmaxf(m_ref, m_tile);
      const bool first = (m_ref == -INFINITY);
      const bool need = !first && (m_new > m_ref + kRescaleThreshold);
      if (__any_sync(kAll, need)) {
        const int u = t - 1;
        if (!__all_sync(kAll, mbar_wait(O_DONE(u & 1), (u >> 1) & 1, abort_flag, kWaitNs))) { ok = false; break; }
        tc_fence_after();
        const float alpha = need ? ex2(m_ref - m_new) : 1.f;
#pragma unroll 1
        for (int q = 0; q < D / 64; ++q) {
          uint32_t rr[32];
          const uint32_t oa = tmem + lane_base + 256 + half * (D / 2) + q * 32;
          tmem_ld_x32(oa, rr);
#pragma unroll
          for (int e = 0; e < 32; ++e) rr[e] = __float_as_uint(__uint_as_float(rr[e]) * alpha);
          tmem_st_x32(oa, rr);
        }
        if (need) {
          l *= alpha;
          m_ref = m_new;
        }
      }
      if (first) m_ref = m_new;
      const float nm = m_ref == -INFINITY ? 0.f : -m_ref;
      float l8[8];
#pragma unroll
      for (int a = 0; a < 8; ++a) l8[a] = 0.f;
      uint32_t pk[32];
#pragma unroll
      for (int e = 0; e < 32; ++e) {
        const float p0 = ex2(fmaf(sv[2 * e], c2, nm));
        const float p1 = ex2(fmaf(sv[2 * e + 1], c2, nm));
        l8[(2 * e) & 7] += p0;
        l8[(2 * e + 1) & 7] += p1;
        pk[e] = pack_bf16(p0, p1);
      }
      l += ((l8[0] + l8[1]) + (l8[2] + l8[3])) + ((l8[4] + l8[5]) + (l8[6] + l8[7]));
      tmem_st_x32(sbuf + half * 32, pk);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(map_to_cta(P_FULL(t & 1), 0));
    }
    // epilogue, as in the one-CTA kernel, for this CTA's own rows: the two
    // halves' sums are added; a sequence with one chunk writes normalised
    // rows directly, otherwise the fp32 tile is staged in the (idle) ring in
    // 128-byte swizzled 32-column boxes, each box's barrier arrived as soon
    // as it is written (in every path, so warp 2's waits always end)
    const int u = T - 1;
    const bool direct = p.out != nullptr && nch == 1;
    const bool epi = ok && __all_sync(kAll, mbar_wait(O_DONE(u & 1), (u >> 1) & 1, abort_flag, kWaitNs));
    bool got = false;
    float lsum = 0.f;
    if (epi) {
      tc_fence_after();
      float* xb = xch + (T & 1) * 256;
      xb[half * 128 + r] = l;
      __syncwarp();
      if (lane == 0) mbar_arrive(XL);
      got = __all_sync(kAll, mbar_wait(XL, 0, abort_flag, kWaitNs));
      lsum = l + xb[(half ^ 1) * 128 + r];
    }
    const float inv = lsum > 0.f ? 1.f / lsum : 0.f;
    const int64_t rowg = o0 + node;
    const int h = g * G + (m0 + r) % G;
#pragma unroll 1
    for (int qq = 0; qq < D / 128; ++qq) {         // 64 columns per TMEM load, two 32-column steps
      uint32_t rv[64];
      if (epi) tmem_ld_x64(tmem + lane_base + 256 + half * (D / 2) + qq * 64, rv);
#pragma unroll
      for (int sub = 0; sub < 2; ++sub) {
        const int q = 2 * qq + sub;
        const uint32_t* rr = rv + 32 * sub;
        if (epi && got && rows_here && direct && row_ok) {
          const int64_t e = (rowg * p.Hq + h) * D + half * (D / 2) + q * 32;
          if (p.out_bf16) {
            uint4* ob = reinterpret_cast<uint4*>(reinterpret_cast<__nv_bfloat16*>(p.out) + e);
#pragma unroll
            for (int e8 = 0; e8 < 4; ++e8) {
              uint4 w4;
              w4.x = pack_bf16(__uint_as_float(rr[8 * e8 + 0]) * inv, __uint_as_float(rr[8 * e8 + 1]) * inv);
              w4.y = pack_bf16(__uint_as_float(rr[8 * e8 + 2]) * inv, __uint_as_float(rr[8 * e8 + 3]) * inv);
              w4.z = pack_bf16(__uint_as_float(rr[8 * e8 + 4]) * inv, __uint_as_float(rr[8 * e8 + 5]) * inv);
              w4.w = pack_bf16(__uint_as_float(rr[8 * e8 + 6]) * inv, __uint_as_float(rr[8 * e8 + 7]) * inv);
              ob[e8] = w4;
            }
          } else {
            float4* of = reinterpret_cast<float4*>(reinterpret_cast<float*>(p.out) + e);
#pragma unroll
            for (int e4 = 0; e4 < 8; ++e4)
              of[e4] = make_float4(__uint_as_float(rr[4 * e4]) * inv, __uint_as_float(rr[4 * e4 + 1]) * inv,
                                   __uint_as_float(rr[4 * e4 + 2]) * inv, __uint_as_float(rr[4 * e4 + 3]) * inv);
          }
        } else if (epi && got && rows_here && !direct) {
          // row r of the partial O_s / l_s: 128-byte box rows, 16-byte chunk
          // c at chunk c ^ (r & 7)
          if (p.part_bf16) {                       // 64 columns per box: this step fills half a row
            uint8_t* box = ring + (uint32_t)(half * (D / 128) + qq) * (BM * 128) + r * 128;
#pragma unroll
            for (int c4 = 0; c4 < 4; ++c4) {
              uint4 w4;
              w4.x = pack_bf16(__uint_as_float(rr[8 * c4 + 0]) * inv, __uint_as_float(rr[8 * c4 + 1]) * inv);
              w4.y = pack_bf16(__uint_as_float(rr[8 * c4 + 2]) * inv, __uint_as_float(rr[8 * c4 + 3]) * inv);
              w4.z = pack_bf16(__uint_as_float(rr[8 * c4 + 4]) * inv, __uint_as_float(rr[8 * c4 + 5]) * inv);
              w4.w = pack_bf16(__uint_as_float(rr[8 * c4 + 6]) * inv, __uint_as_float(rr[8 * c4 + 7]) * inv);
              *reinterpret_cast<uint4*>(box + (((sub * 4 + c4) ^ (r & 7)) * 16)) = w4;
            }
          } else {                                 // 32 fp32 columns per box
            uint8_t* box = ring + (uint32_t)(half * (D / 64) + q) * (BM * 128) + r * 128;
#pragma unroll
            for (int c4 = 0; c4 < 8; ++c4)
              *reinterpret_cast<uint4*>(box + ((c4 ^ (r & 7)) * 16)) =
                  make_uint4(__float_as_uint(__uint_as_float(rr[4 * c4]) * inv),
                             __float_as_uint(__uint_as_float(rr[4 * c4 + 1]) * inv),
                             __float_as_uint(__uint_as_float(rr[4 * c4 + 2]) * inv),
                             __float_as_uint(__uint_as_float(rr[4 * c4 + 3]) * inv));
          }
        }
        if (!p.part_bf16) {                        // an fp32 box is one 32-column step
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) mbar_arrive(BOX(half * (D / 64) + q));
        }
      }
      if (p.part_bf16) {                           // a bf16 box is the whole 64-column load
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(BOX(half * (D / 128) + qq));
      }
    }
    if (epi && got && rows_here && !direct)
      p.ml_part[partial_slot(s, b, g, rt, r, p.Hkv, p.row_tiles, BM, p.splits)] = make_float2(row_ok ? m_ref : -INFINITY, row_ok ? lsum : 0.f);
  }

  // ------------------------------------------------------- teardown (pair)
  // The leader's last commit (FIN) reaches both CTAs after every earlier
  // commit: once the peer has seen it, no arrive from the pair's MMAs is in
  // flight towards its shared memory, and an execution-only cluster barrier
  // keeps either CTA from leaving before the other is done.
  if (active && warp == 1 && lane == 0 && rank != 0) mbar_wait(FIN, 0, abort_flag, kWaitNs);
  tc_fence_before();
  __syncthreads();
  if (tid == 0 && *abort_flag) set_status(p.status, TV_DEV_TIMEOUT);
  cluster_sync_relaxed();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem, 512);
  }
}

// ------------------------------------------------------------------ host

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn2() {
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

bool encode2(CUtensorMap* m, const void* ptr, int rank, const cuuint64_t* dims, const cuuint64_t* strides,
             const cuuint32_t* box, CUtensorMapDataType type = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16) {
  EncodeTiledFn fn = encode_fn2();
  if (!fn) return false;
  cuuint32_t es[3] = {1, 1, 1};
  return fn(m, type, rank, const_cast<void*>(ptr), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
         CUDA_SUCCESS;
}

template <int D>
cudaError_t launch_tc2_t(const AttnParams& p, cudaStream_t st) {
  CUtensorMap mq, mkc, mvc, mkt, mvt, mop;
  const cuuint64_t row_bytes = (cuuint64_t)D * 2;
  {
    cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)p.Hq, (cuuint64_t)p.R};
    cuuint64_t strides[2] = {row_bytes, row_bytes * p.Hq};
    cuuint32_t box[3] = {64, (cuuint32_t)p.G, (cuuint32_t)(BM / p.G)};
    if (!encode2(&mq, p.q, 3, dims, strides, box)) return cudaErrorInvalidValue;
  }
  {
    const cuuint64_t rows = p.paged ? (cuuint64_t)p.num_pages * p.Hkv * kPageSize
                                    : (cuuint64_t)p.B * p.Hkv * p.capacity;
    cuuint64_t dims[2] = {(cuuint64_t)D, rows};
    cuuint64_t strides[1] = {row_bytes};
    cuuint32_t kbox[2] = {64, (cuuint32_t)(p.paged ? kPageSize : KH)};
    cuuint32_t vbox[2] = {64, (cuuint32_t)(p.paged ? kPageSize : BN)};
    if (!encode2(&mkc, p.k_cache, 2, dims, strides, kbox) || !encode2(&mvc, p.v_cache, 2, dims, strides, vbox))
      return cudaErrorInvalidValue;
  }
  {
    cuuint64_t dims[2] = {(cuuint64_t)D, (cuuint64_t)p.Hkv * p.R};
    cuuint64_t strides[1] = {row_bytes};
    cuuint32_t kbox[2] = {64, KH};
    cuuint32_t vbox[2] = {64, BN};
    if (!encode2(&mkt, p.k_tree, 2, dims, strides, kbox) || !encode2(&mvt, p.v_tree, 2, dims, strides, vbox))
      return cudaErrorInvalidValue;
  }
  {
    // partials [rows][splits][D] (partial_slot), fp32 (boxes of 32 columns)
    // or bf16 (64); a CTA stores one split of a 128-row tile
    const cuuint64_t es = p.part_bf16 ? 2 : 4;
    const cuuint64_t rows = (cuuint64_t)p.B * p.Hkv * p.row_tiles * BM;
    cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)p.splits, rows};
    cuuint64_t strides[2] = {(cuuint64_t)D * es, (cuuint64_t)D * es * p.splits};
    cuuint32_t box[3] = {p.part_bf16 ? 64u : 32u, 1u, BM};
    if (!encode2(&mop, p.o_part, 3, dims, strides, box,
                 p.part_bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32))
      return cudaErrorInvalidValue;
  }
  cudaError_t e = ensure_max_dynamic_smem<tv_attn_tc2_kernel<D>>((int)Cfg2<D>::SMEM);
  if (e != cudaSuccess) return e;
  dim3 grid(2 * ((p.row_tiles + 1) / 2), p.Hkv * p.splits, p.B);
  return launch_dep(tv_attn_tc2_kernel<D>, grid, dim3(kThreads), Cfg2<D>::SMEM, st, p, mq, mkc, mvc, mkt, mvt, mop);
}

}  // namespace

cudaError_t launch_attn_tc2(const AttnParams& p, cudaStream_t s) {
  if (p.d == 128) return launch_tc2_t<128>(p, s);
  return launch_tc2_t<256>(p, s);
}

}  // namespace tv
