// tcgen05 tensor-core split-KV tree-verify attention (bf16 Q/K/V, fp32
// accumulation and softmax), head_dim 128 or 256.
//
// The method is flash-decode with a tree mask ("ADR-037 — EAGLE-3 with
// dynamic tree port", phase rows E1.1-E1.5 and E4b.6): each CTA walks a
// chunk of keys with an online softmax and leaves an unnormalised partial
// output O, its running maximum m (base-2 units: score * scale * log2 e) and
// running sum l; merge_kernel combines the chunks.
//
// CTA = (128-row query tile, KV head g, key chunk s, sequence b).  Query row
// m of a tile is node m / G, group head m % G of KV head g, so the G query
// heads that share a KV head form one dense M=128 tile and every K/V tile is
// read once for all of them.
//
//   warp 0      TMA producer: the Q tile once, then 32 KB K/V chunks (128 keys
//               x 128 columns, 128-byte swizzled) through a ring of slots in
//               exactly the order the MMA consumes them: K(0), K(1), V(0),
//               K(2), V(1), ...
//   warp 1      owns tensor memory; lane 0 issues tcgen05.mma:
//               S(t) = Q K(t)^T into one of two 128-column TMEM buffers, then
//               O += P(t-1) V(t-1) with P read from TMEM.
//   warps 4-11  softmax, two threads per query row (its TMEM lane), each
//               taking half of the tile's keys: load the S half-row, mask,
//               exchange the half-row maxima, P = 2^(s*c - m) written back
//               over the S columns as bf16 pairs, running sum; rescale the O
//               row in TMEM only when the maximum grows by more than 2^8; at
//               the end write the partial (O, m, l).
//
// Keys: the chunk's prefix positions in 128-key tiles, then (in the last
// chunk of the sequence) one tile of the sequence's tree keys masked by the
// row's ancestor bits.  Rows past the prefix end in the last tile are masked
// in S and zeroed in the V chunk (0 x NaN would poison P V).
//
// Every mbarrier wait is bounded (1 s); on a timeout the CTA raises
// TV_DEV_TIMEOUT, drains its own copies and MMAs, frees tensor memory and
// returns.
#include <cuda.h>

#include <climits>
#include <mutex>

#include "tc_ptx.cuh"
#include "tv_internal.cuh"

namespace tv {
namespace {

using namespace tc;

constexpr int BM = 128;                         // query rows per tile
constexpr int BN = 128;                         // keys per tile
constexpr int CH = 128;                         // columns of d per chunk
// key tiles of the chunk warmed in L2 before the dependency wait (measured on
// the 4K, 32K and batched workloads: 2 beats 1, 4 and 8 by up to 7%; warming
// further tiles while streaming was slower, up to 35% on the batched one)
constexpr int kPrefetchTiles = 2;
static_assert(kPrefetchTiles >= 0 && kPrefetchTiles <= 32, "one lane per prefetched tile");
constexpr uint32_t BOX_BYTES = BN * 128;        // one TMA box: 128 rows x 64 bf16
constexpr uint32_t CHUNK_BYTES = 2 * BOX_BYTES; // 128 keys x 128 columns
constexpr uint64_t kWaitNs = 1000000000ull;
constexpr float kRescaleThreshold = 8.0f;       // rescale O when the max grows by > 2^8
constexpr int kThreads = 384;                   // warps 0 producer, 1 MMA, 2-3 idle, 4-11 softmax
constexpr int kSoftmax = 256;
constexpr int kSoftmaxWarps = kSoftmax / 32;   // barriers count warps: lane 0 arrives after __syncwarp                   // two warpgroups, each half of a row's keys
constexpr uint32_t kHeader = 3072;              // barriers, TMEM address, row exchange (then 1 KB aligned)

template <int D>
struct Cfg {
  static constexpr int CPT = D / CH;              // chunks per K (or V) tile
  static constexpr int NS = D == 256 ? 5 : 6;     // ring slots
  static constexpr uint32_t Q_BYTES = BM * D * 2;
  static constexpr uint32_t RING_BYTES = NS * CHUNK_BYTES;
  static constexpr int NBARS = 2 * NS + 12 + D / 32;   // ring, pipeline, epilogue boxes
  static constexpr uint32_t SMEM = kHeader + Q_BYTES + RING_BYTES;
  static_assert(NBARS * 8 + 8 <= 256, "barriers overflow the header");
  static_assert(SMEM <= 232448, "shared memory over the 227 KB per-block limit");
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
__global__ void __launch_bounds__(kThreads, 1)
tv_attn_tc_kernel(const __grid_constant__ AttnParams p, const __grid_constant__ CUtensorMap tm_q,
                  const __grid_constant__ CUtensorMap tm_kc, const __grid_constant__ CUtensorMap tm_vc,
                  const __grid_constant__ CUtensorMap tm_kt, const __grid_constant__ CUtensorMap tm_vt,
                  const __grid_constant__ CUtensorMap tm_op) {
  using C = Cfg<D>;
  constexpr int CPT = C::CPT, NS = C::NS;
  constexpr unsigned kAll = 0xffffffffu;
  extern __shared__ __align__(1024) uint8_t smem_raw[];

  // ---------------------------------------------------------------- smem
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem_raw);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem_raw + C::NBARS * 8);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  float* xch = reinterpret_cast<float*>(smem_raw + 256);        // [2 parity][2 half][128 rows]
  uint8_t* sQ = smem_raw + kHeader;
  uint8_t* ring = sQ + C::Q_BYTES;
  auto bar = [&](int i) { return smem_u32(&bars[i]); };
  auto FULL = [&](int i) { return bar(i); };
  auto EMPTY = [&](int i) { return bar(NS + i); };
  const int bq = 2 * NS;
  const uint32_t Q_FULL = bar(bq), TAIL = bar(bq + 7), FIN = bar(bq + 8), XL = bar(bq + 11);
  auto BOX = [&](int i) { return bar(bq + 12 + i); };     // epilogue box i staged (D / 32 boxes)
  auto S_FULL = [&](int i) { return bar(bq + 1 + i); };   // QK(t) done, buffer t & 1
  auto P_FULL = [&](int i) { return bar(bq + 3 + i); };   // softmax wrote P(t), buffer t & 1
  auto O_DONE = [&](int i) { return bar(bq + 5 + i); };   // PV(t) done, alternating by t & 1
  auto XCH = [&](int i) { return bar(bq + 9 + i); };      // row maxima exchanged for tile t, t & 1

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  // the layout below needs the dynamic shared window to start 1 KB aligned
  if (smem_u32(smem_raw) & 1023u) {
    dep_wait();
    if (tid == 0) set_status(p.status, TV_DEV_TIMEOUT);
    return;
  }
  // on-chip setup before the dependency wait: it overlaps the previous
  // kernel's tail when the launch is programmatic
  if (tid == 0) {
    for (int i = 0; i < NS; ++i) {
      mbar_init(FULL(i), 1);
      mbar_init(EMPTY(i), 1);
    }
    mbar_init(Q_FULL, 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(S_FULL(i), 1);
      mbar_init(P_FULL(i), kSoftmaxWarps);         // one arrive per softmax warp
      mbar_init(O_DONE(i), 1);
      mbar_init(XCH(i), kSoftmaxWarps);
    }
    mbar_init(TAIL, 1);
    mbar_init(FIN, 1);
    mbar_init(XL, kSoftmaxWarps);
    // box i: the 4 warps of one half, once per 32-column step it spans
    for (int i = 0; i < D / 32; ++i) mbar_init(BOX(i), (p.part_bf16 ? 2 : 1) * (kSoftmaxWarps / 2));
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (p.rows_per_tile < BM) {
    // pad rows of the query tile (G does not divide 128) hold zeros
    const int pad = BM - p.rows_per_tile;
    for (int e = tid; e < (D / 64) * pad * 8; e += blockDim.x) {
      const int kb = e / (pad * 8), r = p.rows_per_tile + (e / 8) % pad, c = e % 8;
      *reinterpret_cast<uint4*>(sQ + kb * (BM * 128) + r * 128 + c * 16) = make_uint4(0, 0, 0, 0);
    }
    fence_proxy_async_smem();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), 512);
    tmem_relinquish();
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
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  if (warp == 3) {
    // an idle warp warms L2 (and the TLB) for what the first steps read,
    // while the previous kernel may still run: the sequence's lengths, the
    // first kPrefetchTiles K and V tiles the chunk can hold (bounded by the
    // host's max_prefix, since the length itself is not read yet) and, for
    // the first sequence (rows start at 0), the query tile.  These are
    // hints: a prefetch has no effect on memory ordering, so a line the
    // previous kernel writes later is still read fresh, and a page id read
    // here only picks which lines to warm (a stale or invalid id costs a
    // wasted prefetch, never a wrong value).
    const int b = blockIdx.z, g = blockIdx.y / p.splits, s = blockIdx.y % p.splits;
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
      if (lane < npf && row + BN <= (int64_t)INT_MAX)
        for (int bx = 0; bx < D / 64; ++bx) {
          tma_prefetch_2d(&tm_kc, bx * 64, (int)row);
          tma_prefetch_2d(&tm_vc, bx * 64, (int)row);
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
          for (int bx = 0; bx < D / 64; ++bx) {
            tma_prefetch_2d(&tm_kc, bx * 64, row);
            tma_prefetch_2d(&tm_vc, bx * 64, row);
          }
        }
      }
    }
  }
  dep_wait();
  dep_launch();

  // ---------------------------------------------------------------- work
  const int rt = blockIdx.x;
  const int g = blockIdx.y / p.splits;
  const int s = blockIdx.y % p.splits;
  const int b = blockIdx.z;
  const int64_t Praw = p.prefix_len[b];            // read together with the offsets
  int o0 = 0, n = 1;
  bool active = seq_rows(p.node_offsets, b, p.R, p.max_nodes, p.status, &o0, &n);
  const int G = p.G;
  const int nrows = n * G;
  const int m0 = rt * p.rows_per_tile;
  active = active && m0 < nrows;
  const int64_t P = clamp_prefix(Praw, p.max_prefix, p.capacity);
  if (active && P != Praw && tid == 0 && rt == 0 && s == 0 && g == 0) set_status(p.status, TV_DEV_BAD_PREFIX);
  const int nch = num_chunks(P, p.chunk, p.tree_tile);
  active = active && s < nch;                      // uniform over the CTA
  const int64_t k_begin = (int64_t)s * p.chunk;
  const int64_t k_end = min(P, k_begin + p.chunk);
  const bool has_tree = (s == nch - 1);
  const int npt = (int)((k_end - k_begin + BN - 1) / BN);      // prefix tiles
  const int T = npt + (has_tree ? 1 : 0);
  const int tail_valid = npt > 0 ? (int)(k_end - (k_begin + (int64_t)(npt - 1) * BN)) : BN;

  if (!active) {
    // nothing to do for this CTA: straight to teardown
  } else if (warp == 0) {
    // ============================================================ producer
    if (lane == 0) {
      mbar_expect_tx(Q_FULL, (uint32_t)p.rows_per_tile * 128u * (D / 64));
      for (int kb = 0; kb < D / 64; ++kb)
        tma_load_3d(smem_u32(sQ + kb * (BM * 128)), &tm_q, Q_FULL, kb * 64, g * G, o0 + m0 / G);
    }
    int j = 0, tail_uses = 0;
    bool ok = true;
    // paged cache: lane i < 8 owns page i of a key tile; page ids are read
    // well ahead of the copies that use them
    const int oob_row = p.paged ? (int)(p.num_pages * p.Hkv * kPageSize) : 0;
    auto page_id = [&](int tile) -> int {           // raw page id of this lane's page, or INT_MIN (none)
      if (!p.paged || tile >= npt || lane >= BN / kPageSize) return INT_MIN;
      const int64_t pos = k_begin + (int64_t)tile * BN + lane * kPageSize;
      if (pos >= k_end) return INT_MIN;
      return p.page_table[(int64_t)b * p.max_pages + pos / kPageSize];
    };
    auto page_row = [&](int pid) -> int {           // TMA row of a page id, checked where it is used
      if (pid == INT_MIN) return -1;
      if (pid >= 0 && pid < p.num_pages) return (int)(((int64_t)pid * p.Hkv + g) * kPageSize);
      set_status(p.status, TV_DEV_BAD_PAGE);
      return oob_row;                               // out of range: the copy reads zeros
    };
    // page ids four tiles ahead (a read takes about a microsecond; nothing
    // branches on a value until it is used)
    int pid_a = page_id(0), pid_b = page_id(1), pid_c = page_id(2), pid_d = page_id(3);
    int row_k = -1, row_v = -1;
    for (int t = 0; t <= T && ok; ++t) {
      row_v = row_k;                                // tile t-1 (for V)
      row_k = page_row(pid_a);                      // tile t   (for K)
      pid_a = pid_b;
      pid_b = pid_c;
      pid_c = pid_d;
      pid_d = page_id(t + 4);
      for (int kind = 0; kind < 2 && ok; ++kind) {           // 0: K(t), 1: V(t-1)
        const int tile = kind == 0 ? t : t - 1;
        if ((kind == 0 && t >= T) || (kind == 1 && t < 1)) continue;
        const bool tree = (tile == npt);
        const bool tail_fix = (kind == 1) && !tree && tile == npt - 1 && tail_valid < BN;
        for (int c = 0; c < CPT && ok; ++c, ++j) {
          const int slot = j % NS, use = j / NS;
          if (use > 0 && !__all_sync(kAll, mbar_wait(EMPTY(slot), (use - 1) & 1, abort_flag, kWaitNs))) {
            ok = false;
            break;
          }
          uint8_t* dst = ring + slot * CHUNK_BYTES;
          const uint32_t fb = tail_fix ? TAIL : FULL(slot);
          if (tree || !p.paged) {
            if (lane == 0) {
              mbar_expect_tx(fb, CHUNK_BYTES);
              const CUtensorMap* m = tree ? (kind == 0 ? &tm_kt : &tm_vt) : (kind == 0 ? &tm_kc : &tm_vc);
              const int64_t row = tree ? (int64_t)g * p.R + o0
                                       : ((int64_t)b * p.Hkv + g) * p.capacity + k_begin + (int64_t)tile * BN;
              for (int bx = 0; bx < 2; ++bx)
                tma_load_2d(smem_u32(dst + bx * BOX_BYTES), m, fb, c * CH + bx * 64, (int)row);
            }
          } else {
            const CUtensorMap* m = kind == 0 ? &tm_kc : &tm_vc;
            const int my_row = kind == 0 ? row_k : row_v;
            const int npages = __popc(__ballot_sync(kAll, my_row >= 0));
            if (lane == 0) mbar_expect_tx(fb, (uint32_t)npages * 2u * (kPageSize * 128u));
            __syncwarp();
            if (my_row >= 0) {
              for (int bx = 0; bx < 2; ++bx)
                tma_load_2d(smem_u32(dst + bx * BOX_BYTES + lane * kPageSize * 128), m, fb, c * CH + bx * 64,
                            my_row);
            }
          }
          __syncwarp();
          if (tail_fix) {
            // the chunk's rows past the prefix end become zeros before the MMA reads them
            if (!__all_sync(kAll, mbar_wait(TAIL, tail_uses & 1, abort_flag, kWaitNs))) {
              ok = false;
              break;
            }
            ++tail_uses;
            const int nz = BN - tail_valid;
            for (int e = lane; e < 2 * nz * 8; e += 32) {
              const int bx = e / (nz * 8), r = tail_valid + (e / 8) % nz, q16 = e % 8;
              *reinterpret_cast<uint4*>(dst + bx * BOX_BYTES + r * 128 + q16 * 16) = make_uint4(0, 0, 0, 0);
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(FULL(slot));
          }
        }
      }
    }
    // drain: every copy this warp started has landed before the CTA exits
    if (lane == 0) {
      mbar_wait(Q_FULL, 0, abort_flag, kWaitNs);
      for (int jj = (j > NS ? j - NS : 0); jj < j; ++jj) mbar_wait(FULL(jj % NS), (jj / NS) & 1, abort_flag, kWaitNs);
    }
  } else if (warp == 1) {
    // ============================================================ MMA issuer
    if (lane == 0) {
      constexpr uint32_t ID_QK = idesc_bf16_f32(BM, BN, 0, 0);
      constexpr uint32_t ID_PV = idesc_bf16_f32(BM, CH, 0, 1);
      bool ok = mbar_wait(Q_FULL, 0, abort_flag, kWaitNs);
      tc_fence_after();
      const uint32_t q_addr = smem_u32(sQ);
      const uint32_t ring_addr = smem_u32(ring);
      int j = 0;
      for (int t = 0; t <= T && ok; ++t) {
        if (t < T) {
          const uint32_t sbuf = tmem + (uint32_t)((t & 1) * 128);
          for (int c = 0; c < CPT && ok; ++c, ++j) {
            const int slot = j % NS;
            if (!mbar_wait(FULL(slot), (j / NS) & 1, abort_flag, kWaitNs)) { ok = false; break; }
            tc_fence_after();
            const uint32_t kaddr = ring_addr + slot * CHUNK_BYTES;
#pragma unroll
            for (int kk = 0; kk < CH / 16; ++kk) {
              const int kg = c * (CH / 16) + kk;           // 16-column step over d
              const uint64_t a = smem_desc(q_addr + (kg >> 2) * (BM * 128) + (kg & 3) * 32, 16, 1024, 2);
              const uint64_t bd = smem_desc(kaddr + (kk >> 2) * BOX_BYTES + (kk & 3) * 32, 16, 1024, 2);
              mma_ss(sbuf, a, bd, ID_QK, (c > 0 || kk > 0) ? 1u : 0u);
            }
            mma_commit(EMPTY(slot));
          }
          if (!ok) break;
          mma_commit(S_FULL(t & 1));
        }
        if (t >= 1) {
          const int u = t - 1;
          const uint32_t pbuf = tmem + (uint32_t)((u & 1) * 128);
          if (!mbar_wait(P_FULL(u & 1), (u >> 1) & 1, abort_flag, kWaitNs)) { ok = false; break; }
          tc_fence_after();
          for (int c = 0; c < CPT && ok; ++c, ++j) {
            const int slot = j % NS;
            if (!mbar_wait(FULL(slot), (j / NS) & 1, abort_flag, kWaitNs)) { ok = false; break; }
            tc_fence_after();
            const uint32_t vaddr = ring_addr + slot * CHUNK_BYTES;
#pragma unroll
            for (int kk = 0; kk < BN / 16; ++kk) {       // 16 keys per step
              const uint64_t bd = smem_desc(vaddr + kk * (16 * 128), BOX_BYTES, 1024, 2);
              mma_ts(tmem + 256 + c * CH, pbuf + kk * 8, bd, ID_PV, (u > 0 || kk > 0) ? 1u : 0u);
            }
            mma_commit(EMPTY(slot));
          }
          if (!ok) break;
          mma_commit(O_DONE(u & 1));
        }
      }
      // every MMA this thread issued has finished before tensor memory is freed
      mma_commit(FIN);
      mbar_wait(FIN, 0, abort_flag, kWaitNs);
    }
  } else if (warp == 2) {
    // ============================================================ partials store
    // one 128-byte-wide box of the partial tile at a time (32 fp32 or 64 bf16
    // columns), as soon as the softmax warps of its half have staged it;
    // every box barrier is arrived in all paths, so the waits here end
    if (lane == 0) {
      const bool store = !(p.out != nullptr && nch == 1);
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
    // ============================================================ softmax
    // Two warpgroups: `half` 0 takes keys 0-63 of every tile (and O columns
    // [0, D/2)), half 1 keys 64-127 (and O columns [D/2, D)); the two threads
    // of a row share its running maximum through `xch`.  Every tcgen05.ld /
    // st is warp-collective (.sync.aligned): control flow around them stays
    // warp-uniform and per-row choices only pick values.
    const int half = (tid - 128) >> 7;
    const int r = (tid - 128) & 127;                        // row in the tile == TMEM lane
    const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
    const bool row_ok = r < p.rows_per_tile && (m0 + r) < nrows;
    const int node = (m0 + r) / G;
    const uint64_t anc = row_ok ? p.anc[o0 + node] : 0ull;
    const float c2 = p.scale_log2;
    const int kofs = half * (BN / 2);                       // first key of this half
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
        // tree tile: ancestor bits; last prefix tile: key range
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
      // exchange the half-row maximum with the other half
      float* xb = xch + (t & 1) * 256;
      xb[half * 128 + r] = mx;
      __syncwarp();
      if (lane == 0) mbar_arrive(XCH(t & 1));
      if (!__all_sync(kAll, mbar_wait(XCH(t & 1), (t >> 1) & 1, abort_flag, kWaitNs))) { ok = false; break; }
      mx = fmaxf(mx, xb[(half ^ 1) * 128 + r]);
      const float m_tile = mx == -INFINITY ? -INFINITY : mx * c2;
      const float m_new = fmaxf(m_ref, m_tile);
      const bool first = (m_ref == -INFINITY);              // nothing accumulated yet
      const bool need = !first && (m_new > m_ref + kRescaleThreshold);
      if (__any_sync(kAll, need)) {
        // the O rows must hold P(t-1) V(t-1) before they are rescaled (t >= 1 here)
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
      const float nm = m_ref == -INFINITY ? 0.f : -m_ref;   // masked keys: 2^-inf = 0
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
      tmem_st_x32(sbuf + half * 32, pk);                   // P over the S columns, bf16 pairs
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(P_FULL(t & 1));
    }
    // epilogue: the last P V has landed (its commit covers every earlier
    // MMA); add the two halves' sums.  A sequence with one chunk writes its
    // normalised rows directly (the merge's arithmetic for one split).
    // Otherwise the partial O_s / l_s (fp32, or bf16 with a bf16 output) is
    // staged in the ring (idle now; 128-byte swizzled boxes), each box's
    // barrier arrived as soon as it is written (in every path, so warp 2's
    // waits always end), and warp 2 stores the boxes into this CTA's tile.
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
        if (epi && got && direct && row_ok) {
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
        } else if (epi && got && !direct) {
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
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(BOX(p.part_bf16 ? half * (D / 128) + qq : half * (D / 64) + q));
      }
    }
    if (epi && got && !direct)
      p.ml_part[partial_slot(s, b, g, rt, r, p.Hkv, p.row_tiles, BM, p.splits)] = make_float2(row_ok ? m_ref : -INFINITY, row_ok ? lsum : 0.f);
  }

  // ---------------------------------------------------------------- teardown
  tc_fence_before();
  __syncthreads();
  if (tid == 0 && *abort_flag) set_status(p.status, TV_DEV_TIMEOUT);
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// ---------------------------------------------------------------- host

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
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

bool encode(CUtensorMap* m, const void* ptr, int rank, const cuuint64_t* dims, const cuuint64_t* strides,
            const cuuint32_t* box, CUtensorMapDataType type = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  cuuint32_t es[3] = {1, 1, 1};
  return fn(m, type, rank, const_cast<void*>(ptr), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int D>
cudaError_t launch_tc_t(const AttnParams& p, cudaStream_t st) {
  CUtensorMap mq, mkc, mvc, mkt, mvt;
  const cuuint64_t row_bytes = (cuuint64_t)D * 2;
  {
    cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)p.Hq, (cuuint64_t)p.R};
    cuuint64_t strides[2] = {row_bytes, row_bytes * p.Hq};
    cuuint32_t box[3] = {64, (cuuint32_t)p.G, (cuuint32_t)(BM / p.G)};
    if (!encode(&mq, p.q, 3, dims, strides, box)) return cudaErrorInvalidValue;
  }
  {
    const cuuint64_t rows = p.paged ? (cuuint64_t)p.num_pages * p.Hkv * kPageSize
                                    : (cuuint64_t)p.B * p.Hkv * p.capacity;
    cuuint64_t dims[2] = {(cuuint64_t)D, rows};
    cuuint64_t strides[1] = {row_bytes};
    cuuint32_t box[2] = {64, (cuuint32_t)(p.paged ? kPageSize : BN)};
    if (!encode(&mkc, p.k_cache, 2, dims, strides, box) || !encode(&mvc, p.v_cache, 2, dims, strides, box))
      return cudaErrorInvalidValue;
  }
  {
    cuuint64_t dims[2] = {(cuuint64_t)D, (cuuint64_t)p.Hkv * p.R};
    cuuint64_t strides[1] = {row_bytes};
    cuuint32_t box[2] = {64, BN};
    if (!encode(&mkt, p.k_tree, 2, dims, strides, box) || !encode(&mvt, p.v_tree, 2, dims, strides, box))
      return cudaErrorInvalidValue;
  }
  CUtensorMap mop;
  {
    // partials [rows][splits][D] (partial_slot), fp32 (boxes of 32 columns)
    // or bf16 (64); a CTA stores one split of a 128-row tile
    const cuuint64_t es = p.part_bf16 ? 2 : 4;
    const cuuint64_t rows = (cuuint64_t)p.B * p.Hkv * p.row_tiles * BM;
    cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)p.splits, rows};
    cuuint64_t strides[2] = {(cuuint64_t)D * es, (cuuint64_t)D * es * p.splits};
    cuuint32_t box[3] = {p.part_bf16 ? 64u : 32u, 1u, BM};
    if (!encode(&mop, p.o_part, 3, dims, strides, box,
                p.part_bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32))
      return cudaErrorInvalidValue;
  }
  cudaError_t e = ensure_max_dynamic_smem<tv_attn_tc_kernel<D>>((int)Cfg<D>::SMEM);
  if (e != cudaSuccess) return e;
  dim3 grid(p.row_tiles, p.Hkv * p.splits, p.B);
  return launch_dep(tv_attn_tc_kernel<D>, grid, dim3(kThreads), Cfg<D>::SMEM, st, p, mq, mkc, mvc, mkt, mvt, mop);
}

}  // namespace

bool tc_supported(const tv_desc* d, int G) {
  if (d->dtype != TV_BF16 || (d->head_dim != 128 && d->head_dim != 256)) return false;
  if (G < 1 || G > BM) return false;
  // TMA coordinates are int32: every row index must fit
  const int64_t lim = ((int64_t)1 << 31) - 1;
  const int64_t cache_rows = d->page_size ? d->num_pages * d->num_kv_heads * kPageSize
                                          : (int64_t)d->batch * d->num_kv_heads * d->capacity;
  if (cache_rows + BN > lim || (int64_t)d->num_kv_heads * d->total_rows + BN > lim) return false;
  return true;
}

int tc_key_tile(int) { return BN; }

cudaError_t launch_attn_tc(const AttnParams& p, cudaStream_t s) {
  if (p.d == 128) return launch_tc_t<128>(p, s);
  return launch_tc_t<256>(p, s);
}

}  // namespace tv
