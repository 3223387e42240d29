// tcgen05 split-KV tree-verify attention for batches of sequences (bf16
// Q/K/V, head_dim 128, bf16 output): persistent CTA pairs, one CTA per SM.
//
// The arithmetic is the one-CTA kernel's (flash-decode with a tree mask,
// "ADR-037 — EAGLE-3 with dynamic tree port", phase rows E1.1-E1.5 and
// E4b.6, the dk128 retrofit): a work unit is (sequence b, KV head g, a pair
// of query row tiles, key chunk s); CTA r of a two-CTA cluster computes row
// tile 2 p + r of the pair p.  The unit's keys are the chunk's prefix
// positions in 128-key tiles and, in the sequence's last chunk, one tile of
// tree keys masked by each row's ancestor bits; each row tile leaves a
// normalised partial O_s / l_s (bf16) with its running maximum and sum for
// the merge, or the final rows when the sequence has one chunk.
//
// The two CTAs of a pair read the same K/V tiles, so each loads half of
// every tile (its pages, or its 64 keys) with TMA multicast into both CTAs'
// shared memory: L2 serves each K/V byte once per unit, and each SM issues
// half of a paged tile's sixteen 16-row boxes.  A tree whose rows fill one
// tile leaves the second CTA's rows empty; it still takes its half of the
// loads.
//
// In a batch the sequences have different prefix lengths and tree sizes, so
// a grid of one CTA per unit runs in uneven waves and pays the CTA's setup
// (barriers, tensor memory, the first tiles' latency, the epilogue's drain)
// once per unit.  Here each CTA sets up once and takes units from a work
// counter in the workspace until none is left; units are numbered
// chunk-major (every sequence's first chunk first), so the long full chunks
// go out before the short last ones.  Units with no rows or no keys are
// skipped by the scheduler, never queued.
//
//   warp 0      TMA producer: per unit its Q tile, then 32 KB K/V chunks
//               through a ring of slots in MMA order K(0), K(1), V(0),
//               K(2), V(1), ... (sixteen 16-row boxes per chunk on a paged
//               cache).
//   warp 1      owns tensor memory; lane 0 issues the MMAs: S(t) = Q K(t)^T
//               into one of two 128-column buffers, then for each key half h
//               O_h += P(t)[:, half h] V(t)[half h, :] into that half's own
//               O accumulator (TMEM columns 256 + 128 h), as soon as that
//               half's softmax warps have written their P.
//   warp 2      scheduler (lane 0 of the pair's first CTA): takes unit
//               numbers from the counter, decodes them (lengths, offsets,
//               chunk bounds) and hands them through a two-entry queue in
//               both CTAs' shared memory to the other roles of both.
//   warps 3-10  softmax (two threads per query row, each half of a tile's
//               keys with its own running maximum, sum and O accumulator, so
//               the two never wait for each other inside a unit), then each
//               unit's epilogue: the row's two threads exchange their
//               maxima and sums once, combine the two accumulators and write
//               the partial rows straight from registers.
// Barrier phases run on across units: slots by a slot counter, the S / P
// buffers and O products by a tile counter, the epilogue's exchanges by an
// exchange counter, per-unit barriers by a unit counter.  Every wait is bounded
// (1 s); on a timeout the CTA raises TV_DEV_TIMEOUT and every role leaves
// its loop.
//
// Slots are released to the producers when both CTAs' products are done
// with them (each MMA thread's commit arrives on EMPTY in both CTAs), and the
// pair meets at an execution-only cluster barrier before it exits, once no
// copy, commit or queue release of either CTA is still on its way.
//
// The work counter needs no zeroing: it is a tagged word (launch_tag,
// arm_counter), raised to this launch's tag by every pair before it takes
// numbers with atomic adds.
#include <cuda.h>

#include <climits>
#include <mutex>

#include "tc_ptx.cuh"
#include "tv_internal.cuh"

namespace tv {
namespace {

using namespace tc;

constexpr int D = 128;
constexpr int BM = 128;                         // query rows per tile
constexpr int BN = 128;                         // keys per tile
constexpr uint32_t BOX_BYTES = BN * 128;        // one TMA box: 128 rows x 64 bf16
constexpr uint32_t SLOT_BYTES = 2 * BOX_BYTES;  // 128 keys x 128 columns
constexpr int NS = 6;                           // ring slots
constexpr uint32_t kHeader = 3072;              // barriers, TMEM address, exchanges, unit queue
constexpr uint32_t Q_BYTES = BM * D * 2;
constexpr uint32_t SMEM = kHeader + Q_BYTES + NS * SLOT_BYTES;
static_assert(SMEM <= 232448, "shared memory over the 227 KB per-block limit");
constexpr int kThreads = 352;
constexpr int kFirstSoftmaxWarp = 3;
constexpr int kSoftmaxWarps = 8;
constexpr uint64_t kWaitNs = 1000000000ull;
constexpr float kRescaleThreshold = 8.0f;       // rescale O when the max grows by > 2^8
constexpr int kUnitSlots = 2;                   // the unit queue
constexpr int kUnitReaders = 2 * (2 + kSoftmaxWarps);   // both CTAs' producer, MMA lane, softmax warps
constexpr int KH = BN / 2;                      // keys of a tile each CTA of the pair loads

// barrier numbers
constexpr int B_FULL = 0, B_EMPTY = NS, B_QFULL = 2 * NS, B_QEMPTY = B_QFULL + 1, B_SFULL = B_QEMPTY + 1,
              B_PFULL = B_SFULL + 2, B_ODONE = B_PFULL + 4, B_XCH = B_ODONE + 4, B_TAIL = B_XCH + 8,
              B_FIN = B_TAIL + 2, B_UFULL = B_FIN + 1, B_UEMPTY = B_UFULL + kUnitSlots,
              NBARS = B_UEMPTY + kUnitSlots;
static_assert(NBARS * 8 + 8 <= 384, "barriers overflow the header");

struct UnitInfo {
  int32_t valid;           // 0: no more units
  int32_t b, g, rt, s;
  int32_t o0, n, nch;      // the sequence's first row, node count, chunk count
  int32_t npt, T, tail_valid, pad;
  int64_t k_begin, k_end;  // the chunk's prefix keys
};
static_assert(sizeof(UnitInfo) == 64, "unit queue entry");
constexpr uint32_t kXchOfs = 384;               // [2 parity][2 half][128 rows] floats
constexpr uint32_t kQueueOfs = kXchOfs + 2048;
static_assert(kQueueOfs + kUnitSlots * sizeof(UnitInfo) <= kHeader, "unit queue overflows the header");

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ uint32_t pack_bf16(float a, float b) {
  __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&h);
}

// Packed fp32 pairs (f32x2 arithmetic: one instruction for two lanes of
// work on the FMA pipes).
__device__ __forceinline__ uint64_t pk2(float a, float b) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
  return r;
}
__device__ __forceinline__ float2 up2(uint64_t v) {
  float2 r;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(r.x), "=f"(r.y) : "l"(v));
  return r;
}
__device__ __forceinline__ uint64_t ffma2(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ uint64_t fadd2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

__host__ __device__ __forceinline__ int row_pairs(int row_tiles) { return (row_tiles + 1) / 2; }

// Unit u (chunk-major numbering; row tiles in pairs) with everything the
// roles need (rt is the pair's first row tile); false when it has no rows
// (tiles past the tree's rows, invalid offsets) or no keys (chunk past the
// sequence's prefix).  (Unit numbers stay below 2^24, which the host
// checks, so 32-bit arithmetic decodes them.)
__device__ bool decode_unit(const AttnParams& p, int u, UnitInfo& ui) {
  const int rp = row_pairs(p.row_tiles);
  const int per_s = p.B * p.Hkv * rp;
  const int s = u / per_s;
  const int rem = u - s * per_s;
  const int b = rem / (p.Hkv * rp);
  const int g = (rem / rp) % p.Hkv;
  const int rt = 2 * (rem % rp);
  int o0 = 0, n = 1;
  if (!seq_rows(p.node_offsets, b, p.R, p.max_nodes, p.status, &o0, &n)) return false;
  if (rt * p.rows_per_tile >= n * p.G) return false;
  const int64_t Praw = p.prefix_len[b];
  const int64_t P = clamp_prefix(Praw, p.max_prefix, p.capacity);
  if (P != Praw && rt == 0 && s == 0 && g == 0) set_status(p.status, TV_DEV_BAD_PREFIX);
  const int nch = num_chunks(P, p.chunk, p.tree_tile);
  if (s >= nch) return false;
  ui.valid = 1;
  ui.b = b;
  ui.g = g;
  ui.rt = rt;
  ui.s = s;
  ui.o0 = o0;
  ui.n = n;
  ui.nch = nch;
  ui.k_begin = (int64_t)s * p.chunk;
  ui.k_end = min(P, ui.k_begin + p.chunk);
  ui.npt = (int)((ui.k_end - ui.k_begin + BN - 1) / BN);
  ui.T = ui.npt + (s == nch - 1 ? 1 : 0);
  ui.tail_valid = ui.npt > 0 ? (int)(ui.k_end - (ui.k_begin + (int64_t)(ui.npt - 1) * BN)) : BN;
  ui.pad = 0;
  return true;
}

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
tv_attn_tcp_kernel(const __grid_constant__ AttnParams p, const __grid_constant__ CUtensorMap tm_q,
                   const __grid_constant__ CUtensorMap tm_kc, const __grid_constant__ CUtensorMap tm_vc,
                   const __grid_constant__ CUtensorMap tm_kt, const __grid_constant__ CUtensorMap tm_vt) {
  constexpr unsigned kAll = 0xffffffffu;
  extern __shared__ __align__(1024) uint8_t smem_raw[];

  // ---------------------------------------------------------------- smem
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem_raw);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem_raw + NBARS * 8);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  float* xch = reinterpret_cast<float*>(smem_raw + kXchOfs);
  UnitInfo* uqueue = reinterpret_cast<UnitInfo*>(smem_raw + kQueueOfs);
  uint8_t* sQ = smem_raw + kHeader;
  uint8_t* ring = sQ + Q_BYTES;
  auto bar = [&](int i) { return smem_u32(&bars[i]); };
  auto FULL = [&](int i) { return bar(B_FULL + i); };
  auto EMPTY = [&](int i) { return bar(B_EMPTY + i); };
  const uint32_t Q_FULL = bar(B_QFULL), Q_EMPTY = bar(B_QEMPTY), FIN = bar(B_FIN);
  auto TAIL = [&](int i) { return bar(B_TAIL + i); };
  auto S_FULL = [&](int i) { return bar(B_SFULL + i); };
  auto P_FULL = [&](int h, int i) { return bar(B_PFULL + 2 * h + i); };   // key half h, parity i
  auto O_DONE = [&](int h, int i) { return bar(B_ODONE + 2 * h + i); };
  auto XCH = [&](int q, int i) { return bar(B_XCH + 2 * q + i); };   // row quarter q, parity i
  auto UFULL = [&](int i) { return bar(B_UFULL + i); };
  auto UEMPTY = [&](int i) { return bar(B_UEMPTY + i); };

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (smem_u32(smem_raw) & 1023u) {                 // the layout needs a 1 KB aligned window
    dep_wait();
    if (tid == 0) set_status(p.status, TV_DEV_TIMEOUT);
    return;
  }
  // on-chip setup before the dependency wait (overlaps the previous kernel's tail)
  if (tid == 0) {
    for (int i = 0; i < NS; ++i) {
      mbar_init(FULL(i), 1);
      mbar_init(EMPTY(i), 2);                       // both CTAs' MMAs are done with the slot
    }
    mbar_init(Q_FULL, 1);
    mbar_init(Q_EMPTY, 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(S_FULL(i), 1);
      for (int h = 0; h < 2; ++h) {
        mbar_init(P_FULL(h, i), kSoftmaxWarps / 2);   // the warps of key half h
        mbar_init(O_DONE(h, i), 1);
      }
      for (int q = 0; q < 4; ++q) mbar_init(XCH(q, i), 2);   // the row quarter's two warps
    }
    mbar_init(TAIL(0), 1);
    mbar_init(TAIL(1), 1);
    mbar_init(FIN, 2);                              // both CTAs' MMA issuers are done
    for (int i = 0; i < kUnitSlots; ++i) {
      mbar_init(UFULL(i), 1);
      mbar_init(UEMPTY(i), kUnitReaders);
    }
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (p.rows_per_tile < BM) {
    // pad rows of the query tile (G does not divide 128) hold zeros; the Q
    // loads never write them
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
  cluster_sync_all();                               // the peer's barriers are ready before any remote arrive
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  dep_wait();
  dep_launch();

  const int G = p.G;
  const uint32_t rank = cluster_ctarank();          // 0: the pair's first CTA
  constexpr uint16_t kPair = 3;                     // multicast to both CTAs
  // a queue entry is handed back to the scheduler (in CTA 0) once read
  auto release_entry = [&](int kq) {
    if (rank == 0) mbar_arrive(UEMPTY(kq));
    else mbar_arrive_cluster_release(map_to_cta(UEMPTY(kq), 0));
  };
  if (warp == 2 && lane == 0 && rank == 0) {
    // ============================================================ scheduler
    const int U = p.splits * p.B * p.Hkv * row_pairs(p.row_tiles);
    const int pairs = (int)(gridDim.x / 2);
    const unsigned long long tag = launch_tag();
    arm_counter(p.work_counter, tag);
    auto next = [&]() -> int { return pairs + (int)(atomicAdd(p.work_counter, 1ull) & 0xFFFFFFull); };
    int u = (int)(blockIdx.x / 2);
    int k = 0, pushes = 0;
    while (true) {
      UnitInfo ui;
      ui.valid = 0;
      while (u < U && !decode_unit(p, u, ui)) u = next();
      if (pushes >= kUnitSlots &&
          !mbar_wait_cluster(UEMPTY(k), ((pushes / kUnitSlots) - 1) & 1, abort_flag, kWaitNs))
        break;                                      // aborted: every role leaves on the flag
      // the entry, word by word, into this CTA's queue and the peer's
      const uint32_t qa = smem_u32(uqueue + k), qr = map_to_cta(qa, 1);
      const uint32_t words[16] = {(uint32_t)ui.valid, (uint32_t)ui.b, (uint32_t)ui.g, (uint32_t)ui.rt,
                                  (uint32_t)ui.s, (uint32_t)ui.o0, (uint32_t)ui.n, (uint32_t)ui.nch,
                                  (uint32_t)ui.npt, (uint32_t)ui.T, (uint32_t)ui.tail_valid, 0u,
                                  (uint32_t)ui.k_begin, (uint32_t)((uint64_t)ui.k_begin >> 32),
                                  (uint32_t)ui.k_end, (uint32_t)((uint64_t)ui.k_end >> 32)};
      volatile uint32_t* ql = reinterpret_cast<volatile uint32_t*>(uqueue + k);
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        ql[i] = words[i];
        st_cluster_u32(qr + 4 * i, words[i]);
      }
      mbar_arrive(UFULL(k));
      mbar_arrive_cluster_release(map_to_cta(UFULL(k), 1));
      ++pushes;
      k ^= 1;
      if (!ui.valid) {
        // the last real entry's releases (some remote) land before this CTA
        // may leave; the entry before it was waited for to push this one
        if (pushes >= 2) mbar_wait_cluster(UEMPTY(k), ((pushes - 2) / kUnitSlots) & 1, abort_flag, kWaitNs);
        break;
      }
      u = next();
    }
  } else if (warp == 0) {
    // ============================================================ producer
    int j = 0, tail_uses = 0, uq = 0, k = 0;
    bool ok = true;
    const int oob_row = p.paged ? (int)(p.num_pages * p.Hkv * kPageSize) : 0;
    while (ok) {
      if (!__all_sync(kAll, mbar_wait_cluster(UFULL(k), (uq / kUnitSlots) & 1, abort_flag, kWaitNs))) break;
      const volatile UnitInfo* qe = reinterpret_cast<const volatile UnitInfo*>(uqueue + k);
      if (!qe->valid) break;                     // the last entry: nobody waits for its release
      const int b = qe->b, g = qe->g, npt = qe->npt, T = qe->T, tail_valid = qe->tail_valid, o0 = qe->o0;
      const int q_node = o0 + (qe->rt + (int)rank) * p.rows_per_tile / G;   // this CTA's Q tile's first node
      const int64_t k_begin = qe->k_begin, k_end = qe->k_end;
      // The unit's Q tile replaces the previous unit's once that unit's QK
      // products are done (Q_EMPTY).  It is loaded just before the unit's
      // first V chunk: its first K chunks go into the ring before, so they
      // stream in while the previous unit finishes.
      bool q_loaded = false;
      auto load_q = [&]() -> bool {
        if (uq > 0 && !__all_sync(kAll, mbar_wait(Q_EMPTY, (uq - 1) & 1, abort_flag, kWaitNs))) return false;
        if (lane == 0) {
          mbar_expect_tx(Q_FULL, (uint32_t)p.rows_per_tile * 128u * (D / 64));
          for (int kb = 0; kb < D / 64; ++kb)
            tma_load_3d(smem_u32(sQ + kb * (BM * 128)), &tm_q, Q_FULL, kb * 64, g * G, q_node);
        }
        q_loaded = true;
        return true;
      };
      auto page_id = [&](int tile) -> int {         // raw page id of this lane's page, or INT_MIN (none)
        if (!p.paged || tile >= npt || lane >= BN / kPageSize) return INT_MIN;
        const int64_t pos = k_begin + (int64_t)tile * BN + lane * kPageSize;
        if (pos >= k_end) return INT_MIN;
        return p.page_table[(int64_t)b * p.max_pages + pos / kPageSize];
      };
      auto page_row = [&](int pid) -> int {         // TMA row of a page id, checked where it is used
        if (pid == INT_MIN) return -1;
        if (pid >= 0 && pid < p.num_pages) return (int)(((int64_t)pid * p.Hkv + g) * kPageSize);
        set_status(p.status, TV_DEV_BAD_PAGE);
        return oob_row;                             // out of range: the copy reads zeros
      };
      int pid_a = page_id(0), pid_b = page_id(1), pid_c = page_id(2), pid_d = page_id(3);
      int row_k = -1, row_v = -1;
      for (int t = 0; t <= T && ok; ++t) {
        row_v = row_k;                              // tile t - 1
        row_k = page_row(pid_a);
        pid_a = pid_b;
        pid_b = pid_c;
        pid_c = pid_d;
        pid_d = page_id(t + 4);
        for (int kind = 0; kind < 2 && ok; ++kind) {         // 0: K(t), 1: V(t-1)
          const int tile = kind == 0 ? t : t - 1;
          if ((kind == 0 && t >= T) || (kind == 1 && t < 1)) continue;
          if (kind == 1 && !q_loaded && !load_q()) {
            ok = false;
            break;
          }
          const bool tree = (tile == npt);
          const bool tail_fix = (kind == 1) && !tree && tile == npt - 1 && tail_valid < BN;
          const int slot = j % NS, use = j / NS;
          if (use > 0 && !__all_sync(kAll, mbar_wait(EMPTY(slot), (use - 1) & 1, abort_flag, kWaitNs))) {
            ok = false;
            break;
          }
          // Each CTA loads half of the tile into both CTAs' slots: keys
          // 64 r .. 64 r + 63 (pages 4 r .. 4 r + 3 on a paged cache).  The
          // slot's barrier expects the whole tile's bytes; the peer's half
          // may land before this thread's expect_tx, which the transaction
          // count allows within a phase.
          uint8_t* dst = ring + slot * SLOT_BYTES;
          const uint32_t fb = tail_fix ? TAIL(tail_uses & 1) : FULL(slot);
          if (tree || !p.paged) {
            if (lane == 0) {
              mbar_expect_tx(fb, SLOT_BYTES);
              const CUtensorMap* m = tree ? (kind == 0 ? &tm_kt : &tm_vt) : (kind == 0 ? &tm_kc : &tm_vc);
              const int64_t row = (tree ? (int64_t)g * p.R + o0
                                        : ((int64_t)b * p.Hkv + g) * p.capacity + k_begin + (int64_t)tile * BN) +
                                  KH * rank;
              for (int bx = 0; bx < 2; ++bx)
                tma_load_2d_mc(smem_u32(dst + bx * BOX_BYTES + KH * rank * 128), m, fb, bx * 64, (int)row, kPair);
            }
          } else {
            const CUtensorMap* m = kind == 0 ? &tm_kc : &tm_vc;
            const int my_row = kind == 0 ? row_k : row_v;
            const int npages = __popc(__ballot_sync(kAll, my_row >= 0));
            if (lane == 0) mbar_expect_tx(fb, (uint32_t)npages * 2u * (kPageSize * 128u));
            __syncwarp();
            if (my_row >= 0 && (lane >> 2) == (int)rank)
              for (int bx = 0; bx < 2; ++bx)
                tma_load_2d_mc(smem_u32(dst + bx * BOX_BYTES + lane * kPageSize * 128), m, fb, bx * 64, my_row,
                               kPair);
          }
          __syncwarp();
          if (tail_fix) {
            // the chunk's rows past the prefix end become zeros before the
            // MMA reads them (both halves have landed: the TAIL phase counts
            // the whole tile).  Two TAIL barriers alternate: the peer cannot
            // start a second tail tile before this CTA has passed the first.
            if (!__all_sync(kAll, mbar_wait(TAIL(tail_uses & 1), (tail_uses >> 1) & 1, abort_flag, kWaitNs))) {
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
          ++j;
        }
      }
      __syncwarp();
      if (lane == 0) release_entry(k);             // done with the queue entry
      k ^= 1;
      ++uq;
    }
    // drain: every copy this warp started has landed before the CTA exits
    if (lane == 0) {
      if (uq > 0) mbar_wait(Q_FULL, (uq - 1) & 1, abort_flag, kWaitNs);
      for (int jj = (j > NS ? j - NS : 0); jj < j; ++jj) mbar_wait(FULL(jj % NS), (jj / NS) & 1, abort_flag, kWaitNs);
    }
  } else if (warp == 1) {
    // ============================================================ MMA issuer
    if (lane == 0) {
      constexpr uint32_t ID_QK = idesc_bf16_f32(BM, BN, 0, 0);
      constexpr uint32_t ID_PV = idesc_bf16_f32(BM, D, 0, 1);
      const uint32_t q_addr = smem_u32(sQ);
      const uint32_t ring_addr = smem_u32(ring);
      int j = 0, tt = 0, uq = 0, k = 0;
      bool ok = true;
      while (ok) {
        if (!mbar_wait_cluster(UFULL(k), (uq / kUnitSlots) & 1, abort_flag, kWaitNs)) break;
        const int T = reinterpret_cast<const volatile UnitInfo*>(uqueue + k)->valid
                          ? reinterpret_cast<const volatile UnitInfo*>(uqueue + k)->T
                          : 0;
        if (T == 0) break;                          // the last entry: nobody waits for its release
        release_entry(k);                           // only T is needed, and it is read
        k ^= 1;
        if (!mbar_wait(Q_FULL, uq & 1, abort_flag, kWaitNs)) break;
        tc_fence_after();
        for (int t = 0; t <= T && ok; ++t) {
          if (t < T) {
            const int tg = tt + t;
            const uint32_t sbuf = tmem + (uint32_t)((tg & 1) * 128);
            const int slot = j % NS;
            if (!mbar_wait(FULL(slot), (j / NS) & 1, abort_flag, kWaitNs)) { ok = false; break; }
            tc_fence_after();
            const uint32_t kaddr = ring_addr + slot * SLOT_BYTES;
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {   // 16-column steps over d
              const uint64_t a = smem_desc(q_addr + (kk >> 2) * (BM * 128) + (kk & 3) * 32, 16, 1024, 2);
              const uint64_t bd = smem_desc(kaddr + (kk >> 2) * BOX_BYTES + (kk & 3) * 32, 16, 1024, 2);
              mma_ss(sbuf, a, bd, ID_QK, kk > 0 ? 1u : 0u);
            }
            mma_commit_mc(EMPTY(slot), kPair);
            mma_commit(S_FULL(tg & 1));
            if (t == T - 1) mma_commit(Q_EMPTY);    // the unit's last product that reads Q
            ++j;
          }
          if (t >= 1) {
            // O_h += P(:, keys of half h) V(keys of half h, :): each key half
            // of the softmax keeps its own accumulator, maximum and sum, so
            // the halves never wait for each other inside a unit
            const int u = t - 1, ug = tt + u;
            const uint32_t pbuf = tmem + (uint32_t)((ug & 1) * 128);
            const int slot = j % NS;
            if (!mbar_wait(FULL(slot), (j / NS) & 1, abort_flag, kWaitNs)) { ok = false; break; }
            tc_fence_after();
            const uint32_t vaddr = ring_addr + slot * SLOT_BYTES;
            for (int h = 0; h < 2 && ok; ++h) {
              if (!mbar_wait(P_FULL(h, ug & 1), (ug >> 1) & 1, abort_flag, kWaitNs)) { ok = false; break; }
              tc_fence_after();
#pragma unroll
              for (int kq = 0; kq < BN / 32; ++kq) {  // 16 keys per step, 4 steps per half
                const int kk = h * (BN / 32) + kq;
                const uint64_t bd = smem_desc(vaddr + kk * (16 * 128), BOX_BYTES, 1024, 2);
                mma_ts(tmem + 256 + (uint32_t)(h * D), pbuf + kk * 8, bd, ID_PV, (u > 0 || kq > 0) ? 1u : 0u);
              }
              mma_commit(O_DONE(h, ug & 1));
            }
            if (!ok) break;
            mma_commit_mc(EMPTY(slot), kPair);
            ++j;
          }
        }
        tt += T;
        ++uq;
      }
      // every MMA this thread issued has finished before tensor memory is
      // freed, and (FIN being each issuer's last commit, to both CTAs) no
      // commit of either issuer is still on its way to this CTA's barriers
      mma_commit_mc(FIN, kPair);
      mbar_wait(FIN, 0, abort_flag, kWaitNs);
    }
  } else if (warp >= kFirstSoftmaxWarp) {
    // ============================================================ softmax
    // Two warpgroups: `half` 0 takes keys 0-63 of every tile, half 1 keys
    // 64-127.  Each half keeps its own running maximum, sum and O
    // accumulator (TMEM columns 256 + 128 half), so the two threads of a row
    // meet only at the unit's end, where their (maximum, sum) pairs are
    // exchanged through `xch` and the two accumulators combined.
    const int half = (warp - kFirstSoftmaxWarp) >> 2;
    const int r = (warp & 3) * 32 + lane;           // row in the tile == TMEM lane (warp % 4 picks the quarter)
    const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
    const float c2 = p.scale_log2;
    const int kofs = half * (BN / 2);
    const uint32_t obuf = tmem + lane_base + 256 + (uint32_t)(half * D);   // this half's O rows
    int tt = 0, xt = 0, uq = 0, k = 0;
    bool ok = true;
    // the row quarter's two warps exchange one float per row through xch
    auto exchange = [&](float mine, float& theirs) -> bool {
      float* xb = xch + (xt & 1) * 256;
      xb[half * 128 + r] = mine;
      __syncwarp();
      if (lane == 0) mbar_arrive(XCH(warp & 3, xt & 1));
      const bool in = __all_sync(kAll, mbar_wait(XCH(warp & 3, xt & 1), (xt >> 1) & 1, abort_flag, kWaitNs));
      ++xt;
      theirs = xb[(half ^ 1) * 128 + r];
      return in;
    };
    while (ok) {
      if (!__all_sync(kAll, mbar_wait_cluster(UFULL(k), (uq / kUnitSlots) & 1, abort_flag, kWaitNs))) break;
      // the entry stays valid until this warp arrives on UEMPTY at the end of
      // the unit: fields the epilogue needs are read there again (fewer live
      // registers through the tile loop)
      const volatile UnitInfo* qe = reinterpret_cast<const volatile UnitInfo*>(uqueue + k);
      if (!qe->valid) break;                     // the last entry: nobody waits for its release
      const int T = qe->T, npt = qe->npt, tail_valid = qe->tail_valid, n = qe->n;
      const int my_rt = qe->rt + (int)rank;         // this CTA's row tile of the pair
      bool row_ok;
      uint64_t anc;
      {
        const int m0 = my_rt * p.rows_per_tile;
        row_ok = r < p.rows_per_tile && (m0 + r) < n * G;
        anc = row_ok ? p.anc[qe->o0 + (m0 + r) / G] : 0ull;
      }
      float m_ref = -INFINITY, l = 0.f;
      const bool warp_live = __any_sync(kAll, row_ok);
      for (int t = 0; t < T && ok; ++t) {
        const int tg = tt + t;
        if (!__all_sync(kAll, mbar_wait(S_FULL(tg & 1), (tg >> 1) & 1, abort_flag, kWaitNs))) { ok = false; break; }
        tc_fence_after();
        const uint32_t sbuf = tmem + lane_base + (uint32_t)((tg & 1) * 128);
        // a warp whose 32 rows all lie past the tree's rows leaves P as it is:
        // the products of those rows are never read
        if (warp_live) {
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
          float mq[4] = {sv[0], sv[1], sv[2], sv[3]};
  #pragma unroll
          for (int e = 4; e < 64; e += 2) mq[(e >> 1) & 3] = fmax3(mq[(e >> 1) & 3], sv[e], sv[e + 1]);
          const float mx = fmax3(mq[0], mq[1], fmaxf(mq[2], mq[3]));
          const float m_tile = mx == -INFINITY ? -INFINITY : mx * c2;
          const float m_new = fmaxf(m_ref, m_tile);
          const bool first = (m_ref == -INFINITY);
          const bool need = !first && (m_new > m_ref + kRescaleThreshold);
          if (__any_sync(kAll, need)) {
            // this half's O rows must hold P(t-1) V(t-1) before they are rescaled (t >= 1 here)
            const int ug = tg - 1;
            if (!__all_sync(kAll, mbar_wait(O_DONE(half, ug & 1), (ug >> 1) & 1, abort_flag, kWaitNs))) {
              ok = false;
              break;
            }
            tc_fence_after();
            const float alpha = need ? ex2(m_ref - m_new) : 1.f;
  #pragma unroll 1
            for (int c = 0; c < D; c += 32) {
              uint32_t rr[32];
              tmem_ld_x32(obuf + c, rr);
  #pragma unroll
              for (int e = 0; e < 32; ++e) rr[e] = __float_as_uint(__uint_as_float(rr[e]) * alpha);
              tmem_st_x32(obuf + c, rr);
            }
            if (need) {
              l *= alpha;
              m_ref = m_new;
            }
          }
          if (first) m_ref = m_new;
          const float nm = m_ref == -INFINITY ? 0.f : -m_ref;   // masked keys: 2^-inf = 0
          // P = 2^(s c2 - m) in packed pairs (f32x2 products and sums)
          const uint64_t c2x2 = pk2(c2, c2), nmx2 = pk2(nm, nm);
          uint64_t l4[4] = {0ull, 0ull, 0ull, 0ull};   // packed (+0, +0)
          uint32_t pk[32];
  #pragma unroll
          for (int e = 0; e < 32; ++e) {
            const float2 x = up2(ffma2(pk2(sv[2 * e], sv[2 * e + 1]), c2x2, nmx2));
            const uint64_t y = pk2(ex2(x.x), ex2(x.y));
            l4[e & 3] = fadd2(l4[e & 3], y);
            const float2 yf = up2(y);
            pk[e] = pack_bf16(yf.x, yf.y);
          }
          {
            const float2 la = up2(fadd2(fadd2(l4[0], l4[1]), fadd2(l4[2], l4[3])));
            l += la.x + la.y;
          }
          tmem_st_x32(sbuf + half * 32, pk);          // P over the S columns, bf16 pairs
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(P_FULL(half, tg & 1));
      }
      // Epilogue of the unit: both halves' last products have landed; the
      // two threads of a row exchange their maxima and sums, and each writes
      // its 64 columns of (a0 O_0 + a1 O_1) / L with a_h = 2^(m_h - M),
      // M = max(m_0, m_1), L = a0 l_0 + a1 l_1 -- the normalised rows for a
      // sequence with one chunk, else the partial with (M, L) for the merge.
      const int ul = tt + T - 1;
      const bool direct = p.out != nullptr && qe->nch == 1;
      // the pair's second tile may lie past the tree's rows (or past the
      // last row tile): it computes on zeros and writes nothing
      const bool tile_live = my_rt < p.row_tiles && my_rt * p.rows_per_tile < qe->n * G;
      bool epi = ok && __all_sync(kAll, mbar_wait(O_DONE(0, ul & 1), (ul >> 1) & 1, abort_flag, kWaitNs) &&
                                            mbar_wait(O_DONE(1, ul & 1), (ul >> 1) & 1, abort_flag, kWaitNs));
      float m_p = -INFINITY, l_p = 0.f;
      if (epi) {
        tc_fence_after();
        epi = exchange(m_ref, m_p);
        epi = exchange(l, l_p) && epi;
      }
      const float M = fmaxf(m_ref, m_p);
      const float a_self = m_ref == -INFINITY ? 0.f : ex2(m_ref - M);
      const float a_peer = m_p == -INFINITY ? 0.f : ex2(m_p - M);
      const float L = l * a_self + l_p * a_peer;
      const float inv = L > 0.f ? 1.f / L : 0.f;
      const float w0 = (half == 0 ? a_self : a_peer) * inv, w1 = (half == 0 ? a_peer : a_self) * inv;
      __nv_bfloat16* dst = nullptr;
      if (direct && row_ok) {
        const int m = my_rt * p.rows_per_tile + r;   // query row of the KV head: node m / G, head g G + m % G
        dst = reinterpret_cast<__nv_bfloat16*>(p.out) + ((int64_t)(qe->o0 + m / G) * p.Hq + qe->g * G + m % G) * D;
      } else if (!direct && tile_live) {
        dst = reinterpret_cast<__nv_bfloat16*>(p.o_part) +
              partial_slot(qe->s, qe->b, qe->g, my_rt, r, p.Hkv, p.row_tiles, BM, p.splits) * D;
      }
#pragma unroll 1
      for (int c = 0; c < D / 2 && epi; c += 32) {   // this thread's 64 columns, 32 at a time
        const int col = half * (D / 2) + c;
        uint32_t r0[32], r1[32];
        tmem_ld_x32(tmem + lane_base + 256 + col, r0);
        tmem_ld_x32(tmem + lane_base + 256 + D + col, r1);
        if (dst != nullptr) {
          uint4* ob = reinterpret_cast<uint4*>(dst + col);
#pragma unroll
          for (int e8 = 0; e8 < 4; ++e8) {
            float v[8];
#pragma unroll
            for (int q = 0; q < 8; ++q)
              v[q] = __uint_as_float(r0[8 * e8 + q]) * w0 + __uint_as_float(r1[8 * e8 + q]) * w1;
            uint4 w4;
            w4.x = pack_bf16(v[0], v[1]);
            w4.y = pack_bf16(v[2], v[3]);
            w4.z = pack_bf16(v[4], v[5]);
            w4.w = pack_bf16(v[6], v[7]);
            ob[e8] = w4;
          }
        }
      }
      tc_fence_before();
      if (epi && !direct && tile_live && half == 0)
        p.ml_part[partial_slot(qe->s, qe->b, qe->g, my_rt, r, p.Hkv, p.row_tiles, BM, p.splits)] =
            make_float2(row_ok ? M : -INFINITY, row_ok ? L : 0.f);
      __syncwarp();
      if (lane == 0) release_entry(k);             // done with the queue entry
      k ^= 1;
      if (!epi) ok = false;
      tt += T;
      ++uq;
    }
  }

  // ---------------------------------------------------------------- teardown
  tc_fence_before();
  __syncthreads();
  // neither CTA leaves while the peer may still write into its shared memory
  // (multicast copies are waited by both producers, commits by FIN, remote
  // queue releases by the scheduler's last wait): an execution-only barrier
  // suffices
  cluster_sync_relaxed();
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

EncodeTiledFn encode_fn_p() {
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

bool encode_p(CUtensorMap* m, const void* ptr, int rank, const cuuint64_t* dims, const cuuint64_t* strides,
              const cuuint32_t* box) {
  EncodeTiledFn fn = encode_fn_p();
  if (!fn) return false;
  cuuint32_t es[3] = {1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, rank, const_cast<void*>(ptr), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

int64_t tcp_units(const AttnParams& p) { return (int64_t)p.splits * p.B * p.Hkv * row_pairs(p.row_tiles); }

cudaError_t launch_attn_tcp(const AttnParams& p, cudaStream_t st) {
  if (p.d != D || !p.part_bf16 || !p.work_counter) return cudaErrorInvalidValue;
  CUtensorMap mq, mkc, mvc, mkt, mvt;
  const cuuint64_t row_bytes = (cuuint64_t)D * 2;
  {
    cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)p.Hq, (cuuint64_t)p.R};
    cuuint64_t strides[2] = {row_bytes, row_bytes * p.Hq};
    cuuint32_t box[3] = {64, (cuuint32_t)p.G, (cuuint32_t)(BM / p.G)};
    if (!encode_p(&mq, p.q, 3, dims, strides, box)) return cudaErrorInvalidValue;
  }
  {
    const cuuint64_t rows = p.paged ? (cuuint64_t)p.num_pages * p.Hkv * kPageSize
                                    : (cuuint64_t)p.B * p.Hkv * p.capacity;
    cuuint64_t dims[2] = {(cuuint64_t)D, rows};
    cuuint64_t strides[1] = {row_bytes};
    cuuint32_t box[2] = {64, (cuuint32_t)(p.paged ? kPageSize : KH)};
    if (!encode_p(&mkc, p.k_cache, 2, dims, strides, box) || !encode_p(&mvc, p.v_cache, 2, dims, strides, box))
      return cudaErrorInvalidValue;
  }
  {
    cuuint64_t dims[2] = {(cuuint64_t)D, (cuuint64_t)p.Hkv * p.R};
    cuuint64_t strides[1] = {row_bytes};
    cuuint32_t box[2] = {64, KH};
    if (!encode_p(&mkt, p.k_tree, 2, dims, strides, box) || !encode_p(&mvt, p.v_tree, 2, dims, strides, box))
      return cudaErrorInvalidValue;
  }
  cudaError_t e = ensure_max_dynamic_smem<tv_attn_tcp_kernel>((int)SMEM);
  if (e != cudaSuccess) return e;
  const int64_t units = tcp_units(p);                   // pair units
  const int64_t pairs = num_sms() / 2;
  const int grid = 2 * (int)(units < pairs ? (units > 0 ? units : 1) : pairs);
  return launch_dep(tv_attn_tcp_kernel, dim3(grid), dim3(kThreads), SMEM, st, p, mq, mkc, mvc, mkt, mvt);
}

}  // namespace tv
