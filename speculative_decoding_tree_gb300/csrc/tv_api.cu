// Host side of the C ABI declared in include/tree_verify.h: descriptor
// validation (all before any launch, with checked int64 arithmetic), the
// split-KV launch plan, workspace carving, and the launches themselves.
#include <cmath>
#include <cstdint>
#include <cstring>

#include "tree_expand.h"
#include "tv_internal.cuh"
#include "tv_accept.cuh"

namespace tv {
namespace {

bool mul_ok(int64_t a, int64_t b, int64_t* out) { return !__builtin_mul_overflow(a, b, out); }
bool add_ok(int64_t a, int64_t b, int64_t* out) { return !__builtin_add_overflow(a, b, out); }

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int64_t align_up(int64_t x, int64_t a) { return (x + a - 1) / a * a; }

}  // namespace

int num_sms() {
  // per device (plans are made for the current device), safe across host threads
  static std::atomic<int> cached[kAttrDevices];
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();  // clear the error left by a machine without a GPU
    return kNumSMsDefault;
  }
  const bool tracked = dev >= 0 && dev < kAttrDevices;
  if (tracked && (n = cached[dev].load(std::memory_order_relaxed)) > 0) return n;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) {
    cudaGetLastError();
    return kNumSMsDefault;
  }
  if (tracked) cached[dev].store(n, std::memory_order_relaxed);
  return n;
}

namespace {

// Checks shared by every entry point.  Order follows the pages' validation
// list: dtype, head_dim, zero heads before the GQA modulo, shapes, overflow
// ("ADR-037", phase rows E1 gate, E3 gate and E6 dispatcher).
int validate(const tv_desc* d) {
  if (!d) return TV_ERR_NULL;
  if (d->dtype != TV_F32 && d->dtype != TV_BF16) return TV_ERR_DTYPE;
  if (d->head_dim != 128 && d->head_dim != 256 && d->head_dim != 512) return TV_ERR_HEAD_DIM;
  if (d->num_q_heads <= 0 || d->num_kv_heads <= 0) return TV_ERR_ZERO_HEADS;
  if (d->num_q_heads % d->num_kv_heads != 0) return TV_ERR_GQA;
  if (d->batch < 1) return TV_ERR_SHAPE;
  if (d->max_nodes < 1 || d->max_nodes > kMaxNodes) return TV_ERR_TREE;
  if (d->total_rows < d->batch || (int64_t)d->total_rows > (int64_t)d->batch * d->max_nodes) return TV_ERR_TREE;
  if (!(std::isfinite(d->scale)) || d->scale < 0.f) return TV_ERR_SHAPE;
  if (d->capacity < 1 || d->max_prefix < 0 || d->max_prefix > d->capacity) return TV_ERR_SHAPE;
  if (d->page_size != 0 && d->page_size != kPageSize) return TV_ERR_PAGED;
  if (d->page_size == kPageSize && (d->capacity % kPageSize != 0 || d->num_pages < 1)) return TV_ERR_PAGED;
  // every element count the kernels index must fit int64 in bytes
  int64_t esize = d->dtype == TV_BF16 ? 2 : 4, t = 0;
  int64_t per_row = 0;
  if (!mul_ok(d->head_dim, esize, &per_row)) return TV_ERR_OVERFLOW;
  if (d->page_size == 0) {
    if (!mul_ok(d->batch, d->num_kv_heads, &t) || !mul_ok(t, d->capacity, &t) || !mul_ok(t, per_row, &t))
      return TV_ERR_OVERFLOW;
  } else {
    if (!mul_ok(d->num_pages, d->num_kv_heads, &t) || !mul_ok(t, kPageSize, &t) || !mul_ok(t, per_row, &t))
      return TV_ERR_OVERFLOW;
  }
  if (!mul_ok(d->total_rows, d->num_q_heads, &t) || !mul_ok(t, per_row, &t)) return TV_ERR_OVERFLOW;
  return TV_OK;
}

struct Plan {
  tv_plan pub;
  int G;
  int tree_tile;             // num_chunks rule: 0, or the key tile (one-wave plans)
  int tile_stride;
  int64_t o_part_bytes, ml_part_bytes;
  int64_t counter_bytes;     // the persistent kernel's work counter (0 for the other kernels)
  int64_t part_bytes() const { return o_part_bytes + ml_part_bytes + counter_bytes; }
};

int make_plan(const tv_desc* d, Plan* p) {
  int G = d->num_q_heads / d->num_kv_heads;
  bool tc = d->dtype == TV_BF16 && d->max_nodes * G >= 16 && tc_supported(d, G);
  int key_tile = tc ? tc_key_tile(d->head_dim) : 32;
  int rows_per_tile;
  if (tc) {
    rows_per_tile = (128 / G) * G;
  } else {
    int rpw = 1024 / d->head_dim;          // rows per warp in the CUDA-core kernel
    rows_per_tile = 4 * rpw;
  }
  int row_tiles = (d->max_nodes * G + rows_per_tile - 1) / rows_per_tile;
  // two or more 128-row tiles per KV head: CTA pairs (cta_group::2) share
  // each K/V tile -- for one sequence
  const bool pairs = tc && row_tiles >= 2 && d->batch == 1;
  // a batch on head_dim 128 with a bf16 output: persistent CTA pairs, one CTA
  // per SM, take (sequence, KV head, pair of row tiles, chunk) units from a
  // work counter and share each K/V tile through multicast loads
  const bool persist = tc && d->batch > 1 && d->head_dim == 128 && !d->out_f32;
  const int launched_tiles = (pairs || persist) ? 2 * ((row_tiles + 1) / 2) : row_tiles;
  int64_t units = (int64_t)d->batch * d->num_kv_heads * launched_tiles;
  int64_t sms = num_sms();
  int64_t L = d->max_prefix;
  int64_t chunk;
  int tree_tile = 0;
  if (d->batch == 1) {
    // one wave: at most sms / units splits; the fewest key tiles per chunk
    // with which the prefix, and the tree in the last chunk or on its own
    // (num_chunks), fit that many splits
    int64_t want = sms / units;
    if (want < 1) want = 1;
    const int64_t tiles = (L + key_tile - 1) / key_tile;
    if (tiles > ((int64_t)1 << 30) / key_tile) return TV_ERR_OVERFLOW;
    tree_tile = key_tile;
    int64_t c = (tiles + want - 1) / want;
    if (c < 1) c = 1;
    while (c <= tiles && num_chunks(L, (int)(c * key_tile), tree_tile) > want) ++c;
    chunk = c * key_tile;
  } else {
    // ragged batch: fixed 1920-key chunks (15 key tiles of 128), so that the
    // units balance sequences of different lengths.  On the batched
    // workload's persistent kernel, summed over three seeds of its prefixes
    // and trees, the call took 348.8 / 343.1 / 341.0 / 345.0 us with 1664 /
    // 1792 / 1920 / 2048-key chunks; on one seed 1024 and 4096 keys gave
    // 128.9 and 132.2 us against 120.3 at 2048)
    chunk = align_up(1920, key_tile);
  }
  if (chunk > (int64_t)1 << 30) return TV_ERR_OVERFLOW;
  int splits = num_chunks(L, (int)chunk, tree_tile);
  int64_t grid = units * splits;
  if (grid > ((int64_t)1 << 31) - 1) return TV_ERR_OVERFLOW;
  // launch grids put sequences on z and (KV head, split) or (KV head, row
  // tile) on y, whose limit is 65535: refused here rather than at launch
  const int64_t grid_y = tc ? (int64_t)d->num_kv_heads * splits : (int64_t)splits;
  if (d->batch > kMaxGridYZ || (int64_t)d->num_kv_heads * row_tiles > kMaxGridYZ) return TV_ERR_SHAPE;
  // the persistent kernel's work counter counts in 24 bits; the others put
  // (KV head, split) on grid y
  if (persist ? grid + sms >= ((int64_t)1 << 24) : grid_y > kMaxGridYZ) return TV_ERR_SHAPE;
  p->G = G;
  p->tree_tile = tree_tile;
  p->pub.kernel = persist ? 3 : (pairs ? 2 : (tc ? 1 : 0));
  p->pub.num_splits = splits;
  p->pub.chunk = (int)chunk;
  p->pub.row_tiles = row_tiles;
  p->pub.rows_per_tile = rows_per_tile;
  p->pub.grid_ctas = (int)(persist ? (grid < 2 * (sms / 2) ? grid : 2 * (sms / 2)) : grid);
  p->counter_bytes = persist ? 256 : 0;
  // partials are tile-major: every (split, sequence, KV head, row tile) owns
  // tile_stride rows (128 for the tensor-core kernel, whose epilogue stores
  // whole 128-row tiles)
  p->tile_stride = tc ? 128 : rows_per_tile;
  int64_t t;
  if (!mul_ok(splits, d->batch, &t) || !mul_ok(t, d->num_kv_heads, &t) || !mul_ok(t, row_tiles, &t) ||
      !mul_ok(t, p->tile_stride, &t))
    return TV_ERR_OVERFLOW;
  // partial elements are bf16 when the tensor-core kernels feed a bf16 output
  const int64_t pes = (p->pub.kernel != 0 && d->dtype == TV_BF16 && !d->out_f32) ? 2 : 4;
  int64_t o_bytes, ml_bytes;
  if (!mul_ok(t, (int64_t)d->head_dim * pes, &o_bytes) || !mul_ok(t, 8, &ml_bytes)) return TV_ERR_OVERFLOW;
  p->o_part_bytes = align_up(o_bytes, 256);
  p->ml_part_bytes = align_up(ml_bytes, 256);
  return TV_OK;
}

// Vocabulary chunks per row for the pass: about 16K elements per block, but
// about 4 blocks per SM over all rows, never below 2K elements per block and
// never more than kMaxVChunks chunks.  The argmax pass (streaming, bound by
// the SM with the most blocks) takes at most 4 blocks per SM: 8.28 -> 7.90 us
// per accept + commit at 60 rows x 151936 logits (11 -> 10 chunks); the
// sampled pass (arithmetic-bound) at least 4: 37.8 -> 36.1 us with 11.  The
// workspace holds the larger count.
void accept_chunks(int R, int V, bool sampled, int* vchunks, int* vchunk_len) {
  const int64_t sms = num_sms();
  int64_t want = (V + 16383) / 16384;
  const int64_t fill = sampled ? (4 * sms + R - 1) / R : (4 * sms) / R;
  if (fill > want) want = fill;
  int64_t maxc = (V + 2047) / 2048;
  if (maxc > kMaxVChunks) maxc = kMaxVChunks;
  if (want > maxc) want = maxc;
  if (want < 1) want = 1;
  int64_t len = (V + want - 1) / want;
  len = (len + 7) / 8 * 8;
  *vchunk_len = (int)len;
  *vchunks = (int)((V + len - 1) / len);
}

// Accept area of the workspace: the chunk partials (value and index per row
// and vocabulary chunk).
int64_t accept_bytes(const tv_desc* d, int V) {
  if (V <= 0) return 0;
  int vc, vl;
  accept_chunks(d->total_rows, V, true, &vc, &vl);     // the sampled count, never below the greedy one
  return 2 * align_up((int64_t)d->total_rows * vc * 4, 256);
}

cudaStream_t as_stream(void* s) { return reinterpret_cast<cudaStream_t>(s); }

int check_attn_ptrs(const tv_desc* d, const void* q, const void* kc, const void* vc, const int32_t* pt,
                    const int32_t* pl, const int32_t* no, const void* kt, const void* vt, const uint64_t* anc,
                    const void* ws, int32_t* st) {
  if (!q || !kc || !vc || !pl || !no || !kt || !vt || !anc || !ws || !st) return TV_ERR_NULL;
  if (d->page_size == kPageSize && !pt) return TV_ERR_NULL;
  const void* all[] = {q, kc, vc, pl, no, kt, vt, anc, ws, st};
  for (const void* p : all)
    if (!aligned16(p)) return TV_ERR_ALIGN;
  if (pt && !aligned16(pt)) return TV_ERR_ALIGN;
  return TV_OK;
}

// Partials are stored in bf16 by the tensor-core kernels when the output is
// bf16: they are normalised (O_s / l_s), and P already enters the PV product
// rounded to bf16, so they carry no more rounding than the output itself.
int part_bf16(const tv_desc* d, const Plan& pl) {
  return (pl.pub.kernel != 0 && d->dtype == TV_BF16 && !d->out_f32) ? 1 : 0;
}

AttnParams attn_params(const tv_desc* d, const Plan& pl, const void* q, const void* kc, const void* vc,
                       const int32_t* pt, const int32_t* plen, const int32_t* no, const void* kt,
                       const void* vt, const uint64_t* anc, void* ws, int32_t* st) {
  AttnParams a;
  a.q = q; a.k_cache = kc; a.v_cache = vc;
  a.page_table = d->page_size ? pt : nullptr;
  a.prefix_len = plen; a.node_offsets = no; a.k_tree = kt; a.v_tree = vt; a.anc = anc;
  a.o_part = reinterpret_cast<float*>(ws);
  a.ml_part = reinterpret_cast<float2*>(reinterpret_cast<char*>(ws) + pl.o_part_bytes);
  a.out = nullptr;
  a.out_bf16 = (d->dtype == TV_BF16 && !d->out_f32) ? 1 : 0;
  a.status = st;
  a.work_counter = pl.counter_bytes
                       ? reinterpret_cast<unsigned long long*>(reinterpret_cast<char*>(ws) + pl.o_part_bytes +
                                                               pl.ml_part_bytes)
                       : nullptr;
  a.B = d->batch; a.Hq = d->num_q_heads; a.Hkv = d->num_kv_heads; a.G = pl.G; a.d = d->head_dim;
  a.R = d->total_rows; a.max_nodes = d->max_nodes;
  a.paged = d->page_size != 0;
  a.capacity = d->capacity; a.num_pages = d->num_pages;
  a.max_pages = d->capacity / kPageSize;
  a.max_prefix = d->max_prefix;
  float scale = d->scale > 0.f ? d->scale : 1.0f / std::sqrt((float)d->head_dim);
  a.scale_log2 = scale * 1.4426950408889634f;
  a.chunk = pl.pub.chunk; a.tree_tile = pl.tree_tile; a.splits = pl.pub.num_splits;
  a.rows_per_tile = pl.pub.rows_per_tile; a.row_tiles = pl.pub.row_tiles;
  a.tile_stride = pl.tile_stride;
  a.part_bf16 = part_bf16(d, pl);
  return a;
}

int launch_partials(const tv_desc* d, const Plan& pl, const AttnParams& a, cudaStream_t s) {
  cudaError_t e = pl.pub.kernel == 3   ? launch_attn_tcp(a, s)
                  : pl.pub.kernel == 2 ? launch_attn_tc2(a, s)
                  : pl.pub.kernel == 1 ? launch_attn_tc(a, s)
                                       : launch_attn_simt(a, d->dtype, s);
  return e == cudaSuccess ? TV_OK : TV_ERR_CUDA;
}

int launch_merge_from(const tv_desc* d, const Plan& pl, const int32_t* plen, const int32_t* no, void* out,
                      const void* ws, int32_t* st, cudaStream_t s, int skip_single) {
  MergeParams m;
  m.skip_single = skip_single;
  m.early_reads = skip_single;    // tree_verify_attn: the split pass of this call precedes the merge
  m.prefix_len = plen; m.node_offsets = no;
  m.o_part = reinterpret_cast<const float*>(ws);
  m.ml_part = reinterpret_cast<const float2*>(reinterpret_cast<const char*>(ws) + pl.o_part_bytes);
  m.out = out; m.status = st;
  m.part_bf16 = part_bf16(d, pl);
  m.B = d->batch; m.Hq = d->num_q_heads; m.d = d->head_dim; m.R = d->total_rows; m.max_nodes = d->max_nodes;
  m.out_bf16 = (d->dtype == TV_BF16 && !d->out_f32) ? 1 : 0;
  m.max_prefix = d->max_prefix; m.capacity = d->capacity;
  m.chunk = pl.pub.chunk; m.tree_tile = pl.tree_tile; m.splits = pl.pub.num_splits;
  m.Hkv = d->num_kv_heads; m.G = pl.G; m.rows_per_tile = pl.pub.rows_per_tile;
  m.row_tiles = pl.pub.row_tiles; m.tile_stride = pl.tile_stride;
  merge_shape(d->batch * d->num_kv_heads * pl.pub.row_tiles, pl.tile_stride, d->head_dim, m.part_bf16 ? 2 : 4,
              pl.pub.num_splits, num_sms(), &m.slab_rows, &m.batch_splits);
  return launch_merge(m, s) == cudaSuccess ? TV_OK : TV_ERR_CUDA;
}

// tree_accept_commit and its sampled form: validation, workspace, launch.
int accept_commit_impl(const tv_desc* desc, int32_t vocab, int32_t logits_dtype, const void* d_logits, int sampled,
                       float temperature, uint64_t seed, uint64_t offset, const int32_t* d_draft_tokens,
                       const int32_t* d_parents, const int32_t* d_node_offsets, const void* d_k_tree,
                       const void* d_v_tree, void* d_k_cache, void* d_v_cache, const int32_t* d_page_table,
                       int32_t* d_prefix_len, int32_t* d_argmax, int32_t* d_accept_len, int32_t* d_path,
                       int32_t* d_tokens, void* d_workspace, size_t workspace_bytes, int32_t* d_status,
                       void* stream) {
  int rc = validate(desc);
  if (rc) return rc;
  if (desc->total_rows > kMaxGridYZ) return TV_ERR_SHAPE;   // one argmax row per grid y index
  if (logits_dtype != TV_F32 && logits_dtype != TV_BF16) return TV_ERR_DTYPE;
  if (vocab < 1) return TV_ERR_SHAPE;
  if (!d_logits || !d_draft_tokens || !d_parents || !d_node_offsets || !d_k_tree || !d_v_tree || !d_k_cache ||
      !d_v_cache || !d_prefix_len || !d_argmax || !d_accept_len || !d_path || !d_tokens || !d_workspace ||
      !d_status)
    return TV_ERR_NULL;
  if (desc->page_size == kPageSize && !d_page_table) return TV_ERR_NULL;
  const void* all[] = {d_logits, d_draft_tokens, d_parents, d_node_offsets, d_k_tree, d_v_tree, d_k_cache,
                       d_v_cache, d_prefix_len, d_argmax, d_accept_len, d_path, d_tokens, d_workspace, d_status};
  for (const void* ptr : all)
    if (!aligned16(ptr)) return TV_ERR_ALIGN;
  if (d_page_table && !aligned16(d_page_table)) return TV_ERR_ALIGN;
  int64_t lb;
  if (!mul_ok(desc->total_rows, vocab, &lb) || !mul_ok(lb, 4, &lb)) return TV_ERR_OVERFLOW;
  Plan p;
  rc = make_plan(desc, &p);
  if (rc) return rc;
  int64_t off = p.part_bytes();
  if ((int64_t)workspace_bytes < off + accept_bytes(desc, vocab)) return TV_ERR_WORKSPACE;
  AcceptParams a;
  a.given_argmax = 0;
  a.sampled = sampled;
  a.inv_temp = sampled ? 1.f / temperature : 0.f;
  a.seed_lo = (uint32_t)seed;
  a.seed_hi = (uint32_t)(seed >> 32);
  a.off_lo = (uint32_t)offset;
  a.off_hi = (uint32_t)(offset >> 32);
  a.logits = d_logits; a.logits_bf16 = logits_dtype == TV_BF16; a.V = vocab;
  a.draft = d_draft_tokens; a.parents = d_parents; a.node_offsets = d_node_offsets;
  a.k_tree = d_k_tree; a.v_tree = d_v_tree; a.k_cache = d_k_cache; a.v_cache = d_v_cache;
  a.page_table = desc->page_size ? d_page_table : nullptr;
  a.prefix_len = d_prefix_len; a.argmax = d_argmax; a.accept_len = d_accept_len;
  a.path = d_path; a.tokens = d_tokens; a.status = d_status;
  accept_chunks(desc->total_rows, vocab, sampled != 0, &a.vchunks, &a.vchunk_len);
  int64_t part = align_up((int64_t)desc->total_rows * a.vchunks * 4, 256);
  a.am_val = reinterpret_cast<float*>(reinterpret_cast<char*>(d_workspace) + off);
  a.am_idx = reinterpret_cast<int32_t*>(reinterpret_cast<char*>(d_workspace) + off + part);
  a.B = desc->batch; a.R = desc->total_rows; a.Hkv = desc->num_kv_heads; a.d = desc->head_dim;
  a.esize = desc->dtype == TV_BF16 ? 2 : 4; a.max_nodes = desc->max_nodes; a.paged = desc->page_size != 0;
  a.capacity = desc->capacity; a.num_pages = desc->num_pages; a.max_pages = desc->capacity / kPageSize;
  a.stage_bytes = walk_stage_bytes(a.Hkv, a.max_nodes, (int64_t)a.d * a.esize);
  cudaError_t e = launch_accept_commit(a, as_stream(stream));
  return e == cudaSuccess ? TV_OK : TV_ERR_CUDA;
}

}  // namespace
}  // namespace tv

using namespace tv;

extern "C" {

const char* tv_version(void) { return "treeverify 0.1 sm_103a"; }

const char* tv_status_string(int code) {
  switch (code) {
    case TV_OK: return "ok";
    case TV_ERR_NULL: return "null pointer";
    case TV_ERR_DTYPE: return "unsupported dtype";
    case TV_ERR_HEAD_DIM: return "unsupported head_dim (128, 256, 512)";
    case TV_ERR_ZERO_HEADS: return "zero query or KV heads";
    case TV_ERR_GQA: return "num_q_heads not a multiple of num_kv_heads";
    case TV_ERR_SHAPE: return "shape out of range";
    case TV_ERR_TREE: return "tree size out of range (max_nodes 1..64, total_rows)";
    case TV_ERR_PAGED: return "bad paged-cache description";
    case TV_ERR_OVERFLOW: return "size overflows int64";
    case TV_ERR_WORKSPACE: return "workspace too small";
    case TV_ERR_ALIGN: return "device pointer not 16-byte aligned";
    case TV_ERR_CUDA: return "CUDA launch failed";
    case TV_DEV_BAD_TREE: return "device: bad parent pointer";
    case TV_DEV_BAD_OFFSETS: return "device: bad node offsets";
    case TV_DEV_BAD_PREFIX: return "device: prefix length out of range";
    case TV_DEV_BAD_PAGE: return "device: page id out of range";
    case TV_DEV_CAPACITY: return "device: accepted rows do not fit the cache";
    case TV_DEV_TIMEOUT: return "device: bounded wait ran out";
    case TV_DEV_BAD_LOGITS: return "device: +inf draft logit (node not expanded)";
    case TV_DEV_BAD_STEP: return "device: expansion step out of order";
    default: return "unknown";
  }
}

int tv_attn_plan(const tv_desc* desc, tv_plan* plan) {
  int rc = validate(desc);
  if (rc) return rc;
  if (!plan) return TV_ERR_NULL;
  Plan p;
  rc = make_plan(desc, &p);
  if (rc) return rc;
  *plan = p.pub;
  return TV_OK;
}

int tv_workspace_size(const tv_desc* desc, int32_t vocab, size_t* bytes) {
  int rc = validate(desc);
  if (rc) return rc;
  if (!bytes) return TV_ERR_NULL;
  if (vocab < 0) return TV_ERR_SHAPE;
  Plan p;
  rc = make_plan(desc, &p);
  if (rc) return rc;
  int64_t total = 0;
  if (!add_ok(p.part_bytes(), accept_bytes(desc, vocab), &total))
    return TV_ERR_OVERFLOW;
  *bytes = (size_t)total;
  return TV_OK;
}

int tv_build_tree_mask(const tv_desc* desc, const int32_t* d_parents, const int32_t* d_node_offsets,
                       uint64_t* d_anc, int32_t* d_depth, int32_t* d_status, void* stream) {
  int rc = validate(desc);
  if (rc) return rc;
  if (!d_parents || !d_node_offsets || !d_anc || !d_status) return TV_ERR_NULL;
  if (!aligned16(d_parents) || !aligned16(d_node_offsets) || !aligned16(d_anc) || !aligned16(d_status) ||
      (d_depth && !aligned16(d_depth)))
    return TV_ERR_ALIGN;
  cudaError_t e = launch_tree_mask(d_parents, d_node_offsets, d_anc, d_depth, d_status, desc->batch,
                                   desc->total_rows, desc->max_nodes, as_stream(stream));
  return e == cudaSuccess ? TV_OK : TV_ERR_CUDA;
}

int tv_attn_partials(const tv_desc* desc, const void* d_q, const void* d_k_cache, const void* d_v_cache,
                     const int32_t* d_page_table, const int32_t* d_prefix_len, const int32_t* d_node_offsets,
                     const void* d_k_tree, const void* d_v_tree, const uint64_t* d_anc, void* d_workspace,
                     size_t workspace_bytes, int32_t* d_status, void* stream) {
  int rc = validate(desc);
  if (rc) return rc;
  rc = check_attn_ptrs(desc, d_q, d_k_cache, d_v_cache, d_page_table, d_prefix_len, d_node_offsets, d_k_tree,
                       d_v_tree, d_anc, d_workspace, d_status);
  if (rc) return rc;
  Plan p;
  rc = make_plan(desc, &p);
  if (rc) return rc;
  if ((int64_t)workspace_bytes < p.part_bytes()) return TV_ERR_WORKSPACE;
  AttnParams a = attn_params(desc, p, d_q, d_k_cache, d_v_cache, d_page_table, d_prefix_len, d_node_offsets,
                             d_k_tree, d_v_tree, d_anc, d_workspace, d_status);
  return launch_partials(desc, p, a, as_stream(stream));
}

int tv_attn_merge(const tv_desc* desc, const int32_t* d_prefix_len, const int32_t* d_node_offsets, void* d_out,
                  const void* d_workspace, size_t workspace_bytes, int32_t* d_status, void* stream) {
  int rc = validate(desc);
  if (rc) return rc;
  if (!d_prefix_len || !d_node_offsets || !d_out || !d_workspace || !d_status) return TV_ERR_NULL;
  if (!aligned16(d_prefix_len) || !aligned16(d_node_offsets) || !aligned16(d_out) || !aligned16(d_workspace) ||
      !aligned16(d_status))
    return TV_ERR_ALIGN;
  Plan p;
  rc = make_plan(desc, &p);
  if (rc) return rc;
  if ((int64_t)workspace_bytes < p.part_bytes()) return TV_ERR_WORKSPACE;
  return launch_merge_from(desc, p, d_prefix_len, d_node_offsets, d_out, d_workspace, d_status,
                           as_stream(stream), 0);
}

int tree_verify_attn(const tv_desc* desc, const void* d_q, const void* d_k_cache, const void* d_v_cache,
                     const int32_t* d_page_table, const int32_t* d_prefix_len, const int32_t* d_node_offsets,
                     const void* d_k_tree, const void* d_v_tree, const uint64_t* d_anc, void* d_out,
                     void* d_workspace, size_t workspace_bytes, int32_t* d_status, void* stream) {
  int rc = validate(desc);
  if (rc) return rc;
  rc = check_attn_ptrs(desc, d_q, d_k_cache, d_v_cache, d_page_table, d_prefix_len, d_node_offsets, d_k_tree,
                       d_v_tree, d_anc, d_workspace, d_status);
  if (rc) return rc;
  if (!d_out) return TV_ERR_NULL;
  if (!aligned16(d_out)) return TV_ERR_ALIGN;
  Plan p;
  rc = make_plan(desc, &p);
  if (rc) return rc;
  if ((int64_t)workspace_bytes < p.part_bytes()) return TV_ERR_WORKSPACE;
  AttnParams a = attn_params(desc, p, d_q, d_k_cache, d_v_cache, d_page_table, d_prefix_len, d_node_offsets,
                             d_k_tree, d_v_tree, d_anc, d_workspace, d_status);
  a.out = d_out;                      // one-chunk sequences are finished by the split pass
  cudaStream_t s = as_stream(stream);
  rc = launch_partials(desc, p, a, s);
  if (rc) return rc;
  if (p.pub.num_splits == 1) return TV_OK;   // every sequence has one chunk: nothing to merge
  return launch_merge_from(desc, p, d_prefix_len, d_node_offsets, d_out, d_workspace, d_status, s, 1);
}

int tree_accept_commit(const tv_desc* desc, int32_t vocab, int32_t logits_dtype, const void* d_logits,
                       const int32_t* d_draft_tokens, const int32_t* d_parents, const int32_t* d_node_offsets,
                       const void* d_k_tree, const void* d_v_tree, void* d_k_cache, void* d_v_cache,
                       const int32_t* d_page_table, int32_t* d_prefix_len, int32_t* d_argmax,
                       int32_t* d_accept_len, int32_t* d_path, int32_t* d_tokens, void* d_workspace,
                       size_t workspace_bytes, int32_t* d_status, void* stream) {
  return accept_commit_impl(desc, vocab, logits_dtype, d_logits, 0, 0.f, 0, 0, d_draft_tokens, d_parents,
                            d_node_offsets, d_k_tree, d_v_tree, d_k_cache, d_v_cache, d_page_table, d_prefix_len,
                            d_argmax, d_accept_len, d_path, d_tokens, d_workspace, workspace_bytes, d_status, stream);
}

int tree_accept_commit_sampled(const tv_desc* desc, int32_t vocab, int32_t logits_dtype, const void* d_logits,
                               float temperature, uint64_t seed, uint64_t offset, const int32_t* d_draft_tokens,
                               const int32_t* d_parents, const int32_t* d_node_offsets, const void* d_k_tree,
                               const void* d_v_tree, void* d_k_cache, void* d_v_cache, const int32_t* d_page_table,
                               int32_t* d_prefix_len, int32_t* d_sampled, int32_t* d_accept_len, int32_t* d_path,
                               int32_t* d_tokens, void* d_workspace, size_t workspace_bytes, int32_t* d_status,
                               void* stream) {
  if (!(temperature > 0.f) || !std::isfinite(temperature) || !std::isfinite(1.f / temperature)) return TV_ERR_SHAPE;
  return accept_commit_impl(desc, vocab, logits_dtype, d_logits, 1, temperature, seed, offset, d_draft_tokens,
                            d_parents, d_node_offsets, d_k_tree, d_v_tree, d_k_cache, d_v_cache, d_page_table,
                            d_prefix_len, d_sampled, d_accept_len, d_path, d_tokens, d_workspace, workspace_bytes,
                            d_status, stream);
}

int tree_accept_commit_argmax(const tv_desc* desc, const int32_t* d_argmax, const int32_t* d_draft_tokens,
                              const int32_t* d_parents, const int32_t* d_node_offsets, const void* d_k_tree,
                              const void* d_v_tree, void* d_k_cache, void* d_v_cache, const int32_t* d_page_table,
                              int32_t* d_prefix_len, int32_t* d_accept_len, int32_t* d_path, int32_t* d_tokens,
                              int32_t* d_status, void* stream) {
  int rc = validate(desc);
  if (rc) return rc;
  if (!d_argmax || !d_draft_tokens || !d_parents || !d_node_offsets || !d_k_tree || !d_v_tree || !d_k_cache ||
      !d_v_cache || !d_prefix_len || !d_accept_len || !d_path || !d_tokens || !d_status)
    return TV_ERR_NULL;
  if (desc->page_size == kPageSize && !d_page_table) return TV_ERR_NULL;
  const void* all[] = {d_argmax, d_draft_tokens, d_parents, d_node_offsets, d_k_tree, d_v_tree, d_k_cache,
                       d_v_cache, d_prefix_len, d_accept_len, d_path, d_tokens, d_status};
  for (const void* ptr : all)
    if (!aligned16(ptr)) return TV_ERR_ALIGN;
  if (d_page_table && !aligned16(d_page_table)) return TV_ERR_ALIGN;
  AcceptParams a = {};
  a.given_argmax = 1;
  a.draft = d_draft_tokens; a.parents = d_parents; a.node_offsets = d_node_offsets;
  a.k_tree = d_k_tree; a.v_tree = d_v_tree; a.k_cache = d_k_cache; a.v_cache = d_v_cache;
  a.page_table = desc->page_size ? d_page_table : nullptr;
  a.prefix_len = d_prefix_len; a.argmax = const_cast<int32_t*>(d_argmax); a.accept_len = d_accept_len;
  a.path = d_path; a.tokens = d_tokens; a.status = d_status;
  a.B = desc->batch; a.R = desc->total_rows; a.Hkv = desc->num_kv_heads; a.d = desc->head_dim;
  a.esize = desc->dtype == TV_BF16 ? 2 : 4; a.max_nodes = desc->max_nodes; a.paged = desc->page_size != 0;
  a.capacity = desc->capacity; a.num_pages = desc->num_pages; a.max_pages = desc->capacity / kPageSize;
  a.stage_bytes = walk_stage_bytes(a.Hkv, a.max_nodes, (int64_t)a.d * a.esize);
  cudaError_t e = launch_accept_commit(a, as_stream(stream));
  return e == cudaSuccess ? TV_OK : TV_ERR_CUDA;
}

}  // extern "C"
