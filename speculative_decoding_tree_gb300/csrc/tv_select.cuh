// Selection helpers shared by the kernels that pick the largest entries of
// a vocabulary row: an (value, index) entry, the order "larger value first,
// then smaller index" (the pages' tie rule: "ADR-037 — EAGLE-3 with dynamic
// tree port", phase row E4b.10a), and the warp-wide first entry in that
// order.
#pragma once
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

namespace tv {

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

// The first entry of the warp in the order of ent_before, by two warp
// reductions: the largest value (as an order-preserving integer key; an
// empty entry has key 0, below every value), then the smallest index among
// the lanes holding it.
__device__ __forceinline__ uint32_t val_key(float v) {
  uint32_t b = __float_as_uint(v);
  if (b == 0x80000000u) b = 0;                             // -0 orders as +0
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

__device__ __forceinline__ float key_val(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7fffffffu) : ~k);
}

__device__ __forceinline__ Ent warp_first(Ent e) {
  const uint32_t vk = e.i < 0 ? 0u : val_key(e.v);
  const uint32_t best = __reduce_max_sync(0xffffffffu, vk);
  const uint32_t bi = __reduce_min_sync(0xffffffffu, (e.i >= 0 && vk == best) ? (uint32_t)e.i : 0xffffffffu);
  return best == 0u ? Ent{-INFINITY, -1} : Ent{key_val(best), (int)bi};
}

// The same order as one 64-bit integer (larger = first): the value key
// above, then the complemented index (smaller index = larger).  A valid
// entry's key is nonzero; 0 is the empty entry.
__device__ __forceinline__ uint64_t ent_key(float v, int i) {
  return ((uint64_t)val_key(v) << 32) | (uint32_t)~i;
}

__device__ __forceinline__ Ent key_ent(uint64_t k) {
  return k == 0ull ? Ent{-INFINITY, -1} : Ent{key_val((uint32_t)(k >> 32)), (int)~(uint32_t)k};
}

// The warp's largest 64-bit key (two reductions: high word, then the low
// word among the lanes holding that high word).
__device__ __forceinline__ uint64_t warp_max_key(uint64_t k) {
  const uint32_t hi = __reduce_max_sync(0xffffffffu, (uint32_t)(k >> 32));
  const uint32_t lo = __reduce_max_sync(0xffffffffu, (uint32_t)(k >> 32) == hi ? (uint32_t)k : 0u);
  return ((uint64_t)hi << 32) | lo;
}

}  // namespace tv
