// Which 128x128 (query tile, key tile) pairs an attention kernel visits.
//
// A pair is skipped when the mask zeroes every element of it: the key tile starts
// at or beyond the key-padding length, lies wholly above the diagonal of a causal
// mask, or has its bit cleared in the tile-level block mask ("skip tiles that
// correspond to zeroed-out blocks", galileo blog, Innovation #5).  Every visited
// pair has at least one visible key for each of its query rows.
#pragma once

#include <stdint.h>

namespace fa {

__device__ __forceinline__ bool tile_pair_visible(int qt, int kt, int kv_len, int causal, const uint8_t* bm,
                                                  int n_tiles) {
  if (kt * 128 >= kv_len) return false;
  if (causal && kt > qt) return false;
  if (bm != nullptr && bm[qt * n_tiles + kt] == 0) return false;
  return true;
}

// Smallest key tile >= kt that query tile qt visits, or n_tiles if none.
__device__ __forceinline__ int next_key_tile(int qt, int kt, int kv_len, int causal, const uint8_t* bm,
                                             int n_tiles) {
  while (kt < n_tiles && !tile_pair_visible(qt, kt, kv_len, causal, bm, n_tiles)) ++kt;
  return kt;
}

// Smallest query tile >= qt that visits key tile kt, or n_tiles if none.
__device__ __forceinline__ int next_query_tile(int qt, int kt, int kv_len, int causal, const uint8_t* bm,
                                               int n_tiles) {
  while (qt < n_tiles && !tile_pair_visible(qt, kt, kv_len, causal, bm, n_tiles)) ++qt;
  return qt;
}

__device__ __forceinline__ int clamp_kv_len(const int32_t* kv_len, int b, int N) {
  if (kv_len == nullptr) return N;
  int v = kv_len[b];
  return v < 0 ? 0 : (v > N ? N : v);
}

}  // namespace fa
