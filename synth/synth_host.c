/*
 * synth_host.c - host side of the seeded input generator (see synth.h).
 * Built with -ffp-contract=off so that its float steps round exactly as the
 * device build's __f*_rn intrinsics do.  Every function fills a caller-owned
 * host buffer and may be called from several threads on disjoint ranges.
 */
#include "synth.h"

#include <stdint.h>

/* Rows [row0, row0 + nrows) of the N x K bf16 weight matrix (seed, layer, tensor),
 * row-major into out[nrows * K]. */
void syn_weights_rows_ex(uint64_t seed, uint64_t layer, uint64_t tensor, int64_t K, int64_t row0,
                         int64_t nrows, int outliers, uint16_t* out) {
  uint64_t key = syn_key(seed, layer, tensor);
  uint64_t kc = syn_substream(key, SYN_S_CAT), kg = syn_substream(key, SYN_S_GAUSS);
  for (int64_t r = 0; r < nrows; ++r) {
    uint64_t n = (uint64_t)(row0 + r);
    float scale = syn_channel_scale(key, n);
    for (int64_t k = 0; k < K; ++k)
      out[r * K + k] = syn_weight_ex(kc, kg, n * (uint64_t)K + (uint64_t)k, scale, outliers);
  }
}

void syn_weights_rows(uint64_t seed, uint64_t layer, uint64_t tensor, int64_t K, int64_t row0,
                      int64_t nrows, uint16_t* out) {
  syn_weights_rows_ex(seed, layer, tensor, K, row0, nrows, 1, out);
}

/* Channel scales s_n for rows [row0, row0 + nrows). */
void syn_channel_scales(uint64_t seed, uint64_t layer, uint64_t tensor, int64_t row0, int64_t nrows,
                        float* out) {
  uint64_t key = syn_key(seed, layer, tensor);
  for (int64_t r = 0; r < nrows; ++r) out[r] = syn_channel_scale(key, (uint64_t)(row0 + r));
}

/* Elements [i0, i0 + count) of the bf16 N(0,1) activation tensor (seed, layer, tensor). */
void syn_activations(uint64_t seed, uint64_t layer, uint64_t tensor, int64_t i0, int64_t count,
                     uint16_t* out) {
  uint64_t key = syn_key(seed, layer, tensor);
  for (int64_t i = 0; i < count; ++i) out[i] = syn_activation(key, (uint64_t)(i0 + i));
}

/* Random tree of n nodes: parent[0] = -1, parent[i] uniform in 0..i-1. */
void syn_tree(uint64_t seed, uint64_t layer, uint64_t tensor, int64_t n, int32_t* parent) {
  uint64_t key = syn_substream(syn_key(seed, layer, tensor), SYN_S_TREE);
  for (int64_t i = 0; i < n; ++i) parent[i] = i == 0 ? -1 : (int32_t)syn_below(key, (uint64_t)i, (uint32_t)i);
}

/* n draft tokens uniform in 0..V-1. */
void syn_drafts(uint64_t seed, uint64_t layer, uint64_t tensor, int64_t n, int64_t V, int32_t* out) {
  uint64_t key = syn_substream(syn_key(seed, layer, tensor), SYN_S_DRAFT);
  for (int64_t i = 0; i < n; ++i) out[i] = (int32_t)syn_below(key, (uint64_t)i, (uint32_t)V);
}

/* Raw 64-bit draws of a stream, for planting trees and for tests of the generator. */
void syn_u64(uint64_t seed, uint64_t layer, uint64_t tensor, int64_t i0, int64_t count, uint64_t* out) {
  uint64_t key = syn_key(seed, layer, tensor);
  for (int64_t i = 0; i < count; ++i) out[i] = syn_at(key, (uint64_t)(i0 + i));
}
