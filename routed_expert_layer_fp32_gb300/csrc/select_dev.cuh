// Warp-cooperative top-k selection over one token's logits (the decode router).
// Selection rule ("We Ported Aleph Alpha's Kolibri to a MacBook. Our Own Gate Said No.",
// section "The gate"): the kTopK largest scores, the lowest index first among equal scores,
// then the softmax over the selected experts' logits, renormalised over them.
#pragma once

#include "common.cuh"

namespace moe {

// Order-preserving 32-bit key of a logit; 0 means "not selectable" (NaN, or taken).  -0 and +0
// get one key, so they tie as floats do.
__device__ __forceinline__ uint32_t logit_key(float v) {
  const uint32_t u = v == 0.0f ? 0u : __float_as_uint(v);
  const uint32_t key = (u & 0x80000000u) ? ~u : (u | 0x80000000u);
  return v != v ? 0u : key;
}
__device__ __forceinline__ float key_logit(uint32_t key) {
  return __uint_as_float((key & 0x80000000u) ? (key & 0x7fffffffu) : ~key);
}

// The largest of keys[lo, lo + n) and the lowest j holding it, as a balanced tree (a shallow
// dependency chain; equal keys keep the left, lower, j).
template <int n>
__device__ __forceinline__ void key_argmax(const uint32_t* keys, int lo, uint32_t& best, int& bj) {
  if constexpr (n == 1) {
    best = keys[lo];
    bj = lo;
  } else {
    uint32_t b0, b1;
    int j0, j1;
    key_argmax<n / 2>(keys, lo, b0, j0);
    key_argmax<n - n / 2>(keys, lo + n / 2, b1, j1);
    const bool right = b1 > b0;
    best = right ? b1 : b0;
    bj = right ? j1 : j0;
  }
}

// Free selection of one token by one warp, written out with its weights.  Lane l holds the keys
// of experts l + 32 j (j < kPer) and tracks its largest key and the lowest j holding it.  With
// sel_bias (the selection-only bias mode) the keys rank logit + bias while the weights use the
// logits alone.  Each of the kTopK rounds takes the warp's largest key (one warp reduction),
// then the lowest expert index holding it (a second reduction over the lanes' own best
// indices), and the lane owning that expert drops it: the same experts in the same order as
// kTopK rounds of "larger logit, or equal logit and lower index" over all E logits (softmax is
// monotone in the logit, so choosing on logits chooses on probabilities).  Every lane ends
// with all kTopK choices, so the weights need no further exchange: softmax over the selected
// logits, the largest (slot 0) subtracted, summed in slot order; lane r divides its own slot.
// A slot without a selectable expert gets id -1 and weight 0.  With ids_stage the ids also go
// to that shared-memory row.  The row is read through L2, so logits that other CTAs of the
// same grid wrote (made visible by a fence and a ticket) are seen.
template <int kPer>
__device__ __forceinline__ void select_write_free_t(const float* row, int E, int lane, int32_t* ids_row,
                                                    float* w_row, const float* sel_bias, int* ids_stage) {
  // every load unconditional and in bounds (a clamped index), so all are in flight at once
  float raw[kPer];
#pragma unroll
  for (int j = 0; j < kPer; ++j) raw[j] = __ldcg(row + min(lane + 32 * j, E - 1));
  uint32_t key[kPer];
  if (sel_bias) {
    float b[kPer];
#pragma unroll
    for (int j = 0; j < kPer; ++j) b[j] = __ldg(sel_bias + min(lane + 32 * j, E - 1));
#pragma unroll
    for (int j = 0; j < kPer; ++j) key[j] = lane + 32 * j < E ? logit_key(raw[j] + b[j]) : 0u;
  } else {
#pragma unroll
    for (int j = 0; j < kPer; ++j) key[j] = lane + 32 * j < E ? logit_key(raw[j]) : 0u;
  }
  uint32_t best;
  int bj;
  key_argmax<kPer>(key, 0, best, bj);
  int sel[kTopK];
  float val[kTopK];
#pragma unroll
  for (int r = 0; r < kTopK; ++r) {
    const uint32_t M = __reduce_max_sync(0xffffffffu, best);
    const uint32_t I = __reduce_min_sync(0xffffffffu, best == M ? uint32_t(lane + 32 * bj) : 0xffffffffu);
    if (M != 0u && int(I & 31u) == lane) {  // the owner drops the winner and finds its next best
#pragma unroll
      for (int j = 0; j < kPer; ++j)
        if (j == bj) key[j] = 0u;
      key_argmax<kPer>(key, 0, best, bj);
    }
    sel[r] = M != 0u ? int(I) : -1;
    if (sel_bias) {  // the weight needs the winner's own logit: its lane hands it over
      float mine = 0.0f;
#pragma unroll
      for (int j = 0; j < kPer; ++j)
        if (j == int(I >> 5)) mine = raw[j];
      const float v = __shfl_sync(0xffffffffu, mine, int(I & 31u));
      val[r] = M != 0u ? v : 0.0f;
    } else {
      val[r] = M != 0u ? key_logit(M) : 0.0f;
    }
  }
  // the largest selected logit (slot 0 unless the bias reordered them)
  float m = val[0];
#pragma unroll
  for (int r = 1; r < kTopK; ++r)
    if (sel[r] >= 0) m = fmaxf(m, val[r]);
  float ex[kTopK], s = 0.0f;
#pragma unroll
  for (int r = 0; r < kTopK; ++r) {
    ex[r] = sel[r] >= 0 ? expf(val[r] - m) : 0.0f;
    s += ex[r];
  }
  int my_sel = sel[0];
  float my_ex = ex[0];
#pragma unroll
  for (int r = 1; r < kTopK; ++r) {
    my_sel = lane == r ? sel[r] : my_sel;
    my_ex = lane == r ? ex[r] : my_ex;
  }
  if (lane < kTopK) {
    ids_row[lane] = my_sel;
    w_row[lane] = my_sel >= 0 ? my_ex / s : 0.0f;
    if (ids_stage) ids_stage[lane] = my_sel;
  }
}

__device__ __forceinline__ void select_write_free(const float* row, int E, int lane, int32_t* ids_row, float* w_row,
                                                  const float* sel_bias, int* ids_stage = nullptr) {
  if (E <= 128) select_write_free_t<4>(row, E, lane, ids_row, w_row, sel_bias, ids_stage);
  else if (E <= 256) select_write_free_t<8>(row, E, lane, ids_row, w_row, sel_bias, ids_stage);
  else if (E <= 384) select_write_free_t<12>(row, E, lane, ids_row, w_row, sel_bias, ids_stage);
  else if (E <= 512) select_write_free_t<16>(row, E, lane, ids_row, w_row, sel_bias, ids_stage);
  else select_write_free_t<kMaxExperts / 32>(row, E, lane, ids_row, w_row, sel_bias, ids_stage);
}

}  // namespace moe
