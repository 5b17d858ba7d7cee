// Top-k selection of one token by one warp (shared by the grouped path's
// route/rank kernel and the route-direct prep kernel).
//
// Rule (the top-k routing step of "perf: add small-batch route MMA for MoE",
// Motivation; ties to the lower expert id, softmax over the k selected
// scores): every lane holds ceil(E/32) scores as order-preserving 32-bit keys
// (expert i * 32 + lane in slot i); -0.0 is canonicalised to +0.0 first so that
// signed zeros tie.  Each of k rounds takes the warp-wide maximum key and then
// the lowest expert id holding it, so experts come out in slot order; the
// softmax runs in fp32.
#pragma once

#include "common.cuh"

namespace moe {

// Order-preserving 32-bit image of a canonicalised score (-0.0 -> +0.0): the larger
// the score, the larger the key.
__device__ __forceinline__ uint32_t score_bits(float v) {
  v = v + 0.0f;
  const uint32_t u = __float_as_uint(v);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Inverse of score_bits (the canonicalised score itself).
__device__ __forceinline__ float key_score(uint32_t u) {
  return __uint_as_float((u & 0x80000000u) ? (u & 0x7fffffffu) : ~u);
}

// Scores of one token, ceil(E/32) per lane (expert i*32 + lane in slot i).
template <int MAXV>
__device__ __forceinline__ void load_scores(const float* __restrict__ srow, int E, float (&v)[MAXV]) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int i = 0; i < MAXV; ++i) {
    const int e = i * 32 + lane;
    v[i] = e < E ? __ldg(srow + e) : 0.0f;
  }
}

// Route one token from its scores already in registers.  Lane j < k writes
// slot j of each output that is given: ids_row[j], w_row[j], s_ids_row[j].
// Round j takes the warp-wide maximum of the 32-bit score keys still available
// (one redux.sync) and then the lowest expert id holding it: slots are scanned in
// ascending order (expert i * 32 + lane), and within a slot the lowest lane of
// the ballot wins, so equal scores go to the lower expert id.
template <int MAXV>
__device__ __forceinline__ void route_values(const float (&v)[MAXV], int E, int k, int32_t* __restrict__ ids_row,
                                             float* __restrict__ w_row, int* s_ids_row) {
  const int lane = threadIdx.x & 31;
  uint32_t key[MAXV];
  unsigned avail = 0u;  // bit i: expert i * 32 + lane exists and is not taken yet
#pragma unroll
  for (int i = 0; i < MAXV; ++i) {
    key[i] = score_bits(v[i]);
    if (i * 32 + lane < E) avail |= 1u << i;
  }
  int my_id = 0;
  float my_s = 0.0f;
#pragma unroll 1
  for (int j = 0; j < k; ++j) {
    uint32_t best = 0u;
#pragma unroll
    for (int i = 0; i < MAXV; ++i)
      if ((avail >> i) & 1u) best = key[i] > best ? key[i] : best;
    best = __reduce_max_sync(0xffffffffu, best);
    int id = 0;
#pragma unroll
    for (int i = 0; i < MAXV; ++i) {
      const unsigned b = __ballot_sync(0xffffffffu, ((avail >> i) & 1u) && key[i] == best);
      if (b) {
        const int wl = __ffs(b) - 1;
        id = i * 32 + wl;
        if (lane == wl) avail &= ~(1u << i);
        break;
      }
    }
    if (lane == j) {
      my_id = id;
      my_s = key_score(best);
    }
  }
  const float m = __shfl_sync(0xffffffffu, my_s, 0);
  const float ev = lane < k ? expf(my_s - m) : 0.0f;
  float sum = ev;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
  if (lane < k) {
    if (ids_row) ids_row[lane] = my_id;
    if (w_row) w_row[lane] = ev / sum;
    if (s_ids_row) s_ids_row[lane] = my_id;
  }
}

// Lane j < k writes slot j: ids_row[j], w_row[j] and (if given) s_ids_row[j].
template <int MAXV>
__device__ __forceinline__ void route_one_token(const float* __restrict__ srow, int E, int k,
                                                int32_t* __restrict__ ids_row, float* __restrict__ w_row,
                                                int* s_ids_row) {
  float v[MAXV];
  load_scores<MAXV>(srow, E, v);
  route_values<MAXV>(v, E, k, ids_row, w_row, s_ids_row);
}

}  // namespace moe
