// Top-k selection of one token by one warp (shared by the grouped path's
// route/rank kernel and the route-direct prep kernel).
//
// Rule (the top-k routing step of "perf: add small-batch route MMA for MoE",
// Motivation; ties to the lower expert id, softmax over the k selected
// scores): every lane
// holds ceil(E/32) scores as 64-bit keys - order-preserving score bits in the
// high word, the complemented expert id in the low word - so the largest key
// is the largest score and, among equal scores, the lowest id.  -0.0 is
// canonicalised to +0.0 first so that signed zeros tie.  k rounds of a
// warp-wide max pick the experts in slot order; the softmax runs in fp32.
#pragma once

#include "common.cuh"

namespace moe {

__device__ __forceinline__ unsigned long long score_key(float v, int e) {
  v = v + 0.0f;
  uint32_t u = __float_as_uint(v);
  u = (u & 0x80000000u) ? ~u : (u | 0x80000000u);
  return (static_cast<unsigned long long>(u) << 32) | static_cast<uint32_t>(~static_cast<uint32_t>(e));
}

// Inverse of the key's score bits (the canonicalised score itself).
__device__ __forceinline__ float key_score(unsigned long long key) {
  const uint32_t u = static_cast<uint32_t>(key >> 32);
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
template <int MAXV>
__device__ __forceinline__ void route_values(const float (&v)[MAXV], int E, int k, int32_t* __restrict__ ids_row,
                                             float* __restrict__ w_row, int* s_ids_row) {
  const int lane = threadIdx.x & 31;
  unsigned long long key[MAXV];
#pragma unroll
  for (int i = 0; i < MAXV; ++i) {
    const int e = i * 32 + lane;
    key[i] = e < E ? score_key(v[i], e) : 0ull;  // any real key is > 0
  }
  int my_id = 0;
  float my_s = 0.0f;
#pragma unroll 1
  for (int j = 0; j < k; ++j) {
    unsigned long long best = 0ull;
#pragma unroll
    for (int i = 0; i < MAXV; ++i) best = key[i] > best ? key[i] : best;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const unsigned long long other = __shfl_xor_sync(0xffffffffu, best, o);
      best = other > best ? other : best;
    }
    const int id = static_cast<int>(~static_cast<uint32_t>(best & 0xffffffffull));
#pragma unroll
    for (int i = 0; i < MAXV; ++i)
      if (i * 32 + lane == id) key[i] = 0ull;
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
