// Route-direct small-batch path for FP8 weights ("perf: add small-batch route
// MMA for MoE", Summary and Motivation): the data stays in route order - each
// route's Gate/Up product, then one fused pass that sums the K splits, applies
// SwiGLU and quantises the Down input, then each route's Down product, then the
// per-token reduction over contiguous rows - with no expert sort, gather,
// prefix sum or task map.
//
// The work is bound by streaming the selected experts' weights from HBM, so
// every kernel here is organised around that stream:
//   rd_prep     one block: routing of all T tokens, dynamic e4m3 quantisation
//               of x (per tensor, or per token and 128 columns), and the table
//               of distinct selected experts in first-use order with their
//               routes (a route-order scan of at most 1024 routes, no sort), so
//               an expert chosen by several tokens is streamed once.
//   rd_gateup   one CTA per (distinct expert, 64 rows of W1[e], K split):
//               each warp streams 16 rows of e4m3 weights with 16-byte loads
//               straight into mma.sync m16n8k32 e4m3 fragments (weights on M,
//               up to 8 routes of that expert on N), fp32 partials per split.
//   rd_reduce   sums the K splits, applies the scales and SwiGLU; blockwise
//               mode quantises h per (route, 128 columns) here, per-tensor mode
//               records the global amax of h.
//   rd_down     one CTA per (distinct expert, 64 rows of W2[e]); h of the
//               expert's routes is quantised (per-tensor) or copied into
//               shared memory, weights streamed as above; fp32 o in route order.
//   combine     the contiguous top-k reduction shared with the grouped path.
//
// K permutation: a dot product does not depend on the order of its terms, so
// each thread loads 16 consecutive bytes of a weight row and of x and feeds
// bytes 0-7 to one m16n8k32 and bytes 8-15 to the next; A and B use the same
// assignment, which is what makes it exact.
#include "common.cuh"
#include "internal.h"
#include "routing.cuh"

namespace moe {
namespace rd {

constexpr int ROWS_PER_CTA = 64;  // 4 warps x 16 rows
constexpr int THREADS = 128;

// Table of distinct experts, in int32 words:
//   [0] U;  [1 .. 1+maxU) expert of u;  [1+maxU .. 2+2maxU) CSR offsets of u;
//   [2+2maxU .. 2+2maxU+R) routes of u, in route order.
struct UniqView {
  int32_t* base;
  int maxU;
  __host__ __device__ int32_t* U() const { return base; }
  __host__ __device__ int32_t* expert() const { return base + 1; }
  __host__ __device__ int32_t* off() const { return base + 1 + maxU; }
  __host__ __device__ int32_t* routes() const { return base + 2 + 2 * maxU; }
};

__host__ __device__ inline int max_uniq(int R, int E) { return R < E ? R : E; }

__device__ __forceinline__ void mma_e4m3(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k32.row.col.f32.e4m3.e4m3.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint4 ld_stream(const uint8_t* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

// Two m16n8k32 over a 64-wide K slice: A0/A1 = 16 bytes of rows g and g+8, X = 16 bytes of token g.
__device__ __forceinline__ void mma_k64(float (&c)[4], const uint4& A0, const uint4& A1, const uint4& X) {
  mma_e4m3(c, A0.x, A1.x, A0.y, A1.y, X.x, X.y);
  mma_e4m3(c, A0.z, A1.z, A0.w, A1.w, X.z, X.w);
}

// Programmatic dependent launch: every kernel after rd_prep is launched while
// its predecessor still runs; it waits here before touching the predecessor's
// results, and lets its own successor launch as early as possible.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// ------------------------------------------------------------------ rd_prep
template <int MAXV>
__global__ void __launch_bounds__(1024) rd_prep_kernel(DecodeArgs a) {
  __shared__ int s_ids[kRouteDirectMaxRoutes];
  __shared__ int s_first[kMaxE];
  __shared__ int s_isfirst[kRouteDirectMaxRoutes];
  __shared__ int s_pos[kRouteDirectMaxRoutes];
  __shared__ int s_cnt[kRouteDirectMaxRoutes];
  __shared__ float s_red[32];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, nwarps = blockDim.x >> 5;
  const int T = a.T, E = a.E, k = a.k, H = a.H, R = a.R;
  pdl_trigger();
  if (tid == 0) {
    a.hdr->status = 0u;
    a.hdr->info = 0u;
    a.hdr->amax_x = 0u;
    a.hdr->amax_h = 0u;
  }
  // 1. routing
  for (int t = warp; t < T; t += nwarps)
    route_one_token<MAXV>(a.scores + static_cast<size_t>(t) * E, E, k, a.ids + static_cast<size_t>(t) * k,
                           a.w + static_cast<size_t>(t) * k, s_ids + t * k);
  // 2. dynamic e4m3 quantisation of x
  const __nv_bfloat16* x = static_cast<const __nv_bfloat16*>(a.x);
  if (a.quant == MOE_FP8_PER_TENSOR) {
    // loads go out in batches of 8 x 16 bytes per thread: one memory round trip per batch
    float m = 0.0f;
    const int n8 = T * H / 8;
    const uint4* x8 = reinterpret_cast<const uint4*>(x);
    for (int base = tid; base < n8; base += blockDim.x * 8) {
      uint4 v[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const int i = base + j * blockDim.x;
        v[j] = i < n8 ? __ldg(x8 + i) : make_uint4(0, 0, 0, 0);
      }
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const __nv_bfloat162* b = reinterpret_cast<const __nv_bfloat162*>(&v[j]);
#pragma unroll
        for (int h2 = 0; h2 < 4; ++h2) {
          const float2 f = __bfloat1622float2(b[h2]);
          m = fmaxf(m, fmaxf(fabsf(f.x), fabsf(f.y)));
        }
      }
    }
    m = warp_max(m);
    if (lane == 0) s_red[warp] = m;
    __syncthreads();
    if (warp == 0) {
      float v = lane < nwarps ? s_red[lane] : 0.0f;
      v = warp_max(v);
      if (lane == 0) s_red[0] = v;
    }
    __syncthreads();
    const float amax = s_red[0];
    const float s = e4m3_scale(amax);
    if (tid == 0) {
      a.sx[0] = s;
      a.hdr->amax_x = __float_as_uint(amax);
    }
    for (int base = tid; base < n8; base += blockDim.x * 8) {
      uint4 v[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const int i = base + j * blockDim.x;
        v[j] = i < n8 ? __ldg(x8 + i) : make_uint4(0, 0, 0, 0);
      }
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const int i = base + j * blockDim.x;
        if (i < n8) {
          const __nv_bfloat162* b = reinterpret_cast<const __nv_bfloat162*>(&v[j]);
          uint32_t q[2];
#pragma unroll
          for (int h2 = 0; h2 < 2; ++h2) {
            const float2 f0 = __bfloat1622float2(b[2 * h2]), f1 = __bfloat1622float2(b[2 * h2 + 1]);
            q[h2] = static_cast<uint32_t>(cvt_e4m3x2(f0.x / s, f0.y / s)) |
                    (static_cast<uint32_t>(cvt_e4m3x2(f1.x / s, f1.y / s)) << 16);
          }
          reinterpret_cast<uint2*>(a.xq)[i] = make_uint2(q[0], q[1]);
        }
      }
    }
  } else {
    const int ng = H / 128, ntask = T * ng;
    for (int base = warp; base < ntask; base += nwarps * 8) {
      uint2 v[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const int gi = base + j * nwarps;
        const int t = gi / ng, G = gi - (gi / ng) * ng;
        v[j] = gi < ntask ? __ldg(reinterpret_cast<const uint2*>(x + static_cast<size_t>(t) * H + G * 128) + lane)
                          : make_uint2(0, 0);
      }
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const int gi = base + j * nwarps;  // warp-uniform
        if (gi < ntask) {
          const int t = gi / ng, G = gi - (gi / ng) * ng;
          const float2 f0 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&v[j].x));
          const float2 f1 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&v[j].y));
          float m = fmaxf(fmaxf(fabsf(f0.x), fabsf(f0.y)), fmaxf(fabsf(f1.x), fabsf(f1.y)));
          m = warp_max(m);
          const float s = e4m3_scale(m);
          const uint32_t q = static_cast<uint32_t>(cvt_e4m3x2(f0.x / s, f0.y / s)) |
                             (static_cast<uint32_t>(cvt_e4m3x2(f1.x / s, f1.y / s)) << 16);
          *reinterpret_cast<uint32_t*>(a.xq + static_cast<size_t>(t) * H + G * 128 + lane * 4) = q;
          if (lane == 0) a.sx[static_cast<size_t>(t) * ng + G] = s;
        }
      }
    }
  }
  // 3. distinct experts in first-use order, routes of each in route order
  for (int e = tid; e < E; e += blockDim.x) s_first[e] = 0x7fffffff;
  __syncthreads();
  for (int r = tid; r < R; r += blockDim.x) atomicMin(&s_first[s_ids[r]], r);
  __syncthreads();
  for (int r = tid; r < R; r += blockDim.x) s_isfirst[r] = s_first[s_ids[r]] == r ? 1 : 0;
  __syncthreads();
  if (warp == 0) {
    // exclusive scan of s_isfirst (first-use index of each distinct expert), and the
    // position of every route within its expert's list, walking routes in order
    int run = 0;
    for (int c = 0; c < R; c += 32) {
      const int r = c + lane;
      const int f = r < R ? s_isfirst[r] : 0;
      int incl = f;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += v;
      }
      if (r < R) s_isfirst[r] = f ? run + incl - 1 : -1;  // u index for first routes
      run += __shfl_sync(0xffffffffu, incl, 31);
    }
    __syncwarp();
    for (int u = lane; u < run; u += 32) s_cnt[u] = 0;
    __syncwarp();
    for (int c = 0; c < R; c += 32) {
      const int r = c + lane;
      const int u = r < R ? s_isfirst[s_first[s_ids[r]]] : -1 - lane;
      const unsigned peers = __match_any_sync(0xffffffffu, u);
      const int rank = __popc(peers & ((1u << lane) - 1u));
      const int base = r < R ? s_cnt[u] : 0;
      __syncwarp();
      if (r < R && rank == 0) s_cnt[u] = base + __popc(peers);
      __syncwarp();
      if (r < R) s_pos[r] = base + rank;
    }
    __syncwarp();
    if (lane == 0) {
      UniqView uv{a.uniq, max_uniq(R, E)};
      uv.U()[0] = run;
      int acc = 0;
      for (int u = 0; u < run; ++u) {
        uv.off()[u] = acc;
        acc += s_cnt[u];
      }
      uv.off()[run] = acc;
    }
  }
  __syncthreads();
  {
    UniqView uv{a.uniq, max_uniq(R, E)};
    for (int r = tid; r < R; r += blockDim.x) {
      const int u = s_isfirst[s_first[s_ids[r]]];
      if (s_first[s_ids[r]] == r) uv.expert()[u] = s_ids[r];
      uv.routes()[uv.off()[u] + s_pos[r]] = r;
    }
  }
}

// ------------------------------------------------------------------ rd_gateup
// grid = maxU * nMB * S; block = 128 threads (4 warps x 16 rows of W1[e]).
template <bool BLOCKWISE>
__global__ void __launch_bounds__(THREADS) rd_gateup_kernel(DecodeArgs a, int nMB, int S) {
  pdl_trigger();
  pdl_wait();
  const int unit = blockIdx.x;
  const int s = unit % S;
  const int mb = (unit / S) % nMB;
  const int u = unit / (S * nMB);
  UniqView uv{a.uniq, max_uniq(a.R, a.E)};
  if (u >= uv.U()[0]) return;
  const int e = uv.expert()[u];
  const int r_beg = uv.off()[u], cnt = uv.off()[u + 1] - r_beg;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, tig = lane & 3;
  const int twoI = 2 * a.I, H = a.H;
  const int row = mb * ROWS_PER_CTA + warp * 16 + g;  // rows row and row+8 of W1[e]
  const int KS = H / S;
  const int k0 = s * KS;
  const uint8_t* wrow0 = a.w1 + (static_cast<size_t>(e) * twoI + row) * H + 16 * tig;
  const uint8_t* wrow1 = wrow0 + static_cast<size_t>(8) * H;
  const int ng = H / 128;

  for (int n0 = 0; n0 < cnt; n0 += 8) {
    const int nn = min(8, cnt - n0);
    const int my_r = g < nn ? uv.routes()[r_beg + n0 + g] : -1;  // route of token column g
    const int my_t = my_r >= 0 ? my_r / a.k : 0;
    const uint8_t* xrow = a.xq + static_cast<size_t>(my_t) * H + 16 * tig;
    float c[4] = {0.f, 0.f, 0.f, 0.f};
    const int kend = k0 + KS;
    if (!BLOCKWISE) {
      // the loads of NB K-steps are issued before their MMAs: NB x 32 bytes of
      // weights in flight per thread
      constexpr int NB = 8;
      for (int kb0 = k0; kb0 < kend; kb0 += 64 * NB) {
        uint4 A0[NB], A1[NB], X[NB];
#pragma unroll
        for (int i = 0; i < NB; ++i) {
          const int kk = kb0 + 64 * i;
          const bool in = kk < kend;
          A0[i] = in ? ld_stream(wrow0 + kk) : make_uint4(0, 0, 0, 0);
          A1[i] = in ? ld_stream(wrow1 + kk) : make_uint4(0, 0, 0, 0);
          X[i] = in && my_r >= 0 ? __ldg(reinterpret_cast<const uint4*>(xrow + kk)) : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int i = 0; i < NB; ++i) mma_k64(c, A0[i], A1[i], X[i]);
      }
    } else {
      // per 128-wide K block: fresh partial, then scale by s_w1[e, row/128, kb] * s_x[t, kb]
      const int rb = row / 128;
      const int t0 = 2 * tig < nn ? uv.routes()[r_beg + n0 + 2 * tig] / a.k : 0;
      const int t1 = 2 * tig + 1 < nn ? uv.routes()[r_beg + n0 + 2 * tig + 1] / a.k : 0;
      const float* sw = a.w1_scale + (static_cast<size_t>(e) * (twoI / 128) + rb) * ng;
      constexpr int NB = 4;  // 128-wide K blocks per batch of loads
      for (int kb0 = k0; kb0 < kend; kb0 += 128 * NB) {
        uint4 A0[NB], A1[NB], B0[NB], B1[NB], X0[NB], X1[NB];
#pragma unroll
        for (int i = 0; i < NB; ++i) {
          const int kk = kb0 + 128 * i;
          const bool in = kk < kend;
          const uint4 z = make_uint4(0, 0, 0, 0);
          A0[i] = in ? ld_stream(wrow0 + kk) : z;
          A1[i] = in ? ld_stream(wrow1 + kk) : z;
          B0[i] = in ? ld_stream(wrow0 + kk + 64) : z;
          B1[i] = in ? ld_stream(wrow1 + kk + 64) : z;
          X0[i] = in && my_r >= 0 ? __ldg(reinterpret_cast<const uint4*>(xrow + kk)) : z;
          X1[i] = in && my_r >= 0 ? __ldg(reinterpret_cast<const uint4*>(xrow + kk + 64)) : z;
        }
#pragma unroll
        for (int i = 0; i < NB; ++i) {
          const int kk = kb0 + 128 * i;
          if (kk < kend) {
            float cb[4] = {0.f, 0.f, 0.f, 0.f};
            mma_k64(cb, A0[i], A1[i], X0[i]);
            mma_k64(cb, B0[i], B1[i], X1[i]);
            const int kb = kk / 128;
            const float w_s = __ldg(sw + kb);
            const float s0 = w_s * __ldg(a.sx + static_cast<size_t>(t0) * ng + kb);
            const float s1 = w_s * __ldg(a.sx + static_cast<size_t>(t1) * ng + kb);
            c[0] = fmaf(cb[0], s0, c[0]);
            c[1] = fmaf(cb[1], s1, c[1]);
            c[2] = fmaf(cb[2], s0, c[2]);
            c[3] = fmaf(cb[3], s1, c[3]);
          }
        }
      }
    }
    // c0: (row, col 2tig), c1: (row, col 2tig+1), c2/c3: row + 8
    float* part = a.part + static_cast<size_t>(s) * a.R * twoI;
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      const int col = 2 * tig + i;
      if (col < nn) {
        const int r = uv.routes()[r_beg + n0 + col];
        part[static_cast<size_t>(r) * twoI + row] = c[i];
        part[static_cast<size_t>(r) * twoI + row + 8] = c[2 + i];
      }
    }
  }
}

// Sum of the K-split partials of (route r, column i) and of (r, I + i); the
// split loads are issued 8 at a time before they are added, in split order.
__device__ __forceinline__ void sum_splits(const float* part, int splits, int R, int twoI, int I, int r, int i,
                                           float& g, float& u) {
  g = 0.f;
  u = 0.f;
  for (int s0 = 0; s0 < splits; s0 += 8) {
    float gv[8], uv[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int s = s0 + j < splits ? s0 + j : 0;
      const float* pp = part + (static_cast<size_t>(s) * R + r) * twoI;
      gv[j] = pp[i];
      uv[j] = pp[I + i];
    }
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      if (s0 + j < splits) {
        g += gv[j];
        u += uv[j];
      }
    }
  }
}

// ------------------------------------------------------------------ rd_reduce
// per-tensor: one thread per (route, i); blockwise: one warp per (route, 128-column group).
__global__ void __launch_bounds__(256) rd_reduce_tensor_kernel(DecodeArgs a) {
  pdl_trigger();
  pdl_wait();
  const int idx = blockIdx.x * blockDim.x + threadIdx.x;
  const int I = a.I, twoI = 2 * I;
  float av = 0.0f;
  if (idx < a.R * I) {
    const int r = idx / I, i = idx - (idx / I) * I;
    float g, u;
    sum_splits(a.part, a.splits, a.R, twoI, I, r, i, g, u);
    const float sc = a.sx[0] * __ldg(a.w1_scale + a.ids[r]);
    av = silu_mul(sc * g, sc * u);
    static_cast<float*>(a.act)[idx] = av;
  }
  const float m = warp_max(fabsf(av));
  if ((threadIdx.x & 31) == 0 && m > 0.0f) atomicMax(&a.hdr->amax_h, __float_as_uint(m));
}

__global__ void __launch_bounds__(256) rd_reduce_block_kernel(DecodeArgs a) {
  pdl_trigger();
  pdl_wait();
  const int gw = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  const int I = a.I, twoI = 2 * I, ngi = I / 128;
  if (gw >= a.R * ngi) return;
  const int r = gw / ngi, G = gw - (gw / ngi) * ngi;
  float av[4];
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const int i = G * 128 + lane * 4 + q;
    float g, u;
    sum_splits(a.part, a.splits, a.R, twoI, I, r, i, g, u);
    av[q] = silu_mul(g, u);
  }
  float m = fmaxf(fmaxf(fabsf(av[0]), fabsf(av[1])), fmaxf(fabsf(av[2]), fabsf(av[3])));
  m = warp_max(m);
  const float sc = e4m3_scale(m);
  const uint32_t q = static_cast<uint32_t>(cvt_e4m3x2(av[0] / sc, av[1] / sc)) |
                     (static_cast<uint32_t>(cvt_e4m3x2(av[2] / sc, av[3] / sc)) << 16);
  *reinterpret_cast<uint32_t*>(static_cast<uint8_t*>(a.act) + static_cast<size_t>(r) * I + G * 128 + lane * 4) = q;
  if (lane == 0) a.sh[static_cast<size_t>(r) * ngi + G] = sc;
}

// ------------------------------------------------------------------ rd_down
// grid = maxU * nHB; block = 128 threads (4 warps x 16 rows of W2[e]); K = I whole.
template <bool BLOCKWISE>
__global__ void __launch_bounds__(THREADS) rd_down_kernel(DecodeArgs a, int nHB) {
  pdl_trigger();
  pdl_wait();
  extern __shared__ uint8_t s_h[];  // [8][I] e4m3 of the current 8 routes, then [8][I/128] fp32 scales
  const int hb = blockIdx.x % nHB;
  const int u = blockIdx.x / nHB;
  UniqView uv{a.uniq, max_uniq(a.R, a.E)};
  if (u >= uv.U()[0]) return;
  const int e = uv.expert()[u];
  const int r_beg = uv.off()[u], cnt = uv.off()[u + 1] - r_beg;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, tig = lane & 3;
  const int I = a.I, H = a.H, ngi = I / 128;
  float* s_sc = reinterpret_cast<float*>(s_h + 8 * I);
  const int row = hb * ROWS_PER_CTA + warp * 16 + g;  // rows row and row+8 of W2[e] (output columns)
  const uint8_t* wrow0 = a.w2 + (static_cast<size_t>(e) * H + row) * I + 16 * tig;
  const uint8_t* wrow1 = wrow0 + static_cast<size_t>(8) * I;
  const float amax_h = __uint_as_float(a.hdr->amax_h);
  const float s_h_t = e4m3_scale(amax_h);

  for (int n0 = 0; n0 < cnt; n0 += 8) {
    const int nn = min(8, cnt - n0);
    __syncthreads();
    // stage the e4m3 h of these routes (zero rows for unused columns)
    for (int i = threadIdx.x; i < 8 * I / 4; i += THREADS) {
      const int n = (i * 4) / I, c = (i * 4) - n * I;
      uint32_t q = 0;
      if (n < nn) {
        const int r = uv.routes()[r_beg + n0 + n];
        if (BLOCKWISE) {
          q = *reinterpret_cast<const uint32_t*>(static_cast<const uint8_t*>(a.act) + static_cast<size_t>(r) * I + c);
        } else {
          const float4 v = *reinterpret_cast<const float4*>(static_cast<const float*>(a.act) + static_cast<size_t>(r) * I + c);
          q = static_cast<uint32_t>(cvt_e4m3x2(v.x / s_h_t, v.y / s_h_t)) |
              (static_cast<uint32_t>(cvt_e4m3x2(v.z / s_h_t, v.w / s_h_t)) << 16);
        }
      }
      *reinterpret_cast<uint32_t*>(s_h + n * I + c) = q;
    }
    if (BLOCKWISE) {
      for (int i = threadIdx.x; i < 8 * ngi; i += THREADS) {
        const int n = i / ngi, G = i - (i / ngi) * ngi;
        s_sc[i] = n < nn ? a.sh[static_cast<size_t>(uv.routes()[r_beg + n0 + n]) * ngi + G] : 0.0f;
      }
    }
    __syncthreads();
    const uint8_t* xrow = s_h + g * I + 16 * tig;
    float c[4] = {0.f, 0.f, 0.f, 0.f};
    if (!BLOCKWISE) {
      constexpr int NB = 8;  // K-steps whose weight loads are issued before their MMAs
      for (int kb0 = 0; kb0 < I; kb0 += 64 * NB) {
        uint4 A0[NB], A1[NB];
#pragma unroll
        for (int i = 0; i < NB; ++i) {
          const int kk = kb0 + 64 * i;
          A0[i] = kk < I ? ld_stream(wrow0 + kk) : make_uint4(0, 0, 0, 0);
          A1[i] = kk < I ? ld_stream(wrow1 + kk) : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int i = 0; i < NB; ++i) {
          const int kk = kb0 + 64 * i;
          if (kk < I) mma_k64(c, A0[i], A1[i], *reinterpret_cast<const uint4*>(xrow + kk));
        }
      }
      const float sc = s_h_t * __ldg(a.w2_scale + e);
#pragma unroll
      for (int i = 0; i < 4; ++i) c[i] *= sc;
    } else {
      const float* sw = a.w2_scale + (static_cast<size_t>(e) * (H / 128) + row / 128) * ngi;
      constexpr int NB = 4;  // 128-wide K blocks per batch of loads
      for (int kb0 = 0; kb0 < I; kb0 += 128 * NB) {
        uint4 A0[NB], A1[NB], B0[NB], B1[NB];
#pragma unroll
        for (int i = 0; i < NB; ++i) {
          const int kk = kb0 + 128 * i;
          const bool in = kk < I;
          const uint4 z = make_uint4(0, 0, 0, 0);
          A0[i] = in ? ld_stream(wrow0 + kk) : z;
          A1[i] = in ? ld_stream(wrow1 + kk) : z;
          B0[i] = in ? ld_stream(wrow0 + kk + 64) : z;
          B1[i] = in ? ld_stream(wrow1 + kk + 64) : z;
        }
#pragma unroll
        for (int i = 0; i < NB; ++i) {
          const int kk = kb0 + 128 * i;
          if (kk < I) {
            float cb[4] = {0.f, 0.f, 0.f, 0.f};
            mma_k64(cb, A0[i], A1[i], *reinterpret_cast<const uint4*>(xrow + kk));
            mma_k64(cb, B0[i], B1[i], *reinterpret_cast<const uint4*>(xrow + kk + 64));
            const int kb = kk / 128;
            const float w_s = __ldg(sw + kb);
            const float s0 = w_s * s_sc[(2 * tig) * ngi + kb];
            const float s1 = w_s * s_sc[(2 * tig + 1) * ngi + kb];
            c[0] = fmaf(cb[0], s0, c[0]);
            c[1] = fmaf(cb[1], s1, c[1]);
            c[2] = fmaf(cb[2], s0, c[2]);
            c[3] = fmaf(cb[3], s1, c[3]);
          }
        }
      }
    }
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      const int col = 2 * tig + i;
      if (col < nn) {
        const int r = uv.routes()[r_beg + n0 + col];
        a.o[static_cast<size_t>(r) * H + row] = c[i];
        a.o[static_cast<size_t>(r) * H + row + 8] = c[2 + i];
      }
    }
  }
}

}  // namespace rd

size_t route_direct_uniq_bytes(int T, int E, int k) {
  const int R = T * k;
  const int mu = rd::max_uniq(R, E);
  return static_cast<size_t>(2 + 2 * mu + R) * sizeof(int32_t);
}

cudaError_t launch_route_direct(const DecodeArgs& a, cudaStream_t s) {
  using namespace rd;
  if (a.T <= 0) return cudaSuccess;
  int maxv = 1;
  while (maxv * 32 < a.E) maxv *= 2;
  stage_begin("rd_prep", s);
  switch (maxv) {
    case 1: rd_prep_kernel<1><<<1, 1024, 0, s>>>(a); break;
    case 2: rd_prep_kernel<2><<<1, 1024, 0, s>>>(a); break;
    case 4: rd_prep_kernel<4><<<1, 1024, 0, s>>>(a); break;
    case 8: rd_prep_kernel<8><<<1, 1024, 0, s>>>(a); break;
    default: rd_prep_kernel<16><<<1, 1024, 0, s>>>(a); break;
  }
  cudaError_t err = cudaGetLastError();
  stage_end(s);
  if (err != cudaSuccess) return err;

  const int maxU = max_uniq(a.R, a.E);
  const bool bw = a.quant == MOE_FP8_BLOCK128;
  cudaLaunchAttribute pdl[1];
  pdl[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  pdl[0].val.programmaticStreamSerializationAllowed = 1;
  auto config = [&](unsigned grid, unsigned block, size_t smem) {
    cudaLaunchConfig_t c{};
    c.gridDim = dim3(grid);
    c.blockDim = dim3(block);
    c.dynamicSmemBytes = smem;
    c.stream = s;
    c.attrs = pdl;
    c.numAttrs = 1;
    return c;
  };

  const int nMB = 2 * a.I / ROWS_PER_CTA;
  stage_begin("rd_gateup", s);
  {
    const cudaLaunchConfig_t c = config(maxU * nMB * a.splits, THREADS, 0);
    err = bw ? cudaLaunchKernelEx(&c, rd_gateup_kernel<true>, a, nMB, a.splits)
             : cudaLaunchKernelEx(&c, rd_gateup_kernel<false>, a, nMB, a.splits);
  }
  stage_end(s);
  if (err != cudaSuccess) return err;

  stage_begin("rd_reduce", s);
  if (bw) {
    const int warps = a.R * (a.I / 128);
    const cudaLaunchConfig_t c = config((warps * 32 + 255) / 256, 256, 0);
    err = cudaLaunchKernelEx(&c, rd_reduce_block_kernel, a);
  } else {
    const cudaLaunchConfig_t c = config((a.R * a.I + 255) / 256, 256, 0);
    err = cudaLaunchKernelEx(&c, rd_reduce_tensor_kernel, a);
  }
  stage_end(s);
  if (err != cudaSuccess) return err;

  const int nHB = a.H / ROWS_PER_CTA;
  const size_t smem = static_cast<size_t>(8) * a.I + 8 * (a.I / 128 + 1) * sizeof(float) + 16;
  stage_begin("rd_down", s);
  {
    const cudaLaunchConfig_t c = config(maxU * nHB, THREADS, smem);
    err = bw ? cudaLaunchKernelEx(&c, rd_down_kernel<true>, a, nHB) : cudaLaunchKernelEx(&c, rd_down_kernel<false>, a, nHB);
  }
  stage_end(s);
  return err;
}

}  // namespace moe
