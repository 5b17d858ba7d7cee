// Top-k routing, index shuffling and the grouped-GEMM tile map.
//
// Routing: one warp per token (routing.cuh).  For the per-tensor FP8 forward the
// route/rank launch also carries extra blocks that record the amax of x.
//
// Shuffle (index_shuffling of "Port necessary FBGEMM MoE kernels"; the
// counting, sorting and task-map steps of the route-MMA page's Motivation), in
// three launches with no device-to-host copy:
//   1. route_rank: per block of <= 1024 consecutive routes, the rank of each
//      route among the block's earlier routes of the same expert (warp
//      match_any + per-warp running histograms), and the block's per-expert
//      counts.  Ranks follow route order, which makes the sort stable.
//   2. scan_tiles (one block): counts = column sums of the block counts,
//      offsets = their exclusive prefix, per-block base = offsets + the
//      exclusive prefix over earlier blocks; then the tile map.
//   3. scatter: perm[base + rank] = r, inv[r] = base + rank.
#include "common.cuh"
#include "internal.h"
#include "routing.cuh"

namespace moe {

constexpr int kScanSmemBytes = 192 * 1024;  // block-count matrix staged in shared memory up to this size

// Ranking phase of the route/rank kernel (s_ids holds the block's nr expert ids).
__device__ __forceinline__ void rank_block(int* s_ids, int* s_lr, int* hist, int E, int RB, int nr, size_t r0, int blk,
                                           int32_t* __restrict__ lrank, int32_t* __restrict__ blockcounts,
                                           DeviceHeader* hdr) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  constexpr int NW = kRouteThreads / 32;
  for (int i = tid; i < NW * E; i += kRouteThreads) hist[i] = 0;
  __syncthreads();

  // each warp ranks a contiguous segment of the block's routes, 32 at a time, in order
  const int seg = (RB + NW * 32 - 1) / (NW * 32) * 32;
  int* my_hist = hist + warp * E;
  for (int c = 0; c < seg; c += 32) {
    const int rl = warp * seg + c + lane;
    const bool valid = rl < nr;
    const int e = valid ? s_ids[rl] : -1;
    const bool ok = valid && e >= 0 && e < E;
    if (valid && !ok) record_status(hdr, kStatusBounds, static_cast<unsigned int>(r0 + rl));
    const int keyv = ok ? e : -1 - lane;  // invalid lanes match only themselves
    const unsigned peers = __match_any_sync(0xffffffffu, keyv);
    const int rank = __popc(peers & ((1u << lane) - 1u));
    const int base = ok ? my_hist[e] : 0;
    __syncwarp();
    if (ok && rank == 0) my_hist[e] = base + __popc(peers);
    __syncwarp();
    if (valid) s_lr[rl] = ok ? base + rank : -1;
  }
  __syncthreads();
  for (int e = tid; e < E; e += kRouteThreads) {
    int run = 0;
#pragma unroll
    for (int w = 0; w < NW; ++w) {
      const int c = hist[w * E + e];
      hist[w * E + e] = run;
      run += c;
    }
    blockcounts[static_cast<size_t>(blk) * E + e] = run;
  }
  __syncthreads();
  for (int rl = tid; rl < nr; rl += kRouteThreads) {
    int lr = s_lr[rl];
    if (lr >= 0) lr += hist[(rl / seg) * E + s_ids[rl]];
    lrank[r0 + rl] = lr;
  }
}

// Per-tensor amax of x (bf16, n8 pieces of 8 values) by `nb` blocks, block b of
// them here: eight 16-byte loads in flight per thread, one atomic per block.
__device__ void amax_blocks(const uint4* __restrict__ x, size_t n8, int b, int nb, DeviceHeader* hdr) {
  __shared__ float s_m[kRouteThreads / 32];
  float m = 0.0f;
  const size_t stride = static_cast<size_t>(nb) * blockDim.x;
  for (size_t base = b * static_cast<size_t>(blockDim.x) + threadIdx.x; base < n8; base += stride * 8) {
    uint4 v[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const size_t i = base + j * stride;
      v[j] = i < n8 ? __ldg(x + i) : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const __nv_bfloat162* h2 = reinterpret_cast<const __nv_bfloat162*>(&v[j]);
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const float2 f = __bfloat1622float2(h2[q]);
        m = fmaxf(m, fmaxf(fabsf(f.x), fabsf(f.y)));
      }
    }
  }
  m = warp_max(m);
  if ((threadIdx.x & 31) == 0) s_m[threadIdx.x >> 5] = m;
  __syncthreads();
  if (threadIdx.x < 32) {
    m = threadIdx.x < (blockDim.x >> 5) ? s_m[threadIdx.x] : 0.0f;
    m = warp_max(m);
    if (threadIdx.x == 0 && m > 0.0f) atomicMax(&hdr->amax_x, __float_as_uint(m));
  }
}

template <int MAXV, bool ROUTE, bool RANK>
__global__ void __launch_bounds__(kRouteThreads) route_rank_kernel(
    const float* __restrict__ scores, const int32_t* __restrict__ ids_in, int T, int E, int k, int TB,
    int32_t* __restrict__ ids_out, float* __restrict__ w_out, int32_t* __restrict__ lrank,
    int32_t* __restrict__ blockcounts, DeviceHeader* hdr, const uint4* __restrict__ amax_x, size_t amax_n8,
    int nblk) {
  // blocks past the nblk routing blocks compute the per-tensor amax of x (FP8)
  // alongside them: it depends on nothing the routing produces
  if (static_cast<int>(blockIdx.x) >= nblk) {
    amax_blocks(amax_x, amax_n8, static_cast<int>(blockIdx.x) - nblk, static_cast<int>(gridDim.x) - nblk, hdr);
    return;
  }
  extern __shared__ int smem[];
  int* s_ids = smem;                          // [1024]
  int* s_lr = smem + kMaxRoutesPerBlock;      // [1024]
  int* hist = smem + 2 * kMaxRoutesPerBlock;  // [warps][E]
  const int tid = threadIdx.x, warp = tid >> 5;
  const int blk = blockIdx.x;
  const int t0 = blk * TB;
  const int nt = min(TB, T - t0);
  const int nr = nt * k;
  const size_t r0 = static_cast<size_t>(t0) * k;

  if (ROUTE) {
    // each warp routes every NW-th token of the block; the next token's scores are
    // loaded while the current one is being routed
    constexpr int NW = kRouteThreads / 32;
    float cur[MAXV], nxt[MAXV];
    if (warp < nt) load_scores<MAXV>(scores + static_cast<size_t>(t0 + warp) * E, E, cur);
    for (int tb = warp; tb < nt; tb += NW) {
      if (tb + NW < nt) load_scores<MAXV>(scores + static_cast<size_t>(t0 + tb + NW) * E, E, nxt);
      const size_t t = static_cast<size_t>(t0 + tb);
      route_values<MAXV>(cur, E, k, ids_out + t * k, w_out + t * k, RANK ? s_ids + tb * k : nullptr);
#pragma unroll
      for (int i = 0; i < MAXV; ++i) cur[i] = nxt[i];
    }
  } else {
    for (int i = tid; i < nr; i += kRouteThreads) s_ids[i] = ids_in[r0 + i];
  }
  if constexpr (RANK) rank_block(s_ids, s_lr, hist, E, TB * k, nr, r0, blk, lrank, blockcounts, hdr);
}

// Exclusive prefix of s_cnt (E <= 512) by warp 0 into s_off, and of the tile
// counts ceil(c/BM) into s_toff; entries [E] hold the totals.
__device__ __forceinline__ void scan_counts_warp0(const int* s_cnt, int E, int BM, int* s_off, int* s_toff) {
  if ((threadIdx.x >> 5) != 0) return;
  const int lane = threadIdx.x & 31;
  const int per = (E + 31) / 32;
  int a = 0, b = 0;
  for (int i = 0; i < per; ++i) {
    const int e = lane * per + i;
    if (e < E) {
      a += s_cnt[e];
      b += (s_cnt[e] + BM - 1) / BM;
    }
  }
  int ia = a, ib = b;  // inclusive warp scan
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int xa = __shfl_up_sync(0xffffffffu, ia, o);
    const int xb = __shfl_up_sync(0xffffffffu, ib, o);
    if (lane >= o) {
      ia += xa;
      ib += xb;
    }
  }
  int ra = ia - a, rb = ib - b;
  for (int i = 0; i < per; ++i) {
    const int e = lane * per + i;
    if (e < E) {
      s_off[e] = ra;
      s_toff[e] = rb;
      ra += s_cnt[e];
      rb += (s_cnt[e] + BM - 1) / BM;
    }
  }
  if (lane == 31) {
    s_off[E] = ia;
    s_toff[E] = ib;
  }
}

// `extra` tiles follow the routed experts' (the shared experts' tiles, written by the caller).
__device__ __forceinline__ void emit_tiles(const int* s_cnt, const int* s_off, const int* s_toff, int E, int BM,
                                           int32_t* tiles, int32_t* num_tiles, int max_tiles, DeviceHeader* hdr,
                                           int extra = 0) {
  for (int e = threadIdx.x >> 5; e < E; e += blockDim.x >> 5) {
    const int c = s_cnt[e];
    const int nt = (c + BM - 1) / BM;
    for (int j = threadIdx.x & 31; j < nt; j += 32) {
      const int idx = s_toff[e] + j;
      if (idx < max_tiles) {
        int4 t;
        t.x = e;
        t.y = s_off[e] + j * BM;
        t.z = min(BM, c - j * BM);
        t.w = 0;
        reinterpret_cast<int4*>(tiles)[idx] = t;
      }
    }
  }
  if (threadIdx.x == 0) {
    *num_tiles = s_toff[E] + extra;
    if (s_toff[E] + extra > max_tiles) record_status(hdr, kStatusBounds, 0x7100000u);
  }
}

// The block-count matrix is first copied into shared memory with independent,
// coalesced loads (when it fits), so that the per-expert column scans run on
// shared memory instead of a chain of dependent global loads.
__global__ void __launch_bounds__(1024) scan_tiles_kernel(int32_t* __restrict__ bc, int nblk, int E,
                                                          int32_t* __restrict__ counts, int32_t* __restrict__ offsets,
                                                          int32_t* __restrict__ tiles, int32_t* __restrict__ num_tiles,
                                                          int max_tiles, int BM, DeviceHeader* hdr, int use_smem,
                                                          int T, int S, int Rr, int32_t* __restrict__ padbase) {
  __shared__ int s_cnt[kMaxE], s_off[kMaxE + 1], s_toff[kMaxE + 1];
  extern __shared__ int sbc[];
  dep_wait();  // the block counts of the route/rank kernel
  const int n = nblk * E;
  int* col = use_smem ? sbc : bc;
  if (use_smem) {
#pragma unroll 8
    for (int i = threadIdx.x; i < n; i += blockDim.x) sbc[i] = bc[i];
    __syncthreads();
  }
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    int run = 0;
    for (int b = 0; b < nblk; ++b) {
      const int c = col[b * E + e];
      col[b * E + e] = run;
      run += c;
    }
    s_cnt[e] = run;
  }
  __syncthreads();
  scan_counts_warp0(s_cnt, E, BM, s_off, s_toff);
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    counts[e] = s_cnt[e];
    offsets[e] = s_off[e];
  }
  if (threadIdx.x == 0) offsets[E] = s_off[E];
  for (int i = threadIdx.x; i < n; i += blockDim.x) bc[i] = col[i] + s_off[i % E];
  if (!tiles) return;
  // shared expert s is expert E + s of the tile map: every token, rows [Rr + s*T, Rr + (s+1)*T)
  const int nts = (T + BM - 1) / BM;
  emit_tiles(s_cnt, s_off, s_toff, E, BM, tiles, num_tiles, max_tiles, hdr, S * nts);
  for (int i = threadIdx.x; i < S * nts; i += blockDim.x) {
    const int sx = i / nts, j = i - sx * nts;
    const int idx = s_toff[E] + i;
    if (idx < max_tiles)
      reinterpret_cast<int4*>(tiles)[idx] = make_int4(E + sx, Rr + sx * T + j * BM, min(BM, T - j * BM), 0);
  }
  // row p of expert e (or shared expert s) sits at row p + padbase[e] of a layout in
  // which every expert's rows are padded to whole tiles (the blocked MX scales)
  if (padbase) {
    for (int e = threadIdx.x; e < E; e += blockDim.x) padbase[e] = BM * s_toff[e] - s_off[e];
    for (int sx = threadIdx.x; sx < S; sx += blockDim.x) padbase[E + sx] = BM * (s_toff[E] + sx * nts) - (Rr + sx * T);
  }
}

__global__ void __launch_bounds__(1024) tile_map_kernel(const int32_t* __restrict__ counts, int E, int BM,
                                                        int32_t* __restrict__ tiles, int32_t* __restrict__ num_tiles,
                                                        int max_tiles, DeviceHeader* hdr) {
  __shared__ int s_cnt[kMaxE], s_off[kMaxE + 1], s_toff[kMaxE + 1];
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    const int c = counts[e];
    if (c < 0) record_status(hdr, kStatusBounds, 0x7200000u | e);
    s_cnt[e] = c < 0 ? 0 : c;
  }
  __syncthreads();
  scan_counts_warp0(s_cnt, E, BM, s_off, s_toff);
  __syncthreads();
  emit_tiles(s_cnt, s_off, s_toff, E, BM, tiles, num_tiles, max_tiles, hdr);
}

__global__ void scatter_kernel(const int32_t* __restrict__ ids, const int32_t* __restrict__ lrank,
                               const int32_t* __restrict__ blockbase, int R, int E, int RB,
                               int32_t* __restrict__ perm, int32_t* __restrict__ inv) {
  const int r = blockIdx.x * blockDim.x + threadIdx.x;
  if (r >= R) return;
  const int lr = lrank[r];
  if (lr < 0) {
    inv[r] = -1;
    return;
  }
  const int e = ids[r];
  const int p = blockbase[static_cast<size_t>(r / RB) * E + e] + lr;
  perm[p] = r;
  inv[r] = p;
}

// Scatter fused with the gather of the activations, one block per token: the
// block first places the token's k routes (perm/inv like scatter_kernel), then
// reads the token's x row once, one 16-byte piece per thread and pass, and
// stores each piece to the sorted row p of every route, so the Gate/Up GEMM
// reads its A tiles as plain contiguous boxes and x is read from DRAM once.
__global__ void __launch_bounds__(256) scatter_gather_kernel(const int32_t* __restrict__ ids,
                                                             const int32_t* __restrict__ lrank,
                                                             const int32_t* __restrict__ blockbase, int E, int RB,
                                                             int k, int H, const uint4* __restrict__ x,
                                                             uint4* __restrict__ xs, int32_t* __restrict__ perm,
                                                             int32_t* __restrict__ inv, int S, int T) {
  __shared__ int s_p[kMaxK + kMaxShared];
  dep_wait();  // ranks and block bases of the kernels before
  const int t = blockIdx.x;
  for (int j = threadIdx.x; j < k; j += blockDim.x) {
    const int r = t * k + j;
    const int lr = lrank[r];
    int p = -1;
    if (lr >= 0) {
      p = blockbase[static_cast<size_t>(r / RB) * E + ids[r]] + lr;
      perm[p] = r;
    }
    inv[r] = p;
    s_p[j] = p;
  }
  // the token's row of each shared expert: T*k + s*T + t
  for (int j = threadIdx.x; j < S; j += blockDim.x) s_p[k + j] = T * k + j * T + t;
  __syncthreads();
  const int row16 = H / 8;  // 16-byte pieces per row
  const int nrow = k + S;
  const uint4* src = x + static_cast<size_t>(t) * row16;
  for (int c = threadIdx.x; c < row16; c += blockDim.x) {
    const uint4 v = __ldg(src + c);
    for (int j = 0; j < nrow; ++j) {
      const int p = s_p[j];
      if (p >= 0) xs[static_cast<size_t>(p) * row16 + c] = v;
    }
  }
}

// ------------------------------------------------------------------ launchers
// Shared memory of the route/rank kernel: the block's ids and ranks plus one
// histogram of E counters per warp (up to 72 KB at E = 512).
constexpr size_t kRouteSmemMax = (2 * kMaxRoutesPerBlock + (kRouteThreads / 32) * kMaxE) * sizeof(int);

template <int V, bool ROUTE, bool RANK>
static cudaError_t rr_smem_attr() {
  static const cudaError_t st = cudaFuncSetAttribute(route_rank_kernel<V, ROUTE, RANK>,
                                                     cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                     static_cast<int>(kRouteSmemMax));
  return st;
}

template <bool ROUTE, bool RANK>
static cudaError_t launch_rr(int maxv, dim3 grid, size_t smem, cudaStream_t s, const float* scores,
                             const int32_t* ids_in, int T, int E, int k, int TB, int32_t* ids_out, float* w_out,
                             int32_t* lrank, int32_t* bc, DeviceHeader* hdr, const uint4* ax, size_t an8, int nblk) {
#define MOE_RR(V)                                                                                          \
  if (const cudaError_t ae = rr_smem_attr<V, ROUTE, RANK>()) return ae;                                    \
  route_rank_kernel<V, ROUTE, RANK><<<grid, kRouteThreads, smem, s>>>(scores, ids_in, T, E, k, TB, ids_out, \
                                                                     w_out, lrank, bc, hdr, ax, an8, nblk)
  switch (maxv) {
    case 1: MOE_RR(1); break;
    case 2: MOE_RR(2); break;
    case 4: MOE_RR(4); break;
    case 8: MOE_RR(8); break;
    default: MOE_RR(16); break;
  }
#undef MOE_RR
  return cudaGetLastError();
}

cudaError_t launch_route_rank(const float* scores, const int32_t* ids_in, int T, int E, int k, int32_t* ids_out,
                              float* w_out, int32_t* lrank, int32_t* blockcounts, DeviceHeader* hdr, bool route,
                              bool rank, cudaStream_t s, const void* amax_x, size_t amax_n) {
  if (T <= 0) return cudaSuccess;
  const int TB = route_tokens_per_block(k);
  const int nblk = (T + TB - 1) / TB;
  const size_t smem = (2 * kMaxRoutesPerBlock + (kRouteThreads / 32) * E) * sizeof(int);
  int maxv = 1;
  while (maxv * 32 < E) maxv *= 2;
  // amax of x: one extra block per SM; they start on the SMs the routing blocks
  // leave free and take the others as the routing finishes
  const size_t an8 = amax_x ? amax_n / 8 : 0;
  const int nam = an8 > 0 ? (num_sms() > 0 ? num_sms() : 148) : 0;
  const dim3 grid(nblk + nam);
  const uint4* ax = static_cast<const uint4*>(amax_x);
  stage_begin("route_rank", s);
  cudaError_t err;
  if (route && rank) err = launch_rr<true, true>(maxv, grid, smem, s, scores, ids_in, T, E, k, TB, ids_out, w_out, lrank, blockcounts, hdr, ax, an8, nblk);
  else if (route) err = launch_rr<true, false>(maxv, grid, smem, s, scores, ids_in, T, E, k, TB, ids_out, w_out, lrank, blockcounts, hdr, ax, an8, nblk);
  else err = launch_rr<false, true>(maxv, grid, smem, s, scores, ids_in, T, E, k, TB, ids_out, w_out, lrank, blockcounts, hdr, ax, an8, nblk);
  stage_end(s);
  return err;
}

cudaError_t launch_scan_tiles(int32_t* blockcounts, int nblk, int E, int32_t* counts, int32_t* offsets,
                              int32_t* tiles, int32_t* num_tiles, int max_tiles, int BM, int32_t* /*tile_scratch*/,
                              DeviceHeader* hdr, cudaStream_t s, int T, int S, int Rr, int32_t* padbase) {
  static const cudaError_t attr = cudaFuncSetAttribute(scan_tiles_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                       kScanSmemBytes);
  if (attr != cudaSuccess) return attr;
  const size_t need = static_cast<size_t>(nblk) * E * sizeof(int);
  const int use_smem = need <= static_cast<size_t>(kScanSmemBytes) ? 1 : 0;
  stage_begin("scan_tiles", s);
  const cudaError_t err = launch_dependent(scan_tiles_kernel, dim3(1), dim3(1024), use_smem ? need : 0, s, blockcounts,
                                           nblk, E, counts, offsets, tiles, num_tiles, max_tiles, BM, hdr, use_smem, T,
                                           S, Rr, padbase);
  stage_end(s);
  return err;
}

cudaError_t launch_scatter(const int32_t* ids, const int32_t* lrank, const int32_t* blockbase, int T, int E, int k,
                           int32_t* perm, int32_t* inv, cudaStream_t s) {
  const int R = T * k;
  if (R <= 0) return cudaSuccess;
  const int RB = route_tokens_per_block(k) * k;
  stage_begin("scatter", s);
  scatter_kernel<<<(R + 255) / 256, 256, 0, s>>>(ids, lrank, blockbase, R, E, RB, perm, inv);
  const cudaError_t err = cudaGetLastError();
  stage_end(s);
  return err;
}

cudaError_t launch_scatter_gather(const int32_t* ids, const int32_t* lrank, const int32_t* blockbase, int T, int E,
                                  int k, int H, const void* x, void* xs, int32_t* perm, int32_t* inv,
                                  cudaStream_t s, int S) {
  if (T <= 0) return cudaSuccess;
  const int RB = route_tokens_per_block(k) * k;
  stage_begin("scatter_gather", s);
  const cudaError_t err = launch_dependent(scatter_gather_kernel, dim3(T), dim3(256), 0, s, ids, lrank, blockbase, E, RB,
                                           k, H, static_cast<const uint4*>(x), static_cast<uint4*>(xs), perm, inv, S, T);
  stage_end(s);
  return err;
}

cudaError_t launch_tile_map(const int32_t* counts, int E, int BM, int32_t* tiles, int32_t* num_tiles, int max_tiles,
                            int32_t* /*tile_scratch*/, DeviceHeader* hdr, cudaStream_t s) {
  stage_begin("tile_map", s);
  tile_map_kernel<<<1, 1024, 0, s>>>(counts, E, BM, tiles, num_tiles, max_tiles, hdr);
  const cudaError_t err = cudaGetLastError();
  stage_end(s);
  return err;
}

cudaError_t launch_reset_header(DeviceHeader* hdr, cudaStream_t s) {
  stage_begin("header_reset", s);
  const cudaError_t err = cudaMemsetAsync(hdr, 0, sizeof(DeviceHeader), s);
  stage_end(s);
  return err;
}

}  // namespace moe
