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
//               of x (per tensor, or per token and 128 columns), and the table of distinct selected
//               experts in first-use order with their routes (a route-order
//               scan of at most 1024 routes, no sort), so an expert chosen by
//               several tokens is streamed once, cut into column groups of up
//               to 8 routes; plus prefetch CTAs that repeat the routing and
//               start the selected experts' W1 on its way into L2.
//   rd_gateup   persistent, two CTAs per SM over work items (column group, K
//               split, 64 rows of W1[e]): a producer warp streams the rows with
//               TMA into a ring of shared-memory stages; four consumer warps
//               stage the group's e4m3 x slice when the group changes and feed
//               16 weight rows each into mma.sync m16n8k32 e4m3 (weights on M,
//               the group's routes on N); fp32 partials per split.
//   rd_reduce   sums the K splits, applies the scales and SwiGLU; blockwise
//               mode quantises h per (route, 128 columns) here, per-tensor mode
//               records the global amax of h.
//   rd_down     persistent like rd_gateup over (column group, 64 rows of
//               W2[e]), with 256-byte stages for rows of at most 256 bytes; h of
//               the group's routes is quantised (per-tensor) or copied into
//               shared memory; fp32 o in route order.
//   combine     the contiguous top-k reduction shared with the grouped path.
// All but rd_prep are launched as programmatic dependents of their predecessor.
//
// K permutation: a dot product does not depend on the order of its terms, so
// each thread loads 16 consecutive bytes of a weight row and of x and feeds
// bytes 0-7 to one m16n8k32 and bytes 8-15 to the next; A and B use the same
// assignment, which is what makes it exact.
#include <mutex>

#include "common.cuh"
#include "internal.h"
#include "routing.cuh"

namespace moe {
namespace rd {

constexpr int ROWS_PER_CTA = 64;  // weight rows per work item: 4 consumer warps x 16 rows
constexpr int CONSUMERS = 4;      // consumer warps (warps 0-3); warp 4 is the copy producer
constexpr int THREADS = 32 * (CONSUMERS + 1);
constexpr int NS = 3;             // weight stages in flight per CTA (96 KB; two CTAs per SM)
constexpr int CK = 512;           // K bytes of one stage (the last stage of an item may be shorter)
constexpr int BOXK = 128;         // K bytes of one TMA box (64 rows x 128 bytes = 8 KB, 128-byte swizzle)
constexpr int BOX_BYTES = ROWS_PER_CTA * BOXK;
constexpr int STAGE_BYTES = ROWS_PER_CTA * CK;  // CK / BOXK boxes, each [64 rows][128 bytes]
constexpr int GROUP = 8;          // routes per MMA column group (m16n8k32: N = 8)
constexpr double kW2PrefetchBytes = 16.0 * 1024 * 1024;  // W2 prefetched into L2 during Gate/Up
constexpr long long kW1PrefetchBytes = 96ll * 1024 * 1024;  // W1 prefetched into L2 by rd_prep
constexpr uint32_t kPrefetchChunk = 64 * 1024;             // bytes per L2 prefetch instruction
constexpr long long kPrefetchPerCta = 256 * 1024;          // W1 bytes per prefetch CTA of rd_prep

// Table of distinct experts, in int32 words:
//   [0] U;  [1 .. 1+maxU) expert of u;  [1+maxU .. 2+2maxU) CSR offsets of u;
//   [2+2maxU .. 2+2maxU+R) routes of u, in route order;
//   [2+2maxU+R] G = number of column groups (up to 8 routes of one expert);
//   then maxG entries: u of group g, and maxG entries: first route index of g
//   within u's list.
struct UniqView {
  int32_t* base;
  int maxU;
  int R;
  __host__ __device__ int32_t* U() const { return base; }
  __host__ __device__ int32_t* expert() const { return base + 1; }
  __host__ __device__ int32_t* off() const { return base + 1 + maxU; }
  __host__ __device__ int32_t* routes() const { return base + 2 + 2 * maxU; }
  __host__ __device__ int32_t* G() const { return base + 2 + 2 * maxU + R; }
  __host__ __device__ int maxG() const { return maxU + R / GROUP + 1; }
  __host__ __device__ int32_t* gu() const { return base + 3 + 2 * maxU + R; }
  __host__ __device__ int32_t* gn0() const { return gu() + maxG(); }
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
  __shared__ int s_u[kRouteDirectMaxRoutes];    // distinct-expert index of each route
  __shared__ int s_pos[kRouteDirectMaxRoutes];  // position of each route in its expert's list
  __shared__ int s_cnt[kRouteDirectMaxRoutes];  // routes per distinct expert
  __shared__ int s_off[kRouteDirectMaxRoutes];
  __shared__ int s_e2u[kMaxE];
  __shared__ unsigned s_seen[kMaxE / 32];
  __shared__ float s_red[32];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, nwarps = blockDim.x >> 5;
  const int T = a.T, E = a.E, k = a.k, H = a.H, R = a.R;
  pdl_trigger();
  if (blockIdx.x > 0) {
    // W1 prefetch role (every CTA but the first): repeat the routing (scores
    // only, no outputs), list the distinct experts in first-use order as the
    // table below does, and start this CTA's share of their W1 matrices - whole
    // matrices in that order, up to kW1PrefetchBytes in all - on its way into
    // L2, so rd_gateup streams them from L2.  One SM issues bulk prefetches at
    // a few hundred GB/s, hence the spread over many CTAs.
    if (warp == 0)
      for (int i = lane; i < kMaxE / 32; i += 32) s_seen[i] = 0u;
    for (int t = warp; t < T; t += nwarps)
      route_one_token<MAXV>(a.scores + static_cast<size_t>(t) * E, E, k, nullptr, nullptr, s_ids + t * k);
    __syncthreads();
    const long long w1_bytes = 2ll * a.I * H;
    const int maxp = static_cast<int>(kW1PrefetchBytes / w1_bytes < kMaxE ? kW1PrefetchBytes / w1_bytes : kMaxE);
    if (warp == 0) {
      int run = 0;
      for (int c = 0; c < R && run < maxp; c += 32) {
        const int r = c + lane;
        const bool valid = r < R;
        const int e = valid ? s_ids[r] : 0;
        const unsigned peers = __match_any_sync(0xffffffffu, valid ? e : -1 - lane);
        const bool first = valid && lane == __ffs(peers) - 1 && !((s_seen[e >> 5] >> (e & 31)) & 1u);
        const unsigned fb = __ballot_sync(0xffffffffu, first);
        const int n = run + __popc(fb & ((1u << lane) - 1u));
        if (first) {
          if (n < maxp) s_u[n] = e;
          atomicOr(&s_seen[e >> 5], 1u << (e & 31));
        }
        run += __popc(fb);
        __syncwarp();
      }
      if (lane == 0) s_cnt[0] = run < maxp ? run : maxp;
    }
    __syncthreads();
    const int nd = s_cnt[0];
    const long long nch = (w1_bytes + kPrefetchChunk - 1) / kPrefetchChunk;
    const long long npf = gridDim.x - 1;
    for (long long q = (blockIdx.x - 1) + npf * tid; q < nd * nch; q += npf * blockDim.x) {
      const int u = static_cast<int>(q / nch);
      const long long off = (q - u * nch) * kPrefetchChunk;
      const long long left = w1_bytes - off;
      bulk_prefetch_l2(a.w1 + static_cast<size_t>(s_u[u]) * w1_bytes + off,
                       static_cast<uint32_t>(left < kPrefetchChunk ? left : kPrefetchChunk));
    }
    return;
  }
  if (tid == 0) {
    a.hdr->status = 0u;
    a.hdr->info = 0u;
    a.hdr->amax_x = 0u;
    a.hdr->amax_h = 0u;
  }
  // x is quantised by warps 1..31 (NQ threads) while warp 0 builds the expert
  // table; their first batch of x loads goes out before the routing so that both
  // memory round trips overlap.
  constexpr int NQ = 1024 - 32;
  const int tq = tid - 32;
  const int n8 = T * H / 8;  // 16-byte pieces of x (8 values each)
  const uint4* x8 = static_cast<const uint4*>(a.x);
  constexpr int XB = 5;      // pieces per thread per batch
  uint4 xv[XB];
  if (warp > 0) {
#pragma unroll
    for (int j = 0; j < XB; ++j) {
      const int i = tq + j * NQ;
      xv[j] = i < n8 ? __ldg(x8 + i) : make_uint4(0, 0, 0, 0);
    }
  }
  // 1. routing: one warp per token
  for (int t = warp; t < T; t += nwarps)
    route_one_token<MAXV>(a.scores + static_cast<size_t>(t) * E, E, k, a.ids + static_cast<size_t>(t) * k,
                           a.w + static_cast<size_t>(t) * k, s_ids + t * k);
  __syncthreads();
  if (warp == 0) {
    // 2a. distinct experts in first-use order and the routes of each in route
    //     order, by one warp walking the routes 32 at a time: a route is the first
    //     use of its expert if it is the lowest lane of its expert in the chunk and
    //     the expert was not seen in an earlier chunk.
    UniqView uv{a.uniq, max_uniq(R, E), R};
    for (int i = lane; i < kMaxE / 32; i += 32) s_seen[i] = 0u;
    __syncwarp();
    int run = 0;
    for (int c = 0; c < R; c += 32) {
      const int r = c + lane;
      const bool valid = r < R;
      const int e = valid ? s_ids[r] : 0;
      const unsigned peers = __match_any_sync(0xffffffffu, valid ? e : -1 - lane);
      const int leader = __ffs(peers) - 1;
      const bool first = valid && lane == leader && !((s_seen[e >> 5] >> (e & 31)) & 1u);
      const unsigned fb = __ballot_sync(0xffffffffu, first);
      if (first) {
        const int un = run + __popc(fb & ((1u << lane) - 1u));
        s_e2u[e] = un;
        s_cnt[un] = 0;
        uv.expert()[un] = e;
        atomicOr(&s_seen[e >> 5], 1u << (e & 31));
      }
      run += __popc(fb);
      __syncwarp();
      const int u = valid ? s_e2u[e] : 0;
      const int base = valid ? s_cnt[u] : 0;
      __syncwarp();
      if (valid && lane == leader) s_cnt[u] = base + __popc(peers);
      if (valid) {
        s_u[r] = u;
        s_pos[r] = base + __popc(peers & ((1u << lane) - 1u));
      }
      __syncwarp();
    }
    // 2b. CSR offsets of the distinct experts and the table of column groups (up
    //     to 8 routes of one expert each), by warp-wide exclusive scans
    int acc = 0, gacc = 0;
    for (int c = 0; c < run; c += 32) {
      const int u = c + lane;
      const int cnt = u < run ? s_cnt[u] : 0;
      const int ng = (cnt + GROUP - 1) / GROUP;
      int incl = cnt, gincl = ng;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, incl, o);
        const int gv = __shfl_up_sync(0xffffffffu, gincl, o);
        if (lane >= o) {
          incl += v;
          gincl += gv;
        }
      }
      if (u < run) {
        const int off = acc + incl - cnt, g0 = gacc + gincl - ng;
        s_off[u] = off;
        uv.off()[u] = off;
        for (int q = 0; q < ng; ++q) {
          uv.gu()[g0 + q] = u;
          uv.gn0()[g0 + q] = q * GROUP;
        }
      }
      acc += __shfl_sync(0xffffffffu, incl, 31);
      gacc += __shfl_sync(0xffffffffu, gincl, 31);
    }
    __syncwarp();
    for (int r = lane; r < R; r += 32) uv.routes()[s_off[s_u[r]] + s_pos[r]] = r;
    if (lane == 0) {
      uv.U()[0] = run;
      uv.off()[run] = acc;
      uv.G()[0] = gacc;
    }
  } else {
    // 2c. dynamic e4m3 quantisation of x: per tensor (s_x = amax / 448 over all of
    //     x), or per (token, 128 columns) - piece i holds values [8i, 8i + 8), so 16
    //     consecutive threads hold one 128-column group.  When x fits one batch
    //     (T * H <= 8 * XB * NQ) it is read once, into registers.
    const bool one_batch = n8 <= XB * NQ;
    float s_t = 1.0f;
    if (a.quant == MOE_FP8_PER_TENSOR) {
      float m = 0.0f;
      for (int base = 0; base < n8; base += XB * NQ) {
        if (base > 0) {
#pragma unroll
          for (int j = 0; j < XB; ++j) {
            const int i = base + tq + j * NQ;
            xv[j] = i < n8 ? __ldg(x8 + i) : make_uint4(0, 0, 0, 0);
          }
        }
#pragma unroll
        for (int j = 0; j < XB; ++j) {
          const __nv_bfloat162* b = reinterpret_cast<const __nv_bfloat162*>(&xv[j]);
#pragma unroll
          for (int h2 = 0; h2 < 4; ++h2) {
            const float2 f = __bfloat1622float2(b[h2]);
            m = fmaxf(m, fmaxf(fabsf(f.x), fabsf(f.y)));
          }
        }
      }
      m = warp_max(m);
      if (lane == 0) s_red[warp] = m;
      asm volatile("bar.sync 1, %0;" ::"n"(NQ) : "memory");
      if (warp == 1) {
        float v = lane > 0 ? s_red[lane] : 0.0f;  // warps 1..31
        v = warp_max(v);
        if (lane == 0) s_red[0] = v;
      }
      asm volatile("bar.sync 1, %0;" ::"n"(NQ) : "memory");
      s_t = e4m3_scale(s_red[0]);
      if (tq == 0) {
        a.sx[0] = s_t;
        a.hdr->amax_x = __float_as_uint(s_red[0]);
      }
    }
    for (int base = 0; base < n8; base += XB * NQ) {
      if (!(one_batch || (base == 0 && a.quant != MOE_FP8_PER_TENSOR))) {
#pragma unroll
        for (int j = 0; j < XB; ++j) {
          const int i = base + tq + j * NQ;
          xv[j] = i < n8 ? __ldg(x8 + i) : make_uint4(0, 0, 0, 0);
        }
      }
#pragma unroll
      for (int j = 0; j < XB; ++j) {
        const int i = base + tq + j * NQ;  // i < n8 for all 16 threads of a group or none
        float f[8];
        const __nv_bfloat162* b = reinterpret_cast<const __nv_bfloat162*>(&xv[j]);
#pragma unroll
        for (int h2 = 0; h2 < 4; ++h2) {
          const float2 v = __bfloat1622float2(b[h2]);
          f[2 * h2] = v.x;
          f[2 * h2 + 1] = v.y;
        }
        float sc = s_t;
        if (a.quant == MOE_FP8_BLOCK128) {
          float mx = 0.0f;
#pragma unroll
          for (int q = 0; q < 8; ++q) mx = fmaxf(mx, fabsf(f[q]));
#pragma unroll
          for (int o = 1; o < 16; o <<= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
          sc = e4m3_scale(mx);
          if (i < n8 && (i & 15) == 0) a.sx[i / 16] = sc;
        }
        if (i < n8) {
          const uint32_t q0 = static_cast<uint32_t>(cvt_e4m3x2(f[0] / sc, f[1] / sc)) |
                              (static_cast<uint32_t>(cvt_e4m3x2(f[2] / sc, f[3] / sc)) << 16);
          const uint32_t q1 = static_cast<uint32_t>(cvt_e4m3x2(f[4] / sc, f[5] / sc)) |
                              (static_cast<uint32_t>(cvt_e4m3x2(f[6] / sc, f[7] / sc)) << 16);
          reinterpret_cast<uint2*>(a.xq)[i] = make_uint2(q0, q1);
        }
      }
    }
  }
}

// ------------------------------------------------------------------ weight streaming
// Shared layout of rd_gateup / rd_down (dynamic shared memory):
//   [NS weight stages: CK/128 TMA boxes of 64 rows x 128 bytes]
//   [operand: 8 rows x pitch][operand scales: 8 x K/128 fp32]
//   [full[NS], empty[NS] mbarriers][abort flag]
// Boxes are written with the 128-byte swizzle: 16-byte chunk c of row r sits
// at chunk c ^ (r & 7).  MMA row g of a warp's 16-row slab is weight row
// swz_row(g) = g/2 + 4 (g & 1), so the two rows read in one phase of a
// 16-byte fragment load differ in bit 2 and their chunks never share a bank.
// A staged operand row's pitch is 64 (mod 128) bytes, which does the same for
// rows g and g + 1 of the operand.
__host__ __device__ constexpr int swz_row(int g) { return (g >> 1) + 4 * (g & 1); }

// Address of the 16-byte fragment of weight row r (0..63), K bytes [kb, kb + 16)
// of a stage (kb a multiple of 16).
__device__ __forceinline__ const uint4* wfrag(const uint8_t* stage, int r, int kb) {
  const int box = kb / BOXK, c = (kb % BOXK) / 16;
  return reinterpret_cast<const uint4*>(stage + box * BOX_BYTES + r * BOXK + ((c ^ (r & 7)) * 16));
}
struct StreamSmem {
  uint8_t* stages;
  uint8_t* opnd;
  float* osc;
  float* wsc;  // blockwise: the current item's weight scales, 32 per consumer warp
  uint64_t* full;
  uint64_t* empty;
  volatile int* abort_flag;
};

// Pitch of a staged operand row of K bytes: 64 (mod 128).
__host__ __device__ inline int opnd_pitch(int K) { return (K + 127) / 128 * 128 + 64; }

// Ring of a stream kernel whose stages hold RCK K bytes of 64 rows: as many stages
// as fit the default ring's NS x CK bytes per row (Down uses RCK = 256 for short
// rows, I <= 256, so that twice as many items are in flight).
template <int RCK>
__host__ __device__ constexpr int ring_ns() { return NS * CK / RCK; }
template <int RCK>
__host__ __device__ constexpr int ring_stage_bytes() { return ROWS_PER_CTA * RCK; }

template <int RCK = CK>
__host__ __device__ inline size_t stream_smem_bytes(int K) {
  const size_t opnd = static_cast<size_t>(GROUP) * opnd_pitch(K);
  const size_t osc = static_cast<size_t>(GROUP) * ((K + 127) / 128) * 4;
  return 1024 + static_cast<size_t>(ring_ns<RCK>()) * ring_stage_bytes<RCK>() + opnd + ((osc + 15) / 16) * 16 +
         CONSUMERS * 32 * 4 + 2 * ring_ns<RCK>() * 8 + 16;
}

template <int RCK = CK>
__device__ __forceinline__ StreamSmem stream_smem(uint8_t* raw, int K) {
  StreamSmem m;
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(raw) + 1023) & ~uintptr_t(1023));
  m.stages = base;  // swizzled TMA box destinations: 1024-byte aligned
  m.opnd = base + ring_ns<RCK>() * ring_stage_bytes<RCK>();
  m.osc = reinterpret_cast<float*>(m.opnd + GROUP * opnd_pitch(K));
  const size_t osc = static_cast<size_t>(GROUP) * ((K + 127) / 128) * 4;
  m.wsc = reinterpret_cast<float*>(reinterpret_cast<uint8_t*>(m.osc) + ((osc + 15) / 16) * 16);
  m.full = reinterpret_cast<uint64_t*>(m.wsc + CONSUMERS * 32);
  m.empty = m.full + ring_ns<RCK>();
  m.abort_flag = reinterpret_cast<volatile int*>(m.empty + ring_ns<RCK>());
  return m;
}

// Producer side of the ring: streams the 64 rows [row0, row0 + 64) of the
// weight matrix behind `map` (K bytes innermost), columns [k0, k0 + nbytes),
// into successive stages, RCK bytes (RCK / 128 boxes) per stage.  Returns false
// after an abort.
template <int RCK = CK>
__device__ __forceinline__ bool produce_rows(const StreamSmem& m, const CUtensorMap* map, int k0, int row0,
                                             int nbytes, uint32_t& stage, uint32_t& phase, DeviceHeader* hdr,
                                             unsigned int where) {
  const int lane = threadIdx.x & 31;
  for (int c = 0; c < nbytes; c += RCK) {
    const int bytes = min(RCK, nbytes - c);
    int good = 1;
    if (lane == 0) good = mbar_wait(smem_u32(m.empty + stage), phase ^ 1, m.abort_flag, hdr, where);
    if (!__shfl_sync(0xffffffffu, good, 0)) return false;
    const uint32_t full = smem_u32(m.full + stage);
    if (lane == 0) {
      // whole boxes (a box past the end of a row is zero-filled by the TMA unit and
      // its columns are never read); weights are read once: evict them from L2 first
      const int nbox = (bytes + BOXK - 1) / BOXK;
      mbar_arrive_expect_tx(full, static_cast<uint32_t>(nbox) * BOX_BYTES);
      const uint32_t dst = smem_u32(m.stages + stage * ring_stage_bytes<RCK>());
      const uint64_t pol = l2_evict_first_policy();
      for (int j = 0; j < nbox; ++j) tma_load_2d_hint(dst + j * BOX_BYTES, map, k0 + c + j * BOXK, row0, full, pol);
    }
    __syncwarp();
    if (++stage == ring_ns<RCK>()) {
      stage = 0;
      phase ^= 1;
    }
  }
  return true;
}

// Ring setup by thread 0 (full: 1 arrival + bytes; empty: one arrival per consumer warp).
template <int RCK = CK>
__device__ __forceinline__ void init_ring(const StreamSmem& m) {
  if (threadIdx.x == 0) {
    for (int i = 0; i < ring_ns<RCK>(); ++i) {
      mbar_init(smem_u32(m.full + i), 1);
      mbar_init(smem_u32(m.empty + i), CONSUMERS);
    }
    *m.abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
}

// After an abort: let the producer's copies that are still in flight land
// before the CTA exits (bounded).
template <int RCK = CK>
__device__ __forceinline__ void drain_ring(const StreamSmem& m, uint32_t stage, uint32_t phase, int issued) {
  constexpr int ns = ring_ns<RCK>();
  for (int i = 0; i < min(issued, ns); ++i) {
    stage = (stage + ns - 1) % ns;
    if (stage == ns - 1) phase ^= 1;
    mbar_wait_quiet(smem_u32(m.full + stage), phase, 50000000ull);
  }
}

__device__ __forceinline__ void consumer_sync() { asm volatile("bar.sync 1, %0;" ::"n"(32 * CONSUMERS) : "memory"); }

// ------------------------------------------------------------------ rd_gateup
// Persistent: two CTAs per SM, each walking a contiguous range of work items
// (column group g, K split s, 64 rows mb of W1[e]) ordered so that consecutive
// items share (g, s) and with it the staged x slice.  Per item the warps
// compute a [64 rows x 8 routes] partial over the K slice [s*KS, (s+1)*KS).
template <bool BLOCKWISE>
__global__ void __launch_bounds__(THREADS, 2) rd_gateup_kernel(const __grid_constant__ CUtensorMap tmw, const __grid_constant__ CUtensorMap tmw2, DecodeArgs a,
                     int nMB, int S, int KS, int down_grid) {
  extern __shared__ __align__(128) uint8_t smem_raw[];
  pdl_trigger();
  const StreamSmem m = stream_smem(smem_raw, KS);
  init_ring(m);
  pdl_wait();
  const UniqView uv{a.uniq, max_uniq(a.R, a.E), a.R};
  const int G = *uv.G();
  const int per_g = S * nMB;
  const int N = G * per_g;
  const int it0 = static_cast<int>(static_cast<long long>(N) * blockIdx.x / gridDim.x);
  const int it1 = static_cast<int>(static_cast<long long>(N) * (blockIdx.x + 1) / gridDim.x);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int twoI = 2 * a.I, H = a.H;
  const int xpitch = opnd_pitch(KS);

  if (warp == CONSUMERS) {
    // ---------------------------------------------------------------- producer
    if (lane == 0) {
      prefetch_tensormap(&tmw);
      prefetch_tensormap(&tmw2);
    }
    uint32_t stage = 0, phase = 0;
    int issued = 0;
    bool ok = true;
    for (int it = it0; it < it1 && ok; ++it) {
      const int g = it / per_g, rest = it - g * per_g, s = rest / nMB, mb = rest - s * nMB;
      const int e = uv.expert()[uv.gu()[g]];
      ok = produce_rows(m, &tmw, s * KS, e * twoI + mb * ROWS_PER_CTA, KS, stage, phase, a.hdr, 0x90000u);
      issued += (KS + CK - 1) / CK;
    }
    if (!ok && lane == 0) drain_ring(m, stage, phase, issued);
    // With its W1 boxes issued, the producer prefetches W2 into L2 for the Down
    // kernel that follows: for each Down CTA d it serves, the first items of d's
    // work range (the same split rd_down makes), up to kW2PrefetchBytes in all,
    // so that the Down GEMV starts from L2 while this kernel's tail still runs.
    if (ok) {
      const int nHB = H / ROWS_PER_CTA, nbx = (a.I + BOXK - 1) / BOXK;
      const long long Nd = static_cast<long long>(G) * nHB;
      const double frac = fmin(1.0, static_cast<double>(kW2PrefetchBytes) / (static_cast<double>(Nd) * ROWS_PER_CTA * a.I));
      for (int d = blockIdx.x; d < down_grid; d += gridDim.x) {
        const long long i0 = Nd * d / down_grid, i1 = Nd * (d + 1) / down_grid;
        const long long iend = i0 + static_cast<long long>(ceil(frac * static_cast<double>(i1 - i0)));
        for (long long q = i0 * nbx + lane; q < iend * nbx; q += 32) {
          const long long item = q / nbx;
          const int bx = static_cast<int>(q - item * nbx);
          const int g = static_cast<int>(item / nHB), hb = static_cast<int>(item - static_cast<long long>(g) * nHB);
          tma_prefetch_2d(&tmw2, bx * BOXK, uv.expert()[uv.gu()[g]] * H + hb * ROWS_PER_CTA);
        }
      }
    }
  } else {
    // ---------------------------------------------------------------- consumers
    const int g8 = lane >> 2, tig = lane & 3;
    uint32_t stage = 0, phase = 0;
    bool ok = true;
    int cur = -1;  // (g, s) of the staged x slice
    int u = 0, e = 0, r_beg = 0, nn = 0;
    for (int it = it0; it < it1; ++it) {
      const int g = it / per_g, rest = it - g * per_g, s = rest / nMB, mb = rest - s * nMB;
      const int k0 = s * KS;
      if (g * S + s != cur) {
        // stage x of this group's tokens, K slice [k0, k0 + KS) (zeros for absent columns)
        cur = g * S + s;
        u = uv.gu()[g];
        e = uv.expert()[u];
        r_beg = uv.off()[u] + uv.gn0()[g];
        nn = min(GROUP, uv.off()[u + 1] - r_beg);
        consumer_sync();
        // copy this group's e4m3 x rows, K slice [k0, k0 + KS), and their scales
        // (zeros for absent columns); loads issued 8 at a time
        const int c16 = KS / 16;
        for (int base = 0; base < GROUP * c16; base += 8 * 32 * CONSUMERS) {
          uint4 v[8];
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            const int i = base + threadIdx.x + j * 32 * CONSUMERS;
            const int n = i / c16, c = i - n * c16;
            v[j] = make_uint4(0, 0, 0, 0);
            if (n < nn) {
              const int t = uv.routes()[r_beg + n] / a.k;
              v[j] = __ldg(reinterpret_cast<const uint4*>(a.xq + static_cast<size_t>(t) * H + k0) + c);
            }
          }
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            const int i = base + threadIdx.x + j * 32 * CONSUMERS;
            const int n = i / c16, c = i - n * c16;
            if (n < GROUP) *reinterpret_cast<uint4*>(m.opnd + n * xpitch + c * 16) = v[j];
          }
        }
        if (BLOCKWISE) {
          const int ng = H / 128, kb0 = k0 / 128, nkb = KS / 128;
          for (int i = threadIdx.x; i < GROUP * nkb; i += 32 * CONSUMERS) {
            const int n = i / nkb, q = i - n * nkb;
            m.osc[i] = n < nn ? __ldg(a.sx + static_cast<size_t>(uv.routes()[r_beg + n] / a.k) * ng + kb0 + q) : 0.0f;
          }
        }
        consumer_sync();
      }
      const int wr = warp * 16 + swz_row(g8);              // slab rows wr and wr + 8 of this item
      const int row = mb * ROWS_PER_CTA + wr;               // rows row and row + 8 of W1[e]
      const uint8_t* xs = m.opnd + g8 * xpitch + 16 * tig;
      const float* sw = BLOCKWISE ? a.w1_scale + (static_cast<size_t>(e) * (twoI / 128) + row / 128) * (H / 128) : nullptr;
      // the item's weight scales (one per 128 K bytes, the same for all its rows):
      // one coalesced load per warp, written to the warp's slot after the first
      // stage wait so that the load overlaps it (KS / 128 <= 32 by validation)
      float* wsl = m.wsc + warp * 32;
      float wreg = 0.0f;
      if (BLOCKWISE && lane < KS / 128) wreg = __ldg(sw + k0 / 128 + lane);
      bool wsl_ready = !BLOCKWISE;
      float c[4] = {0.f, 0.f, 0.f, 0.f};
      for (int cc = 0; cc < KS; cc += CK) {
        const int bytes = min(CK, KS - cc);
        // every lane observes the stage's completion; the outcome is made
        // warp-uniform before the (warp-synchronous) MMAs
        ok = __all_sync(0xffffffffu, ok && mbar_wait(smem_u32(m.full + stage), phase, m.abort_flag, a.hdr, 0x91000u));
        if (ok) {
          const uint8_t* st = m.stages + stage * STAGE_BYTES;
          if (!wsl_ready) {
            __syncwarp();  // the previous item's reads of the slot are done
            if (lane < KS / 128) wsl[lane] = wreg;
            __syncwarp();
            wsl_ready = true;
          }
          if (!BLOCKWISE) {
            for (int kk = 0; kk < bytes; kk += 64) {
              const uint4 A0 = *wfrag(st, wr, kk + 16 * tig);
              const uint4 A1 = *wfrag(st, wr + 8, kk + 16 * tig);
              const uint4 X = *reinterpret_cast<const uint4*>(xs + cc + kk);
              mma_k64(c, A0, A1, X);
            }
          } else {
            for (int kk = 0; kk < bytes; kk += 128) {
              float cb[4] = {0.f, 0.f, 0.f, 0.f};
              mma_k64(cb, *wfrag(st, wr, kk + 16 * tig), *wfrag(st, wr + 8, kk + 16 * tig),
                      *reinterpret_cast<const uint4*>(xs + cc + kk));
              mma_k64(cb, *wfrag(st, wr, kk + 64 + 16 * tig), *wfrag(st, wr + 8, kk + 64 + 16 * tig),
                      *reinterpret_cast<const uint4*>(xs + cc + kk + 64));
              const int q = (cc + kk) / 128;
              const float w_s = wsl[q];
              const float s0 = w_s * m.osc[(2 * tig) * (KS / 128) + q];
              const float s1 = w_s * m.osc[(2 * tig + 1) * (KS / 128) + q];
              c[0] = fmaf(cb[0], s0, c[0]);
              c[1] = fmaf(cb[1], s1, c[1]);
              c[2] = fmaf(cb[2], s0, c[2]);
              c[3] = fmaf(cb[3], s1, c[3]);
            }
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(m.empty + stage));
        if (++stage == NS) {
          stage = 0;
          phase ^= 1;
        }
      }
      // c0: (row, col 2tig), c1: (row, col 2tig+1), c2/c3: row + 8
      if (ok) {
        float* part = a.part + static_cast<size_t>(s) * a.R * twoI;
#pragma unroll
        for (int i = 0; i < 2; ++i) {
          const int col = 2 * tig + i;
          if (col < nn) {
            const int r = uv.routes()[r_beg + col];
            part[static_cast<size_t>(r) * twoI + row] = c[i];
            part[static_cast<size_t>(r) * twoI + row + 8] = c[2 + i];
          }
        }
      }
    }
  }
  __syncthreads();
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
// Four consecutive columns [i, i + 4) at once (i a multiple of 4): one 16-byte load
// per split for g and for u, all splits of a batch in flight together; the sums
// run over the splits in the same ascending order as sum_splits.
__device__ __forceinline__ void sum_splits4(const float* part, int splits, int R, int twoI, int I, int r, int i,
                                            float (&g)[4], float (&u)[4]) {
#pragma unroll
  for (int q = 0; q < 4; ++q) g[q] = u[q] = 0.f;
  for (int s0 = 0; s0 < splits; s0 += 8) {
    float4 gv[8], uv[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int s = s0 + j < splits ? s0 + j : 0;
      const float* pp = part + (static_cast<size_t>(s) * R + r) * twoI;
      gv[j] = *reinterpret_cast<const float4*>(pp + i);
      uv[j] = *reinterpret_cast<const float4*>(pp + I + i);
    }
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      if (s0 + j < splits) {
        g[0] += gv[j].x; g[1] += gv[j].y; g[2] += gv[j].z; g[3] += gv[j].w;
        u[0] += uv[j].x; u[1] += uv[j].y; u[2] += uv[j].z; u[3] += uv[j].w;
      }
    }
  }
}

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
  // groups of 128 columns; the last one holds I % 128 columns when I % 128 == 64
  const int I = a.I, twoI = 2 * I, ngi = (I + 127) / 128;
  if (gw >= a.R * ngi) return;
  const int r = gw / ngi, G = gw - (gw / ngi) * ngi;
  const int col = G * 128 + lane * 4;
  const bool valid = col < I;
  float av[4] = {0.f, 0.f, 0.f, 0.f}, g[4], u[4];
  if (valid) {
    sum_splits4(a.part, a.splits, a.R, twoI, I, r, col, g, u);
#pragma unroll
    for (int q = 0; q < 4; ++q) av[q] = silu_mul(g[q], u[q]);
  }
  float m = fmaxf(fmaxf(fabsf(av[0]), fabsf(av[1])), fmaxf(fabsf(av[2]), fabsf(av[3])));
  m = warp_max(m);
  const float sc = e4m3_scale(m);
  const uint32_t q = static_cast<uint32_t>(cvt_e4m3x2(av[0] / sc, av[1] / sc)) |
                     (static_cast<uint32_t>(cvt_e4m3x2(av[2] / sc, av[3] / sc)) << 16);
  if (valid) *reinterpret_cast<uint32_t*>(static_cast<uint8_t*>(a.act) + static_cast<size_t>(r) * I + col) = q;
  if (lane == 0) a.sh[static_cast<size_t>(r) * ngi + G] = sc;
}

// ------------------------------------------------------------------ rd_down
// Persistent like rd_gateup: work items (column group g, 64 rows hb of W2[e]),
// consecutive items share g and with it the staged h rows; K = I whole.
template <bool BLOCKWISE, int RCK>
__global__ void __launch_bounds__(THREADS, 2) rd_down_kernel(const __grid_constant__ CUtensorMap tmw, DecodeArgs a, int nHB) {
  extern __shared__ __align__(128) uint8_t smem_raw[];
  pdl_trigger();
  const int I = a.I, H = a.H, ngi = (I + 127) / 128;  // 128-column scale groups of h (last may be 64)
  const StreamSmem m = stream_smem<RCK>(smem_raw, I);
  init_ring<RCK>(m);
  pdl_wait();
  const UniqView uv{a.uniq, max_uniq(a.R, a.E), a.R};
  const int G = *uv.G();
  const int N = G * nHB;
  const int it0 = static_cast<int>(static_cast<long long>(N) * blockIdx.x / gridDim.x);
  const int it1 = static_cast<int>(static_cast<long long>(N) * (blockIdx.x + 1) / gridDim.x);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int hpitch = opnd_pitch(I);

  if (warp == CONSUMERS) {
    if (lane == 0) prefetch_tensormap(&tmw);
    uint32_t stage = 0, phase = 0;
    int issued = 0;
    bool ok = true;
    for (int it = it0; it < it1 && ok; ++it) {
      const int g = it / nHB, hb = it - g * nHB;
      const int e = uv.expert()[uv.gu()[g]];
      ok = produce_rows<RCK>(m, &tmw, 0, e * H + hb * ROWS_PER_CTA, I, stage, phase, a.hdr, 0x92000u);
      issued += (I + RCK - 1) / RCK;
    }
    if (!ok && lane == 0) drain_ring<RCK>(m, stage, phase, issued);
  } else {
    const int g8 = lane >> 2, tig = lane & 3;
    const float s_h_t = BLOCKWISE ? 1.0f : e4m3_scale(__uint_as_float(a.hdr->amax_h));
    uint32_t stage = 0, phase = 0;
    bool ok = true;
    int cur = -1;
    int e = 0, r_beg = 0, nn = 0;
    for (int it = it0; it < it1; ++it) {
      const int g = it / nHB, hb = it - g * nHB;
      if (g != cur) {
        // stage the e4m3 h rows of this group's routes (zeros for absent columns)
        cur = g;
        const int u = uv.gu()[g];
        e = uv.expert()[u];
        r_beg = uv.off()[u] + uv.gn0()[g];
        nn = min(GROUP, uv.off()[u + 1] - r_beg);
        consumer_sync();
        // blockwise MMAs read whole 128-byte K blocks: columns past I are staged as zeros.
        // Blockwise rows are copied with 8 loads in flight per thread; per-tensor rows
        // are quantised on the way (an IEEE division per value), one piece at a time:
        // batching those measured 3 us slower per call
        if (BLOCKWISE) {
          const int c4 = ngi * 128 / 4;
          constexpr int SB = 8;
          for (int base = 0; base < GROUP * c4; base += SB * 32 * CONSUMERS) {
            uint32_t v[SB];
#pragma unroll
            for (int j = 0; j < SB; ++j) {
              const int i = base + threadIdx.x + j * 32 * CONSUMERS;
              const int n = i / c4, c = (i - n * c4) * 4;
              v[j] = 0u;
              if (n < nn && c < I)
                v[j] = __ldg(reinterpret_cast<const uint32_t*>(static_cast<const uint8_t*>(a.act) +
                                                               static_cast<size_t>(uv.routes()[r_beg + n]) * I + c));
            }
#pragma unroll
            for (int j = 0; j < SB; ++j) {
              const int i = base + threadIdx.x + j * 32 * CONSUMERS;
              const int n = i / c4, c = (i - n * c4) * 4;
              if (n < GROUP) *reinterpret_cast<uint32_t*>(m.opnd + n * hpitch + c) = v[j];
            }
          }
        } else {
          const int c4 = I / 4;
          for (int i = threadIdx.x; i < GROUP * c4; i += 32 * CONSUMERS) {
            const int n = i / c4, c = (i - n * c4) * 4;
            uint32_t q = 0;
            if (n < nn) {
              const int r = uv.routes()[r_beg + n];
              const float4 v = __ldg(reinterpret_cast<const float4*>(static_cast<const float*>(a.act) + static_cast<size_t>(r) * I + c));
              q = static_cast<uint32_t>(cvt_e4m3x2(v.x / s_h_t, v.y / s_h_t)) |
                  (static_cast<uint32_t>(cvt_e4m3x2(v.z / s_h_t, v.w / s_h_t)) << 16);
            }
            *reinterpret_cast<uint32_t*>(m.opnd + n * hpitch + c) = q;
          }
        }
        if (BLOCKWISE) {
          for (int i = threadIdx.x; i < GROUP * ngi; i += 32 * CONSUMERS) {
            const int n = i / ngi, q = i - n * ngi;
            m.osc[i] = n < nn ? __ldg(a.sh + static_cast<size_t>(uv.routes()[r_beg + n]) * ngi + q) : 0.0f;
          }
        }
        consumer_sync();
      }
      const int wr = warp * 16 + swz_row(g8);              // slab rows wr and wr + 8 of this item
      const int row = hb * ROWS_PER_CTA + wr;               // rows row and row + 8 of W2[e]
      const uint8_t* hs = m.opnd + g8 * hpitch + 16 * tig;
      const float* sw = BLOCKWISE ? a.w2_scale + (static_cast<size_t>(e) * (H / 128) + row / 128) * ngi : nullptr;
      // the item's weight scales, staged like rd_gateup's (ngi = ceil(I / 128) <= 32)
      float* wsl = m.wsc + warp * 32;
      float wreg = 0.0f;
      if (BLOCKWISE && lane < ngi) wreg = __ldg(sw + lane);
      bool wsl_ready = !BLOCKWISE;
      float c[4] = {0.f, 0.f, 0.f, 0.f};
      for (int cc = 0; cc < I; cc += RCK) {
        const int bytes = min(RCK, I - cc);
        ok = __all_sync(0xffffffffu, ok && mbar_wait(smem_u32(m.full + stage), phase, m.abort_flag, a.hdr, 0x93000u));
        if (ok) {
          const uint8_t* st = m.stages + stage * ring_stage_bytes<RCK>();
          if (!wsl_ready) {
            __syncwarp();  // the previous item's reads of the slot are done
            if (lane < ngi) wsl[lane] = wreg;
            __syncwarp();
            wsl_ready = true;
          }
          if (!BLOCKWISE) {
            for (int kk = 0; kk < bytes; kk += 64)
              mma_k64(c, *wfrag(st, wr, kk + 16 * tig), *wfrag(st, wr + 8, kk + 16 * tig),
                      *reinterpret_cast<const uint4*>(hs + cc + kk));
          } else {
            for (int kk = 0; kk < bytes; kk += 128) {
              float cb[4] = {0.f, 0.f, 0.f, 0.f};
              mma_k64(cb, *wfrag(st, wr, kk + 16 * tig), *wfrag(st, wr + 8, kk + 16 * tig),
                      *reinterpret_cast<const uint4*>(hs + cc + kk));
              mma_k64(cb, *wfrag(st, wr, kk + 64 + 16 * tig), *wfrag(st, wr + 8, kk + 64 + 16 * tig),
                      *reinterpret_cast<const uint4*>(hs + cc + kk + 64));
              const int q = (cc + kk) / 128;
              const float w_s = wsl[q];
              const float s0 = w_s * m.osc[(2 * tig) * ngi + q];
              const float s1 = w_s * m.osc[(2 * tig + 1) * ngi + q];
              c[0] = fmaf(cb[0], s0, c[0]);
              c[1] = fmaf(cb[1], s1, c[1]);
              c[2] = fmaf(cb[2], s0, c[2]);
              c[3] = fmaf(cb[3], s1, c[3]);
            }
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(m.empty + stage));
        if (++stage == ring_ns<RCK>()) {
          stage = 0;
          phase ^= 1;
        }
      }
      if (ok) {
        if (!BLOCKWISE) {
          const float sc = s_h_t * __ldg(a.w2_scale + e);
#pragma unroll
          for (int i = 0; i < 4; ++i) c[i] *= sc;
        }
#pragma unroll
        for (int i = 0; i < 2; ++i) {
          const int col = 2 * tig + i;
          if (col < nn) {
            const int r = uv.routes()[r_beg + col];
            a.o[static_cast<size_t>(r) * H + row] = c[i];
            a.o[static_cast<size_t>(r) * H + row + 8] = c[2 + i];
          }
        }
      }
    }
  }
  __syncthreads();
}

}  // namespace rd

size_t route_direct_uniq_bytes(int T, int E, int k) {
  const int R = T * k;
  const int mu = rd::max_uniq(R, E);
  const int mg = mu + R / rd::GROUP + 1;
  return static_cast<size_t>(3 + 2 * mu + R + 2 * mg) * sizeof(int32_t);
}

cudaError_t launch_route_direct(const DecodeArgs& a, cudaStream_t s) {
  using namespace rd;
  if (a.T <= 0) return cudaSuccess;
  int maxv = 1;
  while (maxv * 32 < a.E) maxv *= 2;
  // one prep CTA, plus prefetch CTAs of about kPrefetchPerCta of W1 each for the
  // most W1 the batch can select (distinct experts <= min(T k, E)), within the budget
  const long long w1_bytes = 2ll * a.I * a.H;
  const long long cap = kW1PrefetchBytes / w1_bytes * w1_bytes;
  const long long most = static_cast<long long>(max_uniq(a.R, a.E)) * w1_bytes;
  const long long pf = most < cap ? most : cap;
  const int nsm = num_sms();
  long long npf = (pf + kPrefetchPerCta - 1) / kPrefetchPerCta;
  if (npf > nsm - 1) npf = nsm > 1 ? nsm - 1 : 0;
  const unsigned pgrid = 1u + static_cast<unsigned>(npf);
  stage_begin("rd_prep", s);
  switch (maxv) {
    case 1: rd_prep_kernel<1><<<pgrid, 1024, 0, s>>>(a); break;
    case 2: rd_prep_kernel<2><<<pgrid, 1024, 0, s>>>(a); break;
    case 4: rd_prep_kernel<4><<<pgrid, 1024, 0, s>>>(a); break;
    case 8: rd_prep_kernel<8><<<pgrid, 1024, 0, s>>>(a); break;
    default: rd_prep_kernel<16><<<pgrid, 1024, 0, s>>>(a); break;
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
  const int nHB = a.H / ROWS_PER_CTA;
  const int KS = a.H / a.splits;
  const int maxG = maxU + a.R / GROUP + 1;
  const int sms = 2 * num_sms();  // two persistent CTAs per SM
  if (sms <= 0) return cudaErrorNoDevice;
  // Down rows are I bytes long: short rows (I <= 256) take 256-byte stages, twice as many
  const bool short_rows = a.I <= 256;
  const size_t smem_gu = stream_smem_bytes(KS);
  const size_t smem_dn = short_rows ? stream_smem_bytes<256>(a.I) : stream_smem_bytes<CK>(a.I);
  auto down_kernel = [&]() {
    return bw ? (short_rows ? rd_down_kernel<true, 256> : rd_down_kernel<true, CK>)
              : (short_rows ? rd_down_kernel<false, 256> : rd_down_kernel<false, CK>);
  };
  {
    // raise the dynamic shared-memory limit once per instantiation to the largest size used
    static size_t set_gu[2] = {0, 0}, set_dn[4] = {0, 0, 0, 0};
    static std::mutex mu;
    std::lock_guard<std::mutex> lk(mu);
    if (smem_gu > set_gu[bw]) {
      err = bw ? cudaFuncSetAttribute(rd_gateup_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem_gu)
               : cudaFuncSetAttribute(rd_gateup_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem_gu);
      if (err != cudaSuccess) return err;
      set_gu[bw] = smem_gu;
    }
    const int dk = 2 * (bw ? 1 : 0) + (short_rows ? 1 : 0);
    if (smem_dn > set_dn[dk]) {
      err = cudaFuncSetAttribute(down_kernel(), cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem_dn);
      if (err != cudaSuccess) return err;
      set_dn[dk] = smem_dn;
    }
  }

  // weight matrices as 2D u8 tensors [rows][K bytes], boxes of 64 rows x 128 bytes, 128-byte swizzle
  CUtensorMap tm1, tm2;
  {
    EncodeTiledFn fn = get_encode_tiled();
    if (!fn) return cudaErrorInvalidValue;
    auto enc = [&](CUtensorMap* map, const void* base, uint64_t inner, uint64_t rows) {
      const cuuint64_t dims[2] = {inner, rows};
      const cuuint64_t strides[1] = {inner};
      const cuuint32_t box[2] = {static_cast<cuuint32_t>(BOXK), static_cast<cuuint32_t>(ROWS_PER_CTA)};
      const cuuint32_t estr[2] = {1, 1};
      return fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, estr,
                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
    };
    if (!enc(&tm1, a.w1, a.H, static_cast<uint64_t>(a.E) * 2 * a.I) ||
        !enc(&tm2, a.w2, a.I, static_cast<uint64_t>(a.E) * a.H))
      return cudaErrorInvalidValue;
  }

  const long long dn_items = static_cast<long long>(maxG) * nHB;
  const int down_grid = static_cast<int>(dn_items < sms ? dn_items : sms);
  stage_begin("rd_gateup", s);
  {
    const long long items = static_cast<long long>(maxG) * nMB * a.splits;
    const cudaLaunchConfig_t c = config(static_cast<unsigned>(items < sms ? items : sms), THREADS, smem_gu);
    err = bw ? cudaLaunchKernelEx(&c, rd_gateup_kernel<true>, tm1, tm2, a, nMB, a.splits, KS, down_grid)
             : cudaLaunchKernelEx(&c, rd_gateup_kernel<false>, tm1, tm2, a, nMB, a.splits, KS, down_grid);
  }
  stage_end(s);
  if (err != cudaSuccess) return err;

  stage_begin("rd_reduce", s);
  if (bw) {
    const int warps = a.R * ((a.I + 127) / 128);
    const cudaLaunchConfig_t c = config((warps * 32 + 255) / 256, 256, 0);
    err = cudaLaunchKernelEx(&c, rd_reduce_block_kernel, a);
  } else {
    const cudaLaunchConfig_t c = config((a.R * a.I + 255) / 256, 256, 0);
    err = cudaLaunchKernelEx(&c, rd_reduce_tensor_kernel, a);
  }
  stage_end(s);
  if (err != cudaSuccess) return err;

  stage_begin("rd_down", s);
  {
    const cudaLaunchConfig_t c = config(static_cast<unsigned>(down_grid), THREADS, smem_dn);
    err = cudaLaunchKernelEx(&c, down_kernel(), tm2, a, nHB);
  }
  stage_end(s);
  return err;
}

}  // namespace moe
