// Per-tensor e4m3 quantisation passes of the grouped FP8 path ("perf: add
// small-batch route MMA for MoE", Summary: per-tensor FP8 with dynamic
// activation scales): the expert-sorted copy of x quantised with s_x = amax/448
// (the amax of x comes from extra blocks of the route/rank kernel), and the
// quantisation of a (the SwiGLU output, held in bf16) with its global scale s_h;
// plus the blockwise form of the scatter (x quantised per (row, 128 columns); the
// blockwise h is quantised in the Gate/Up epilogue).  Scales: amax / 448 in fp32
// (1 when amax == 0); codes: round to nearest even with saturation
// (cvt.rn.satfinite).
#include "common.cuh"
#include "internal.h"

namespace moe {

// Scatter fused with the gather and quantisation of the activations, one block
// per token: the block quantises the token's x row once into shared memory (with
// s_x, or per 128 columns with a scale of its own: 16 consecutive threads hold a
// group, 8 values each, and reduce its amax), then one warp per route writes
// perm / inv and copies the e4m3 row (and its scales) to sorted row p of xs.
template <bool BLOCKWISE>
__global__ void __launch_bounds__(256) scatter_gather_tok_q_kernel(
    const int32_t* __restrict__ ids, const int32_t* __restrict__ lrank, const int32_t* __restrict__ blockbase, int E,
    int RB, int k, int H, const uint4* __restrict__ x, uint4* __restrict__ xs, float* __restrict__ xs_scale,
    int32_t* __restrict__ perm, int32_t* __restrict__ inv, const DeviceHeader* hdr, int S, int T) {
  extern __shared__ __align__(16) uint8_t s_row[];  // [H] e4m3, then [H/128] fp32 scales
  dep_wait();  // block bases and (per tensor) the amax of x
  float* s_sc = reinterpret_cast<float*>(s_row + H);
  const int t = blockIdx.x;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int n8 = H / 8;  // 8-value pieces of the row
  const float st = BLOCKWISE ? 1.0f : e4m3_scale(__uint_as_float(hdr->amax_x));
  const uint4* src = x + static_cast<size_t>(t) * n8;
  for (int base = 0; base < n8; base += blockDim.x) {
    const int c = base + tid;
    const bool act = c < n8;  // whole 16-thread groups are active together (H % 128 == 0)
    const uint4 v = act ? __ldg(src + c) : make_uint4(0, 0, 0, 0);
    float f[8];
    const __nv_bfloat162* b = reinterpret_cast<const __nv_bfloat162*>(&v);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float2 u = __bfloat1622float2(b[j]);
      f[2 * j] = u.x;
      f[2 * j + 1] = u.y;
    }
    float sc = st;
    if (BLOCKWISE) {
      float m = 0.0f;
#pragma unroll
      for (int j = 0; j < 8; ++j) m = fmaxf(m, fabsf(f[j]));
#pragma unroll
      for (int o = 1; o < 16; o <<= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
      sc = e4m3_scale(m);
      if (act && (c & 15) == 0) s_sc[c / 16] = sc;
    }
    if (act) {
      const uint32_t q0 = static_cast<uint32_t>(cvt_e4m3x2(f[0] / sc, f[1] / sc)) |
                          (static_cast<uint32_t>(cvt_e4m3x2(f[2] / sc, f[3] / sc)) << 16);
      const uint32_t q1 = static_cast<uint32_t>(cvt_e4m3x2(f[4] / sc, f[5] / sc)) |
                          (static_cast<uint32_t>(cvt_e4m3x2(f[6] / sc, f[7] / sc)) << 16);
      *reinterpret_cast<uint2*>(s_row + 8 * c) = make_uint2(q0, q1);
    }
  }
  __syncthreads();
  const int row16 = H / 16, groups = H / 128;
  // rows of the token's k routes, then its rows T*k + s*T + t of the S shared experts
  for (int j = warp; j < k + S; j += blockDim.x >> 5) {
    int p;
    if (j < k) {
      const int r = t * k + j;
      const int lr = lrank[r];
      if (lr < 0) {
        if (lane == 0) inv[r] = -1;
        continue;
      }
      const int e = ids[r];
      p = blockbase[static_cast<size_t>(r / RB) * E + e] + lr;
      if (lane == 0) {
        perm[p] = r;
        inv[r] = p;
      }
    } else {
      p = T * k + (j - k) * T + t;
    }
    uint4* dst = xs + static_cast<size_t>(p) * row16;
    for (int c = lane; c < row16; c += 32) dst[c] = reinterpret_cast<const uint4*>(s_row)[c];
    if (BLOCKWISE)
      for (int g = lane; g < groups; g += 32) xs_scale[static_cast<size_t>(p) * groups + g] = s_sc[g];
  }
}

// h = e4m3(a / s_h), s_h = e4m3_scale(amax of a); 4 values per thread-iteration.
// 8 bf16 values (one 16-byte piece) / s -> 8 e4m3 codes.
__device__ __forceinline__ uint2 quant_bf16x8(const uint4& v, float s) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
  uint32_t q[2];
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const float f0 = __uint_as_float(w[2 * i] << 16), f1 = __uint_as_float(w[2 * i] & 0xFFFF0000u);
    const float f2 = __uint_as_float(w[2 * i + 1] << 16), f3 = __uint_as_float(w[2 * i + 1] & 0xFFFF0000u);
    q[i] = static_cast<uint32_t>(cvt_e4m3x2(f0 / s, f1 / s)) | (static_cast<uint32_t>(cvt_e4m3x2(f2 / s, f3 / s)) << 16);
  }
  return make_uint2(q[0], q[1]);
}

__global__ void __launch_bounds__(256) quant_rows_kernel(const uint4* __restrict__ a, uint2* __restrict__ h,
                                                         size_t n8, const DeviceHeader* hdr) {
  dep_wait();  // a and its amax from the Gate/Up GEMM
  const float s = e4m3_scale(__uint_as_float(hdr->amax_h));
  const size_t stride = static_cast<size_t>(gridDim.x) * blockDim.x;
  // four independent loads in flight per thread; a is read once, so its lines are
  // evicted from L2 first and the h rows just written stay for the Down GEMM
  const uint64_t pol = l2_evict_first_policy();
  size_t i = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x;
  for (; i + 3 * stride < n8; i += 4 * stride) {
    uint4 v[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) v[j] = ld_nc_v4_hint(a + i + j * stride, pol);
#pragma unroll
    for (int j = 0; j < 4; ++j) h[i + j * stride] = quant_bf16x8(v[j], s);
  }
  for (; i < n8; i += stride) h[i] = quant_bf16x8(__ldg(a + i), s);
}

static unsigned grid_for(size_t work, unsigned per_block) {
  const int sms = num_sms();
  const size_t cap = static_cast<size_t>(sms > 0 ? sms : 148) * 16;
  size_t b = (work + per_block - 1) / per_block;
  if (b > cap) b = cap;
  return static_cast<unsigned>(b < 1 ? 1 : b);
}

static cudaError_t launch_tok_q(bool blockwise, const int32_t* ids, const int32_t* lrank, const int32_t* blockbase,
                                int T, int E, int k, int H, const void* x, void* xs, float* xs_scale, int32_t* perm,
                                int32_t* inv, const DeviceHeader* hdr, cudaStream_t s, int S) {
  if (T <= 0) return cudaSuccess;
  const int RB = route_tokens_per_block(k) * k;
  const size_t smem = static_cast<size_t>(H) + static_cast<size_t>(H / 128) * sizeof(float);
  if (smem > 48 * 1024) return cudaErrorInvalidValue;  // H <= 47K: far above any supported shape
  stage_begin("scatter_gather", s);
  const cudaError_t err =
      blockwise ? launch_dependent(scatter_gather_tok_q_kernel<true>, dim3(T), dim3(256), smem, s, ids, lrank, blockbase,
                                   E, RB, k, H, static_cast<const uint4*>(x), static_cast<uint4*>(xs), xs_scale, perm,
                                   inv, hdr, S, T)
                : launch_dependent(scatter_gather_tok_q_kernel<false>, dim3(T), dim3(256), smem, s, ids, lrank,
                                   blockbase, E, RB, k, H, static_cast<const uint4*>(x), static_cast<uint4*>(xs),
                                   static_cast<float*>(nullptr), perm, inv, hdr, S, T);
  stage_end(s);
  return err;
}

cudaError_t launch_scatter_gather_q(const int32_t* ids, const int32_t* lrank, const int32_t* blockbase, int T, int E,
                                    int k, int H, const void* x, void* xs, int32_t* perm, int32_t* inv,
                                    const DeviceHeader* hdr, cudaStream_t s, int S) {
  return launch_tok_q(false, ids, lrank, blockbase, T, E, k, H, x, xs, nullptr, perm, inv, hdr, s, S);
}

cudaError_t launch_quant_rows(const void* a, void* h, size_t n, const DeviceHeader* hdr, cudaStream_t s) {
  const size_t n8 = n / 8;
  if (n8 == 0) return cudaSuccess;
  stage_begin("quant_h", s);
  const cudaError_t err = launch_dependent(quant_rows_kernel, dim3(grid_for(n8, 256)), dim3(256), 0, s,
                                           static_cast<const uint4*>(a), static_cast<uint2*>(h), n8, hdr);
  stage_end(s);
  return err;
}

cudaError_t launch_scatter_gather_qb(const int32_t* ids, const int32_t* lrank, const int32_t* blockbase, int T, int E,
                                     int k, int H, const void* x, void* xs, float* xs_scale, int32_t* perm,
                                     int32_t* inv, cudaStream_t s, int S) {
  return launch_tok_q(true, ids, lrank, blockbase, T, E, k, H, x, xs, xs_scale, perm, inv, nullptr, s, S);
}

}  // namespace moe
