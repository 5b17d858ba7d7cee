// Grouped GEMMs of the grouped (prefill) path on the 5th-generation tensor
// cores ("perf: add small-batch route MMA for MoE", Motivation: Gate/Up grouped
// GEMM -> activation -> Down grouped GEMM).
//
// One persistent CTA per SM walks work units (row tile, N tile) of a task map
// built on the device (tile count read from device memory, no host sync).
// Warp roles (256 threads; 384 for the FP8 Gate/Up):
//   warp 0      TMA producer: A (activations) and B (weights) K-slices into a
//               4-stage shared-memory ring, 128-byte swizzled.
//   warp 1      one thread issues tcgen05.mma (M=128, N=256; K=16 bf16 or K=32
//               e4m3 per instruction, fp32 accumulate) into one of two TMEM
//               accumulators (2 x 256 columns).
//   warp 2      allocates / frees the 512 TMEM columns.
//   warps 4+    epilogue, one warp per 32-lane TMEM quadrant (two for the FP8
//               Gate/Up, each draining half of the accumulator's columns):
//               tcgen05.ld (one row per thread), the fused epilogue, stores
//               (Down: staged in shared memory as 128-byte-swizzled boxes and
//               written by TMA tile stores).
// Every launch is a programmatic dependent of the kernel before it: barrier
// and TMEM set-up run before the wait for the predecessor's results.
//
// Gate/Up (MODE_GATEUP): A = the expert-sorted activation rows that the
//   scatter kernel copied (plain TMA tile loads); or, as a selectable
//   variant, rows gathered straight from x with TMA tile::gather4 (row = token
//   of sorted route p = perm[p] / k).  B = the expert's gate rows [n0, n0+128)
//   and up rows [I+n0, I+n0+128) of W1, so one 128x256 accumulator holds
//   matching gate and up columns; the epilogue writes h = bf16(silu(g) * u)
//   (or fp32 a for the FP8 path) for sorted rows, columns [n0, n0+128).
// Down (MODE_DOWN): A = h rows of the tile, B = 256 rows of W2[e]; the
//   epilogue writes bf16 o in the same expert-sorted row order as h, so the
//   8 N tiles of one row tile together fill a contiguous block of o; the
//   combine finds route r's row at inv[r].
#include <cstdio>
#include <mutex>

#include "common.cuh"
#include "internal.h"

namespace moe {
namespace gg {

constexpr int BM = kGemmBM;  // 128
constexpr int BK = 64;       // bf16 elements per stage row = 128 bytes (e4m3: 128 elements)
constexpr int BN = 256;
constexpr int STAGES = 4;
constexpr int A_BYTES = BM * BK * 2;
constexpr int B_BYTES = BN * BK * 2;
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
constexpr int TMEM_COLS = 512;
// Epilogue warps (from warp 4): one or two per 32-lane TMEM quadrant.  Two, each
// draining half of the accumulator's columns, pay off where the mainloop of a
// tile is short next to its epilogue (FP8 Gate/Up: 16 K stages and fp32 output).
__host__ __device__ constexpr int epi_warps(int mode, bool f8) { return (mode == 0 && f8) ? 8 : 4; }
__host__ __device__ constexpr int threads_of(int mode, bool f8) { return 32 * (4 + epi_warps(mode, f8)); }
constexpr int NUM_BARS = 2 * STAGES + 4 + 1;
// epilogue staging: 4 warps x 32 rows x 256 bytes, after the barriers, 1024-byte
// aligned (the source of a 128-byte-swizzled TMA store)
constexpr int STAGING_OFFSET = (STAGES * STAGE_BYTES + 256 + 1023) / 1024 * 1024;
constexpr int STAGING_BYTES = 4 * 32 * 256;  // Down: 32 rows x 256 bytes per epilogue warp
constexpr size_t SMEM_BYTES = 1024 + STAGING_OFFSET + STAGING_BYTES;

constexpr int MODE_GATEUP = 0;
constexpr int MODE_DOWN = 1;

struct Params {
  const int32_t* tiles;
  const int32_t* num_tiles;
  int max_tiles;
  const int32_t* perm;
  int k;
  int nN;                // N tiles per row tile
  int K;                 // reduction length
  int b_rows_per_expert; // rows of W per expert (2I or H)
  int up_offset;         // I (Gate/Up)
  int n_valid;           // valid output columns (I or H)
  int out_ld;
  int a_gather;          // Gate/Up: 1 = A rows gathered from x by tile::gather4, 0 = sorted rows
  __nv_bfloat16* out;
  DeviceHeader* hdr;
  int E;                 // routed experts; tiles of expert E + s belong to shared expert s (weights in tmB2)
  // e4m3 inputs (per-tensor scales)
  const float* wscale;            // [E] scale of each expert's weight matrix
  const float* wscale2;           // [S] scales of the shared experts' matrices
  const unsigned int* amax_in;    // fp32 bits of the amax of the A operand's source (x or a)
  unsigned int* amax_out;         // Gate/Up: receives the amax of a
  __nv_bfloat16* out_a;           // F8 Gate/Up: a [R, I] bf16 (quantised by the next pass)
};

__device__ __forceinline__ uint4 pack_bf16x8(const float* v) {
  uint4 r;
  uint32_t* w = reinterpret_cast<uint32_t*>(&r);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    __nv_bfloat162 b = __floats2bfloat162_rn(v[2 * i], v[2 * i + 1]);
    w[i] = *reinterpret_cast<uint32_t*>(&b);
  }
  return r;
}

// Per-tensor weight scale of expert e (a shared expert's for e >= p.E).
__device__ __forceinline__ float wscale_of(const Params& p, int e) {
  return e < p.E ? __ldg(p.wscale + e) : __ldg(p.wscale2 + (e - p.E));
}

// F8: e4m3 operands (tcgen05 kind::f8f6f4, 128 K elements per 128-byte stage
// row, per-tensor scales applied in the epilogue); otherwise bf16 (kind::f16).
template <int MODE, bool F8>
__global__ void __launch_bounds__(threads_of(MODE, F8), 1)
    grouped_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                        const __grid_constant__ CUtensorMap tmO, const __grid_constant__ CUtensorMap tmB2,
                        const Params p) {
  constexpr int BKE = F8 ? 128 : BK;  // K elements per stage
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + STAGES * STAGE_BYTES);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + NUM_BARS);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t full0 = smem_u32(bars), empty0 = smem_u32(bars + STAGES);
  const uint32_t tfull0 = smem_u32(bars + 2 * STAGES), tempty0 = smem_u32(bars + 2 * STAGES + 2);
  const uint32_t mma_done = smem_u32(bars + 2 * STAGES + 4);

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(full0 + 8 * s, 1);
      mbar_init(empty0 + 8 * s, 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(tfull0 + 8 * a, 1);
      mbar_init(tempty0 + 8 * a, epi_warps(MODE, F8));  // one arrival per epilogue warp
    }
    mbar_init(mma_done, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tensormap(&tmA);
    prefetch_tensormap(&tmB);
    prefetch_tensormap(&tmB2);
  }
  if (warp == 2) {
    tmem_alloc(smem_u32(tmem_slot), TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  dep_wait();  // the tile map and the A rows come from the kernels before (the set-up above overlaps them)

  const int ntiles = min(*p.num_tiles, p.max_tiles);
  const int total = ntiles * p.nN;
  const int nk = (p.K + BKE - 1) / BKE;
  const int4* tiles = reinterpret_cast<const int4*>(p.tiles);

  if (warp == 0) {
    // ---------------------------------------------------------------- producer
    uint32_t stage = 0, phase = 0;
    int issued = 0;
    bool ok = true;
    for (int u = blockIdx.x; u < total && ok; u += gridDim.x) {
      const int tile = u / p.nN, n = u - (u / p.nN) * p.nN;
      const int4 tl = tiles[tile];
      const int e = tl.x, row0 = tl.y, nrows = tl.z;
      int tok[4] = {0, 0, 0, 0};
      if (MODE == MODE_GATEUP && p.a_gather) {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int pr = row0 + min(lane * 4 + i, nrows - 1);
          tok[i] = __ldg(p.perm + pr) / p.k;
        }
      }
      const bool shx = e >= p.E;  // a shared expert's tile: its own weight tensor
      const CUtensorMap* tb = shx ? &tmB2 : &tmB;
      const int brow = (shx ? e - p.E : e) * p.b_rows_per_expert + n * (MODE == MODE_GATEUP ? BN / 2 : BN);
      for (int kb = 0; kb < nk; ++kb) {
        int good = 1;
        if (lane == 0) good = mbar_wait(empty0 + 8 * stage, phase ^ 1, abort_flag, p.hdr, 0x10000u | MODE);
        good = __shfl_sync(0xffffffffu, good, 0);
        if (!good) {
          ok = false;
          break;
        }
        const uint32_t full = full0 + 8 * stage;
        if (lane == 0) mbar_arrive_expect_tx(full, STAGE_BYTES);
        __syncwarp();
        const uint32_t a_dst = smem_u32(smem + stage * STAGE_BYTES);
        const uint32_t b_dst = a_dst + A_BYTES;
        const int kc = kb * BKE;
        if (MODE == MODE_GATEUP) {
          if (p.a_gather)
            tma_gather4(a_dst + lane * 4 * 128, &tmA, kc, tok[0], tok[1], tok[2], tok[3], full);
          if (lane == 0) {
            if (!p.a_gather) tma_load_2d(a_dst, &tmA, kc, row0, full);
            tma_load_2d(b_dst, tb, kc, brow, full);
            tma_load_2d(b_dst + B_BYTES / 2, tb, kc, brow + p.up_offset, full);
          }
        } else {
          if (lane == 0) {
            tma_load_2d(a_dst, &tmA, kc, row0, full);
            tma_load_2d(b_dst, tb, kc, brow, full);
          }
        }
        ++issued;
        if (++stage == STAGES) {
          stage = 0;
          phase ^= 1;
        }
      }
    }
    if (!ok && lane == 0) {
      // aborted: let the copies already issued land before shared memory is released
      for (int i = 0; i < min(issued, STAGES); ++i) {
        stage = (stage + STAGES - 1) % STAGES;
        if (stage == STAGES - 1) phase ^= 1;
        mbar_wait_quiet(full0 + 8 * stage, phase, 50000000ull);
      }
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------------- MMA issuer
    if (lane == 0) {
      const uint32_t idesc = F8 ? make_idesc(0, 0, BM, BN) : make_idesc(1, 1, BM, BN);
      uint32_t stage = 0, phase = 0, acc = 0, acc_phase = 0;
      bool ok = true;
      for (int u = blockIdx.x; u < total && ok; u += gridDim.x) {
        if (!mbar_wait(tempty0 + 8 * acc, acc_phase ^ 1, abort_flag, p.hdr, 0x20000u | MODE)) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + acc * BN;
        for (int kb = 0; kb < nk; ++kb) {
          if (!mbar_wait(full0 + 8 * stage, phase, abort_flag, p.hdr, 0x30000u | MODE)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a_addr = smem_u32(smem + stage * STAGE_BYTES);
          const uint32_t b_addr = a_addr + A_BYTES;
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {  // 4 x 32 bytes of K per stage: K=16 bf16 or K=32 e4m3 each
            if (F8)
              mma_f8(d_tmem, sw128_kmajor_desc(a_addr + kk * 32), sw128_kmajor_desc(b_addr + kk * 32), idesc,
                     (kb | kk) != 0);
            else
              mma_f16(d_tmem, sw128_kmajor_desc(a_addr + kk * 32), sw128_kmajor_desc(b_addr + kk * 32), idesc,
                      (kb | kk) != 0);
          }
          mma_commit(empty0 + 8 * stage);
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1;
          }
        }
        if (!ok) break;
        mma_commit(tfull0 + 8 * acc);
        acc ^= 1;
        if (acc == 0) acc_phase ^= 1;
      }
      // every MMA issued by this thread has completed once mma_done fires
      mma_commit(mma_done);
      mbar_wait_quiet(mma_done, 0, 1000000000ull);
    }
    __syncwarp();
  } else if (warp >= 4) {
    // ---------------------------------------------------------------- epilogue
    // NH warps per 32-lane TMEM quadrant q; warp h of a quadrant drains 1/NH of
    // the accumulator's columns (Gate/Up: its gate columns with the matching up
    // columns; Down: a contiguous range of output columns).
    constexpr int NH = epi_warps(MODE, F8) / 4;  // warps per TMEM quadrant
    const int e8 = warp - 4;
    const int q = e8 & 3, h = e8 >> 2;
    const int row = q * 32 + lane;
    uint32_t acc = 0, acc_phase = 0;
    for (int u = blockIdx.x; u < total; u += gridDim.x) {
      const int tile = u / p.nN, n = u - (u / p.nN) * p.nN;
      const int4 tl = tiles[tile];
      const int row0 = tl.y, nrows = tl.z;
      int good = 1;
      if (lane == 0) good = mbar_wait(tfull0 + 8 * acc, acc_phase, abort_flag, p.hdr, 0x40000u | MODE);
      good = __shfl_sync(0xffffffffu, good, 0);
      if (!good) break;
      tc_fence_after();
      const uint32_t tbase = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + acc * BN;
      if (MODE == MODE_GATEUP) {
        // bf16: direct stores (each thread writes whole 64-byte pieces of its own
        // sorted row).  F8: a = silu(sc g) * (sc u) with sc = s_x * s_w1[e]; the
        // amax of a (fp32) for the per-tensor quantisation of h is recorded here, and
        // a itself is kept in bf16 for that second pass: the two 32-column halves of
        // a warp's 64 columns fill one [32 rows][64 bf16] box of its staging
        // (128-byte swizzle), stored by TMA when all 32 rows belong to the tile.
        const float sc = F8 ? e4m3_scale(__uint_as_float(*p.amax_in)) * wscale_of(p, tl.x) : 1.0f;
        float amax = 0.0f;
        __nv_bfloat16* out_row = p.out + static_cast<size_t>(row0 + row) * p.out_ld;
        constexpr int GC = BN / 2 / NH;  // gate columns of this warp (and as many up columns)
#pragma unroll 1
        for (int c = h * GC; c < h * GC + GC; c += 32) {
          float g[32], up[32];
          tmem_ld32(tbase + c, g);
          tmem_ld32(tbase + BN / 2 + c, up);
          tmem_ld_wait();
          if (c == h * GC + GC - 32) {  // this warp's last columns read: release the accumulator
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(tempty0 + 8 * acc);
          }
          const int col = n * (BN / 2) + c;
          if (F8) {
            static_assert(MODE != MODE_GATEUP || !F8 || GC == 64, "F8 Gate/Up: 64 columns (two halves of 32) per warp");
            uint8_t* stg = smem + STAGING_OFFSET + e8 * 4096;
            const int wrows = min(32, nrows - q * 32), wrow0 = row0 + q * 32;
            const int half = (c - h * GC) >> 5;  // which 32 of the box's 64 columns
            if (half == 0) {
              if (lane == 0) bulk_wait_group_read0();  // the previous box has left the staging
              __syncwarp();
            }
            float hv[32];
#pragma unroll
            for (int i = 0; i < 32; ++i) hv[i] = silu_mul(sc * g[i], sc * up[i]);
            const bool valid = row < nrows && col < p.n_valid;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              *reinterpret_cast<uint4*>(stg + lane * 128 + (((half * 4 + i) ^ (lane & 7)) << 4)) = pack_bf16x8(hv + 8 * i);
              if (valid)
#pragma unroll
                for (int j = 0; j < 8; ++j) amax = fmaxf(amax, fabsf(hv[8 * i + j]));
            }
            if (half == 1) {
              const int col0 = col - 32;  // the box's first column (a multiple of 64; I % 64 == 0)
              if (wrows == 32) {
                fence_proxy_async_shared();
                __syncwarp();
                if (lane == 0) {
                  if (col0 < p.n_valid) tma_store_2d(&tmO, smem_u32(stg), col0, wrow0);
                  bulk_commit_group();
                }
                __syncwarp();
              } else {
                __syncwarp();
#pragma unroll
                for (int it = 0; it < 8; ++it) {  // 4 rows of 64 bf16 (8 lanes each) per instruction
                  const int r = it * 4 + (lane >> 3), j = lane & 7;
                  if (r < wrows && col0 + 8 * j < p.n_valid)
                    *reinterpret_cast<uint4*>(p.out_a + static_cast<size_t>(wrow0 + r) * p.out_ld + col0 + 8 * j) =
                        *reinterpret_cast<const uint4*>(stg + r * 128 + ((j ^ (r & 7)) << 4));
                }
                __syncwarp();
              }
            }
          } else if (row < nrows && col < p.n_valid) {
            float hv[32];
#pragma unroll
            for (int i = 0; i < 32; ++i) hv[i] = silu_mul(g[i], up[i]);
            uint4* dst = reinterpret_cast<uint4*>(out_row + col);
#pragma unroll
            for (int i = 0; i < 4; ++i) dst[i] = pack_bf16x8(hv + 8 * i);
          }
        }
        if (F8) {
          amax = warp_max(amax);
          if (lane == 0 && amax > 0.0f) atomicMax(p.amax_out, __float_as_uint(amax));
        }
      } else {
        // Down: o rows in sorted order.  Each pass stages 128 bf16 columns of the
        // warp's 32 rows in shared memory as two [32 rows][128 bytes] boxes with the
        // 128-byte swizzle (16-byte chunk c of row r at c ^ (r & 7): both the row-per-
        // thread writes and the row-segment reads below take the minimum 4 wavefronts).
        // A warp whose 32 rows all belong to the tile hands the boxes to TMA stores
        // (lane 0 issues them; it waits for them to have read the staging before the
        // next pass overwrites it); a warp of a partial tile writes its valid rows with
        // 16-byte stores.  F8: o = s_h * s_w2[e] * acc.
        static_assert(MODE == MODE_GATEUP || epi_warps(MODE, F8) == 4, "Down epilogue: one warp per TMEM quadrant");
        uint8_t* stg = smem + STAGING_OFFSET + q * (32 * 256);
        const int wrows = min(32, nrows - q * 32);  // valid rows of this warp (may be <= 0)
        const float post = F8 ? e4m3_scale(__uint_as_float(*p.amax_in)) * wscale_of(p, tl.x) : 1.0f;
        const int wrow0 = row0 + q * 32;            // first o row of this warp
#pragma unroll 1
        for (int pass = 0; pass < 2; ++pass) {
          if (lane == 0) bulk_wait_group_read0();   // the staging's previous TMA stores have read it
          __syncwarp();
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            float v[32];
            tmem_ld32(tbase + pass * 128 + c * 32, v);
            tmem_ld_wait();
            if (F8) {
#pragma unroll
              for (int i = 0; i < 32; ++i) v[i] *= post;
            }
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              const int cc = c * 4 + i;  // 16-byte chunk of the row, 0..15
              *reinterpret_cast<uint4*>(stg + (cc >> 3) * 4096 + lane * 128 + (((cc & 7) ^ (lane & 7)) << 4)) =
                  pack_bf16x8(v + 8 * i);
            }
          }
          if (pass == 1) {  // every accumulator column read: hand the buffer back to the MMA
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(tempty0 + 8 * acc);  // one arrival per warp
          }
          const int col0 = n * BN + pass * 128;
          if (wrows == 32) {
            fence_proxy_async_shared();
            __syncwarp();
            if (lane == 0) {
#pragma unroll
              for (int b = 0; b < 2; ++b)
                if (col0 + b * 64 < p.n_valid) tma_store_2d(&tmO, smem_u32(stg + b * 4096), col0 + b * 64, wrow0);
              bulk_commit_group();
            }
            __syncwarp();
          } else {
            __syncwarp();
#pragma unroll 4
            for (int it = 0; it < 16; ++it) {
              const int r = it * 2 + (lane >> 4), j = lane & 15;
              const int col = col0 + j * 8;
              if (r < wrows && col < p.n_valid)
                *reinterpret_cast<uint4*>(p.out + static_cast<size_t>(wrow0 + r) * p.out_ld + col) =
                    *reinterpret_cast<const uint4*>(stg + (j >> 3) * 4096 + r * 128 + (((j & 7) ^ (r & 7)) << 4));
            }
            __syncwarp();
          }
        }
      }
      acc ^= 1;
      if (acc == 0) acc_phase ^= 1;
    }
    if ((MODE == MODE_DOWN || F8) && lane == 0) bulk_wait_group0();  // this warp's TMA stores have completed
    __syncwarp();
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 2) {
    tc_fence_after();
    tmem_dealloc(tmem_base, TMEM_COLS);
  }
}

static bool encode_2d(CUtensorMap* map, const void* base, uint64_t inner, uint64_t outer, uint32_t box_inner,
                      uint32_t box_outer, bool u8 = false) {
  EncodeTiledFn fn = get_encode_tiled();
  if (!fn) return false;
  const cuuint64_t dims[2] = {inner, outer};
  const cuuint64_t strides[1] = {inner * (u8 ? 1 : 2)};
  const cuuint32_t box[2] = {box_inner, box_outer};
  const cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(map, u8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base),
                  dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

template <int MODE, bool F8>
static cudaError_t set_smem_attr() {
  static cudaError_t st = cudaFuncSetAttribute(grouped_gemm_kernel<MODE, F8>,
                                               cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SMEM_BYTES);
  return st;
}

}  // namespace gg

namespace gg {

static cudaError_t prepare(const GroupedArgs& a, int* sms) {
  const cudaError_t e[4] = {set_smem_attr<MODE_GATEUP, false>(), set_smem_attr<MODE_DOWN, false>(),
                            set_smem_attr<MODE_GATEUP, true>(), set_smem_attr<MODE_DOWN, true>()};
  for (cudaError_t x : e)
    if (x != cudaSuccess) return x;
  *sms = num_sms();
  return *sms > 0 ? cudaSuccess : cudaErrorNoDevice;
}

static Params base_params(const GroupedArgs& a) {
  Params p{};
  p.tiles = a.tiles;
  p.num_tiles = a.num_tiles;
  p.max_tiles = a.max_tiles;
  p.perm = a.perm;
  p.k = a.k;
  p.hdr = a.hdr;
  p.E = a.E;
  p.wscale = a.w1_scale;
  return p;
}

}  // namespace gg

// Gate/Up: N tiles of 128 h columns (gate 128 + up 128 accumulator columns).
cudaError_t launch_gateup_bf16(const GroupedArgs& a, cudaStream_t s) {
  using namespace gg;
  if (a.R <= 0) return cudaSuccess;
  int sms = 0;
  cudaError_t err = prepare(a, &sms);
  if (err != cudaSuccess) return err;
  CUtensorMap tmx, tmw1, tmw1s;
  const bool gather = a.xs == nullptr && !a.f8;
  const uint32_t bke = a.f8 ? 128 : BK;
  if (!(gather ? encode_2d(&tmx, a.x, a.H, a.T, BK, 1) : encode_2d(&tmx, a.xs, a.H, a.R, bke, BM, a.f8)) ||
      !encode_2d(&tmw1, a.w1, a.H, static_cast<uint64_t>(a.E) * 2 * a.I, bke, BN / 2, a.f8))
    return cudaErrorInvalidValue;
  tmw1s = tmw1;
  if (a.S > 0 && !encode_2d(&tmw1s, a.w1s, a.H, static_cast<uint64_t>(a.S) * 2 * a.I, bke, BN / 2, a.f8))
    return cudaErrorInvalidValue;
  Params p = base_params(a);
  p.a_gather = gather ? 1 : 0;
  p.wscale = a.w1_scale;
  p.wscale2 = a.w1s_scale;
  p.amax_in = &a.hdr->amax_x;
  p.amax_out = &a.hdr->amax_h;
  p.out_a = static_cast<__nv_bfloat16*>(a.a_bf16);
  CUtensorMap tmab = tmx;  // F8: a [R rows][I] bf16, stored in [32 rows][64 columns] boxes
  if (a.f8 && !encode_2d(&tmab, a.a_bf16, a.I, a.R, 64, 32)) return cudaErrorInvalidValue;
  p.nN = (a.I + BN / 2 - 1) / (BN / 2);
  p.K = a.H;
  p.b_rows_per_expert = 2 * a.I;
  p.up_offset = a.I;
  p.n_valid = a.I;
  p.out_ld = a.I;
  p.out = static_cast<__nv_bfloat16*>(a.h);
  const long long units = static_cast<long long>(a.max_tiles) * p.nN;
  const int grid = static_cast<int>(units < sms ? units : sms);
  stage_begin("gateup_gemm", s);
  if (a.f8)
    err = launch_dependent(grouped_gemm_kernel<MODE_GATEUP, true>, dim3(grid), dim3(threads_of(MODE_GATEUP, true)),
                           SMEM_BYTES, s, tmx, tmw1, tmab, tmw1s, p);
  else
    err = launch_dependent(grouped_gemm_kernel<MODE_GATEUP, false>, dim3(grid), dim3(threads_of(MODE_GATEUP, false)),
                           SMEM_BYTES, s, tmx, tmw1, tmx, tmw1s, p);
  stage_end(s);
  return err;
}

// Down: N tiles of 256 output columns of H.
cudaError_t launch_down_bf16(const GroupedArgs& a, cudaStream_t s) {
  using namespace gg;
  if (a.R <= 0) return cudaSuccess;
  int sms = 0;
  cudaError_t err = prepare(a, &sms);
  if (err != cudaSuccess) return err;
  CUtensorMap tmh, tmw2, tmo, tmw2s;
  const uint32_t bke = a.f8 ? 128 : BK;
  // o: bf16 [R rows][H], stored by the epilogue in [32 rows][64 columns] boxes
  if (!encode_2d(&tmh, a.h, a.I, a.R, bke, BM, a.f8) ||
      !encode_2d(&tmw2, a.w2, a.I, static_cast<uint64_t>(a.E) * a.H, bke, BN, a.f8) ||
      !encode_2d(&tmo, a.o, a.H, a.R, 64, 32))
    return cudaErrorInvalidValue;
  tmw2s = tmw2;
  if (a.S > 0 && !encode_2d(&tmw2s, a.w2s, a.I, static_cast<uint64_t>(a.S) * a.H, bke, BN, a.f8))
    return cudaErrorInvalidValue;
  Params p = base_params(a);
  p.wscale = a.w2_scale;
  p.wscale2 = a.w2s_scale;
  p.amax_in = &a.hdr->amax_h;
  p.nN = (a.H + BN - 1) / BN;
  p.K = a.I;
  p.b_rows_per_expert = a.H;
  p.up_offset = 0;
  p.n_valid = a.H;
  p.out_ld = a.H;
  p.out = static_cast<__nv_bfloat16*>(a.o);
  const long long units = static_cast<long long>(a.max_tiles) * p.nN;
  const int grid = static_cast<int>(units < sms ? units : sms);
  stage_begin("down_gemm", s);
  if (a.f8)
    err = launch_dependent(grouped_gemm_kernel<MODE_DOWN, true>, dim3(grid), dim3(threads_of(MODE_DOWN, true)),
                           SMEM_BYTES, s, tmh, tmw2, tmo, tmw2s, p);
  else
    err = launch_dependent(grouped_gemm_kernel<MODE_DOWN, false>, dim3(grid), dim3(threads_of(MODE_DOWN, false)),
                           SMEM_BYTES, s, tmh, tmw2, tmo, tmw2s, p);
  stage_end(s);
  return err;
}

// ------------------------------------------------------------------ combine
// y[t, c] = bf16( sum_{j < k} w[t, j] * o[row(t*k + j), c] ), fp32, j ascending
// (the final top-k reduction of the route-MMA page's Motivation), with
// row(r) = inv[r] for the grouped path's expert-sorted o and row(r) = r for the
// route-direct path's route-order o.  Deterministic: no atomics, fixed
// summation order.
// Loads the 8 values of route row r at column c as fp32.
template <typename OT>
__device__ __forceinline__ void combine_load8(const OT* __restrict__ o, long long r, int H, int c, float (&v)[8],
                                              uint64_t pol) {
  if (r < 0) {
#pragma unroll
    for (int i = 0; i < 8; ++i) v[i] = 0.0f;
  } else if (sizeof(OT) == 2) {
    const uint4 raw = ld_nc_v4_hint(o + r * H + c, pol);
    const __nv_bfloat162* b = reinterpret_cast<const __nv_bfloat162*>(&raw);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 f = __bfloat1622float2(b[i]);
      v[2 * i] = f.x;
      v[2 * i + 1] = f.y;
    }
  } else {
    const float4 f0 = __ldg(reinterpret_cast<const float4*>(o + r * H + c));
    const float4 f1 = __ldg(reinterpret_cast<const float4*>(o + r * H + c) + 1);
    v[0] = f0.x; v[1] = f0.y; v[2] = f0.z; v[3] = f0.w;
    v[4] = f1.x; v[5] = f1.y; v[6] = f1.z; v[7] = f1.w;
  }
}

// The k rows of a token are loaded four at a time before any of them is summed,
// so each thread keeps four loads in flight; the sum still runs j ascending.
// Then the token's rows T*k + s*T + t of the S shared experts are added with
// weight 1, s ascending.  YF32: y is the unrounded fp32 sum.
template <typename OT, bool YF32>
__global__ void __launch_bounds__(256) combine_kernel(const OT* __restrict__ o, const float* __restrict__ w, int T,
                                                      int k, int H, void* __restrict__ y,
                                                      const int32_t* __restrict__ inv, int S) {
  // launched as a programmatic dependent (route-direct path): wait for the producer
  // of o; a no-op for an ordinary launch
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int cpt = H / 8;
  const size_t total = static_cast<size_t>(T) * cpt;
  const uint64_t pol = l2_evict_first_policy();
  for (size_t idx = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; idx < total;
       idx += static_cast<size_t>(gridDim.x) * blockDim.x) {
    const int t = static_cast<int>(idx / cpt);
    const int c = static_cast<int>(idx - static_cast<size_t>(t) * cpt) * 8;
    const size_t r0 = static_cast<size_t>(t) * k;
    float acc[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) acc[i] = 0.0f;
    int j = 0;
    for (; j + 4 <= k; j += 4) {
      float v[4][8], wj[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        wj[q] = __ldg(w + r0 + j + q);
        combine_load8(o, inv ? __ldg(inv + r0 + j + q) : static_cast<long long>(r0 + j + q), H, c, v[q], pol);
      }
#pragma unroll
      for (int q = 0; q < 4; ++q)
#pragma unroll
        for (int i = 0; i < 8; ++i) acc[i] = fmaf(wj[q], v[q][i], acc[i]);
    }
    for (; j < k; ++j) {
      float v[8];
      const float wj = __ldg(w + r0 + j);
      combine_load8(o, inv ? __ldg(inv + r0 + j) : static_cast<long long>(r0 + j), H, c, v, pol);
#pragma unroll
      for (int i = 0; i < 8; ++i) acc[i] = fmaf(wj, v[i], acc[i]);
    }
    for (int sx = 0; sx < S; ++sx) {
      float v[8];
      combine_load8(o, static_cast<long long>(T) * k + static_cast<long long>(sx) * T + t, H, c, v, pol);
#pragma unroll
      for (int i = 0; i < 8; ++i) acc[i] += v[i];
    }
    if (YF32) {
      float4* dst = reinterpret_cast<float4*>(static_cast<float*>(y) + static_cast<size_t>(t) * H + c);
      dst[0] = make_float4(acc[0], acc[1], acc[2], acc[3]);
      dst[1] = make_float4(acc[4], acc[5], acc[6], acc[7]);
    } else {
      *reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(y) + static_cast<size_t>(t) * H + c) =
          gg::pack_bf16x8(acc);
    }
  }
}

// y = bf16(y32): 8 values per thread and iteration.
__global__ void __launch_bounds__(256) round_bf16_kernel(const float4* __restrict__ y32, uint4* __restrict__ y,
                                                         size_t n8) {
  for (size_t i = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; i < n8;
       i += static_cast<size_t>(gridDim.x) * blockDim.x) {
    const float4 a = __ldg(y32 + 2 * i), b = __ldg(y32 + 2 * i + 1);
    const float v[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
    y[i] = gg::pack_bf16x8(v);
  }
}

cudaError_t launch_round_bf16(const float* y32, void* y, size_t n, cudaStream_t s) {
  const size_t n8 = n / 8;
  if (n8 == 0) return cudaSuccess;
  const int sms = num_sms();
  size_t blocks = (n8 + 255) / 256;
  const size_t cap = static_cast<size_t>(sms > 0 ? sms : 148) * 8;
  if (blocks > cap) blocks = cap;
  stage_begin("round_bf16", s);
  round_bf16_kernel<<<static_cast<unsigned>(blocks), 256, 0, s>>>(reinterpret_cast<const float4*>(y32),
                                                                  static_cast<uint4*>(y), n8);
  const cudaError_t err = cudaGetLastError();
  stage_end(s);
  return err;
}

cudaError_t launch_combine_pdl(const CombineArgs& a, cudaStream_t s) {
  if (a.T <= 0) return cudaSuccess;
  const size_t total = static_cast<size_t>(a.T) * (a.H / 8);
  const int sms = num_sms();
  size_t blocks = (total + 255) / 256;
  const size_t cap = static_cast<size_t>(sms > 0 ? sms : 148) * 8;
  if (blocks > cap) blocks = cap;
  cudaLaunchAttribute pdl[1];
  pdl[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  pdl[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(static_cast<unsigned>(blocks));
  cfg.blockDim = dim3(256);
  cfg.stream = s;
  cfg.attrs = pdl;
  cfg.numAttrs = 1;
  stage_begin("combine", s);
  const float* of = static_cast<const float*>(a.o);
  const __nv_bfloat16* ob = static_cast<const __nv_bfloat16*>(a.o);
  cudaError_t err;
  if (a.o_is_f32)
    err = a.y_f32 ? cudaLaunchKernelEx(&cfg, combine_kernel<float, true>, of, a.w, a.T, a.k, a.H, a.y, a.inv, a.S)
                  : cudaLaunchKernelEx(&cfg, combine_kernel<float, false>, of, a.w, a.T, a.k, a.H, a.y, a.inv, a.S);
  else
    err = a.y_f32
              ? cudaLaunchKernelEx(&cfg, combine_kernel<__nv_bfloat16, true>, ob, a.w, a.T, a.k, a.H, a.y, a.inv, a.S)
              : cudaLaunchKernelEx(&cfg, combine_kernel<__nv_bfloat16, false>, ob, a.w, a.T, a.k, a.H, a.y, a.inv, a.S);
  stage_end(s);
  return err;
}

cudaError_t launch_combine(const CombineArgs& a, cudaStream_t s) { return launch_combine_pdl(a, s); }

}  // namespace moe
