// Grouped GEMMs for 128x128-blockwise FP8 ("perf: add small-batch route MMA for
// MoE", Summary: 128x128 blockwise FP8; the grouped path of its Motivation).
//
// The weights carry one fp32 scale per 128x128 block and the activations one
// per (row, 128 columns), so every 128-wide K block has its own scale pair and
// the products cannot be summed inside one accumulator.  Each K block is a
// 128-byte stage of e4m3: the MMA thread writes that block's partial product
// (tcgen05.mma kind::f8f6f4, M=128, N=256, 4 x K=32) into one of two 256-column
// TMEM buffers, and eight epilogue warps read it with tcgen05.ld, multiply by
// s_a[row, kb] * s_w[block, kb] and add it into fp32 registers ("promotion")
// while the MMA fills the other buffer.  Two warps share each 32-lane TMEM
// quadrant (one accumulator row per thread), each holding 128 of the 256
// columns.  A 256-column tile moves 96 bytes of operands per MMA cycle where a
// 128-column one moves 128: the tile width, not the promotion, bounded the
// 128-column version of these kernels.
//
// Gate/Up: a work item is (row tile, group g of 128 h columns); B = the 128 gate
//   rows [g*128, g*128 + 128) and the matching 128 up rows [I + g*128, ...) of
//   W1[e] (two 128-row TMA boxes), so one K loop covers a whole scale group of h.
//   Warp c of a quadrant holds gate columns [64c, 64c + 64) and the matching up
//   columns of its rows; after the last K block it computes a = silu(g) * u, the
//   two warps exchange their row maxima through shared memory (bounded mbarrier
//   waits), and each quantises its 64 values of the row with the group's scale
//   amax / 448 straight into e4m3 h and the fp32 scale.  In a ragged last group
//   (I % 128 == 64) the warp whose columns are >= I skips its stores and
//   contributes 0 to the row maximum.
// Down: a work item is (row tile, 256 rows n of W2[e], two weight scale blocks);
//   warp c holds o columns [n*256 + 128c, + 128) (one scale block) and writes them
//   as bf16 for the tile's sorted rows, staged in shared memory in two passes of
//   64 columns.  A ragged last N tile (H % 256 == 128) has no columns for c = 1.
#include "common.cuh"
#include "internal.h"

namespace moe {
namespace gb {

constexpr int BM = kGemmBM;  // 128
constexpr int BN = 256;
constexpr int BKB = 128;     // K bytes (= e4m3 elements) per stage, one scale block
constexpr int STAGES = 4;
constexpr int A_BYTES = BM * BKB;  // 16 KB
constexpr int B_BYTES = BN * BKB;  // 32 KB: two 128-row boxes
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
constexpr int NBUF = 2;            // TMEM partial buffers of 256 columns
constexpr int TMEM_COLS = NBUF * BN;
constexpr int EPI_WARPS = 8;       // warps 2..9 (the block's registers come in 4-warp groups: 168 a thread)
constexpr int THREADS = 32 * (2 + EPI_WARPS);
constexpr int NUM_BARS = 2 * STAGES + 2 * NBUF + 8;
constexpr int BAR_OFFSET = STAGES * STAGE_BYTES;
// epilogue scratch, 1024-byte aligned: Gate/Up row maxima [8 warps][32] fp32; Down output
// staging [8 warps][32 rows][128 bytes], each warp's 4 KB a 128-byte-swizzled TMA store box
constexpr int SCRATCH_OFFSET = (BAR_OFFSET + 256 + 1023) / 1024 * 1024;
constexpr int SCRATCH_BYTES = EPI_WARPS * 32 * 128;
constexpr size_t SMEM_BYTES = 1024 + SCRATCH_OFFSET + SCRATCH_BYTES;
static_assert(NUM_BARS * 8 + 8 <= 256, "barrier region");
static_assert(SMEM_BYTES <= 232448, "shared memory per block");

constexpr int MODE_GATEUP = 0;
constexpr int MODE_DOWN = 1;

struct Params {
  const int32_t* tiles;
  const int32_t* num_tiles;
  int max_tiles;
  int nN;          // work items per row tile (Gate/Up: 128-column groups of h; Down: 256-column tiles of o)
  int K;           // reduction length (bytes = elements)
  int I, H;
  const float* a_scale;  // [R][ceil(K/128)] scales of the A rows (sorted order)
  const float* w_scale;  // Gate/Up: [E][2I/128][H/128]; Down: [E][H/128][ceil(I/128)]
  const float* w_scale2; // the same for the S shared experts (tiles of expert E + s, weights in tmB2)
  int E;
  uint8_t* h;            // Gate/Up: e4m3 h [R][I]
  float* h_scale;        // Gate/Up: [R][ceil(I/128)]
  __nv_bfloat16* out;    // Down: o [R][H]
  DeviceHeader* hdr;
};


// silu(g) * u with the fast exponential and division intrinsics: a is rounded to
// e4m3 next, far coarser than their error.  Here the SwiGLU runs in the tile's
// epilogue tail after the last K block's promotion, which nothing overlaps (the
// accurate form costs this kernel 21 us at T=16384; the bf16 and per-tensor
// kernels hide it behind the next tile's mainloop and keep silu_mul).
__device__ __forceinline__ float silu_mul_fast(float g, float u) { return __fdividef(g, 1.0f + __expf(-g)) * u; }

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

// 32 values * inv -> 32 e4m3 codes (RNE, saturating), as two 16-byte stores.  inv is
// the correctly rounded 1 / s: a * inv can differ from the quotient a / s by one fp32
// ulp, which changes an e4m3 code only for a value within one ulp of a rounding
// midpoint (h's codes are not unique anyway: a itself carries the tensor cores'
// summation order).
__device__ __forceinline__ void store_e4m3x32(uint8_t* dst, const float* a, float inv) {
  uint32_t w[8];
#pragma unroll
  for (int i = 0; i < 8; ++i)
    w[i] = static_cast<uint32_t>(cvt_e4m3x2(a[4 * i] * inv, a[4 * i + 1] * inv)) |
           (static_cast<uint32_t>(cvt_e4m3x2(a[4 * i + 2] * inv, a[4 * i + 3] * inv)) << 16);
  reinterpret_cast<uint4*>(dst)[0] = make_uint4(w[0], w[1], w[2], w[3]);
  reinterpret_cast<uint4*>(dst)[1] = make_uint4(w[4], w[5], w[6], w[7]);
}

// Work items: Gate/Up pairs (row tile, group g = units 2g and 2g + 1, or just 2g for

template <int MODE>
__global__ void __launch_bounds__(THREADS, 1)
    grouped_blockwise_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                             const __grid_constant__ CUtensorMap tmB2, const __grid_constant__ CUtensorMap tmO,
                             const Params p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + BAR_OFFSET);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + NUM_BARS);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  uint8_t* scratch = smem + SCRATCH_OFFSET;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t full0 = smem_u32(bars), empty0 = smem_u32(bars + STAGES);
  const uint32_t pfull0 = smem_u32(bars + 2 * STAGES), pempty0 = smem_u32(bars + 2 * STAGES + NBUF);
  // Gate/Up, per quadrant q: xbar0 + 8q (row maxima written), xbar0 + 8 (4 + q) (row maxima read)
  const uint32_t xbar0 = smem_u32(bars + 2 * STAGES + 2 * NBUF);

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(full0 + 8 * s, 1);
      mbar_init(empty0 + 8 * s, 1);
    }
    for (int b = 0; b < NBUF; ++b) {
      mbar_init(pfull0 + 8 * b, 1);
      mbar_init(pempty0 + 8 * b, EPI_WARPS);  // one arrival per epilogue warp
    }
    for (int b = 0; b < 8; ++b) mbar_init(xbar0 + 8 * b, 2);  // the two warps of a quadrant
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tensormap(&tmA);
    prefetch_tensormap(&tmB);
    prefetch_tensormap(&tmB2);
    if (MODE == MODE_DOWN) prefetch_tensormap(&tmO);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  dep_wait();  // the tile map, the A rows and their scales come from the kernels before

  const int ntiles = min(*p.num_tiles, p.max_tiles);
  const int items = ntiles * p.nN;
  const int nk = (p.K + BKB - 1) / BKB;
  const int4* tiles = reinterpret_cast<const int4*>(p.tiles);

  if (warp == 0) {
    // ---------------------------------------------------------------- producer
    uint32_t stage = 0, phase = 0;
    int issued = 0;
    bool ok = true;
    for (int it = blockIdx.x; it < items && ok; it += gridDim.x) {
      const int tile = it / p.nN, n = it - tile * p.nN;
      const int4 tl = tiles[tile];
      const bool shx = tl.x >= p.E;  // a shared expert's tile: its own weight tensor
      const int e = shx ? tl.x - p.E : tl.x;
      const CUtensorMap* tb = shx ? &tmB2 : &tmB;
      // B: Gate/Up the 128 gate rows of group n and the matching 128 up rows; Down 256 rows of W2[e]
      const int brow0 = MODE == MODE_GATEUP ? e * 2 * p.I + n * 128 : e * p.H + n * BN;
      const int brow1 = MODE == MODE_GATEUP ? brow0 + p.I : brow0 + 128;
      for (int kb = 0; kb < nk; ++kb) {
        int good = 1;
        if (lane == 0) good = mbar_wait(empty0 + 8 * stage, phase ^ 1, abort_flag, p.hdr, 0x80000u | MODE);
        if (!__shfl_sync(0xffffffffu, good, 0)) {
          ok = false;
          break;
        }
        if (lane == 0) {
          const uint32_t full = full0 + 8 * stage;
          const uint32_t a_dst = smem_u32(smem + stage * STAGE_BYTES), b_dst = a_dst + A_BYTES;
          const int kc = kb * BKB;
          mbar_arrive_expect_tx(full, STAGE_BYTES);
          tma_load_2d(a_dst, &tmA, kc, tl.y, full);
          tma_load_2d(b_dst, tb, kc, brow0, full);
          tma_load_2d(b_dst + B_BYTES / 2, tb, kc, brow1, full);
        }
        __syncwarp();
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
      const uint32_t idesc = make_idesc(0, 0, BM, BN);
      uint32_t stage = 0, phase = 0, pb = 0, pphase = 0;
      bool ok = true;
      for (int it = blockIdx.x; it < items && ok; it += gridDim.x) {
        for (int kb = 0; kb < nk; ++kb) {
          if (!mbar_wait(full0 + 8 * stage, phase, abort_flag, p.hdr, 0x81000u | MODE) ||
              !mbar_wait(pempty0 + 8 * pb, pphase ^ 1, abort_flag, p.hdr, 0x82000u | MODE)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a_addr = smem_u32(smem + stage * STAGE_BYTES), b_addr = a_addr + A_BYTES;
          const uint32_t d_tmem = tmem_base + pb * BN;
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)  // a fresh partial for this K block
            mma_f8(d_tmem, sw128_kmajor_desc(a_addr + kk * 32), sw128_kmajor_desc(b_addr + kk * 32), idesc, kk != 0);
          mma_commit(empty0 + 8 * stage);
          mma_commit(pfull0 + 8 * pb);
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1;
          }
          if (++pb == NBUF) {
            pb = 0;
            pphase ^= 1;
          }
        }
      }
      // wait for every MMA issued by this thread before TMEM is released (the last
      // committed buffer; a fresh barrier passes at once when nothing was issued)
      const uint32_t lb = (pb + NBUF - 1) % NBUF;
      mbar_wait_quiet(pfull0 + 8 * lb, pb == 0 ? (pphase ^ 1) : pphase, 1000000000ull);
    }
    __syncwarp();
  } else {
    // ---------------------------------------------------------------- epilogue (promotion)
    const int e8 = warp - 2;
    const int q = warp & 3;   // TMEM lane quadrant
    const int c = e8 >> 2;    // which 128 of the tile's 256 accumulator columns (Gate/Up: 64 gate + 64 up)
    const int row = q * 32 + lane;
    float* rowmax = reinterpret_cast<float*>(scratch);  // Gate/Up: [8 warps][32]
    uint32_t pb = 0, pphase = 0, xphase = 0;
    bool ok = true;
    for (int it = blockIdx.x; it < items && ok; it += gridDim.x) {
      const int tile = it / p.nN, n = it - tile * p.nN;
      const int4 tl = tiles[tile];
      const int row0 = tl.y, nrows = tl.z;
      const bool shx = tl.x >= p.E;
      const int e = shx ? tl.x - p.E : tl.x;
      const float* wsc = shx ? p.w_scale2 : p.w_scale;
      // this warp's first output column: Gate/Up an h column, Down an o column
      const int col = MODE == MODE_GATEUP ? n * 128 + 64 * c : n * BN + 128 * c;
      const bool valid = col < (MODE == MODE_GATEUP ? p.I : p.H);
      const float* sa = p.a_scale + static_cast<size_t>(row0 + min(row, nrows - 1)) * nk;
      // weight scale rows: Gate/Up gate block col/128 and up block (I + col)/128 of
      // [E][2I/128][H/128]; Down block col/128 of [E][H/128][nk]
      const int wrows = MODE == MODE_GATEUP ? 2 * p.I / 128 : p.H / 128;
      const float* sw0 = wsc + (static_cast<size_t>(e) * wrows + col / 128) * nk;
      const float* sw1 = MODE == MODE_GATEUP ? wsc + (static_cast<size_t>(e) * wrows + (p.I + col) / 128) * nk : sw0;
      float acc[128];  // Gate/Up: [0, 64) gate, [64, 128) up
#pragma unroll
      for (int i = 0; i < 128; ++i) acc[i] = 0.0f;
      float sa_next = 0.0f, s0_next = 0.0f, s1_next = 0.0f;
      if (valid) {
        sa_next = __ldg(sa);
        s0_next = __ldg(sw0);
        s1_next = __ldg(sw1);
      }
      for (int kb = 0; kb < nk; ++kb) {
        const float sak = sa_next, s0k = s0_next, s1k = s1_next;
        if (valid && kb + 1 < nk) {
          sa_next = __ldg(sa + kb + 1);
          s0_next = __ldg(sw0 + kb + 1);
          s1_next = __ldg(sw1 + kb + 1);
        }
        int good = 1;
        if (lane == 0) good = mbar_wait(pfull0 + 8 * pb, pphase, abort_flag, p.hdr, 0x83000u | MODE);
        if (!__shfl_sync(0xffffffffu, good, 0)) {
          ok = false;
          break;
        }
        tc_fence_after();
        // Gate/Up: gate columns at 64c, up columns at 128 + 64c; Down: columns at 128c
        const uint32_t tq = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + pb * BN;
        const uint32_t t0 = tq + (MODE == MODE_GATEUP ? 64 * c : 128 * c);
        const uint32_t t1 = MODE == MODE_GATEUP ? tq + 128 + 64 * c : t0 + 64;
        const float s0 = sak * s0k, s1 = sak * s1k;
        float v[16];
        // 16 columns at a time (the accumulators take 128 of the 168 registers a thread)
#pragma unroll
        for (int h = 0; h < 4; ++h) {
          tmem_ld16(t0 + 16 * h, v);
          tmem_ld_wait_regs16(v);
#pragma unroll
          for (int i = 0; i < 16; i += 2) fma2(acc[16 * h + i], acc[16 * h + i + 1], v[i], v[i + 1], s0, s0);
        }
#pragma unroll
        for (int h = 0; h < 3; ++h) {
          tmem_ld16(t1 + 16 * h, v);
          tmem_ld_wait_regs16(v);
#pragma unroll
          for (int i = 0; i < 16; i += 2)
            fma2(acc[64 + 16 * h + i], acc[64 + 16 * h + i + 1], v[i], v[i + 1], s1, s1);
        }
        tmem_ld16(t1 + 48, v);
        tmem_ld_wait_regs16(v);
        // the last columns are in registers: hand the buffer back before their FMAs
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(pempty0 + 8 * pb);
#pragma unroll
        for (int i = 0; i < 16; i += 2) fma2(acc[112 + i], acc[113 + i], v[i], v[i + 1], s1, s1);
        if (++pb == NBUF) {
          pb = 0;
          pphase ^= 1;
        }
      }
      if (!ok) break;
      if (MODE == MODE_GATEUP) {
        float m = 0.0f;
#pragma unroll
        for (int i = 0; i < 64; ++i) {
          acc[i] = silu_mul_fast(acc[i], acc[64 + i]);  // a
          m = fmaxf(m, fabsf(acc[i]));
        }
        // the group's scale: row maximum over the quadrant's two warps (64 columns each)
        rowmax[e8 * 32 + lane] = (valid && row < nrows) ? m : 0.0f;
        __syncwarp();
        int good = 1;
        if (lane == 0) {
          mbar_arrive(xbar0 + 8 * q);
          good = mbar_wait(xbar0 + 8 * q, xphase, abort_flag, p.hdr, 0x84000u);
        }
        if (!__shfl_sync(0xffffffffu, good, 0)) {
          ok = false;
          break;
        }
        const float gm = fmaxf(rowmax[e8 * 32 + lane], rowmax[(e8 ^ 4) * 32 + lane]);
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(xbar0 + 8 * (4 + q));
          good = mbar_wait(xbar0 + 8 * (4 + q), xphase, abort_flag, p.hdr, 0x85000u);
        }
        if (!__shfl_sync(0xffffffffu, good, 0)) {
          ok = false;
          break;
        }
        xphase ^= 1;
        if (valid && row < nrows) {
          const float sc = e4m3_scale(gm);
          const float inv = 1.0f / sc;
          const size_t r = static_cast<size_t>(row0 + row);
          store_e4m3x32(p.h + r * p.I + col, acc, inv);
          store_e4m3x32(p.h + r * p.I + col + 32, acc + 32, inv);
          if (c == 0) p.h_scale[r * p.nN + n] = sc;
        }
      } else if (valid) {
        // o rows (sorted order, like h): each thread's 128 bf16 outputs go through this
        // warp's 4 KB of staging in two passes of 64 columns, 16-byte pieces placed as the
        // 128-byte swizzle has them (piece c of row r at c ^ (r & 7)); a warp whose 32 rows
        // all belong to the tile hands the box to a TMA tile store, otherwise it writes
        // four whole 128-byte row segments per store instruction.
        uint4* stg = reinterpret_cast<uint4*>(scratch) + e8 * (32 * 8);
        const int vrows = min(32, nrows - q * 32);  // valid rows of this warp (may be <= 0)
        const int slot = row0 + row;
#pragma unroll
        for (int pass = 0; pass < 2; ++pass) {
          if (lane == 0) bulk_wait_group_read0();  // the previous TMA store has read the staging
          __syncwarp();                            // and the previous pass's loads are done
#pragma unroll
          for (int i = 0; i < 8; ++i) stg[lane * 8 + (i ^ (lane & 7))] = pack_bf16x8(acc + 64 * pass + 8 * i);
          if (vrows == 32) {
            fence_proxy_async_shared();
            __syncwarp();
            if (lane == 0) {
              tma_store_2d(&tmO, smem_u32(stg), col + 64 * pass, row0 + q * 32);
              bulk_commit_group();
            }
          } else {
            __syncwarp();
#pragma unroll
            for (int it2 = 0; it2 < 8; ++it2) {
              const int r = it2 * 4 + (lane >> 3), j = lane & 7;
              const int rslot = __shfl_sync(0xffffffffu, slot, r);
              if (r < vrows)
                *reinterpret_cast<uint4*>(p.out + static_cast<size_t>(rslot) * p.H + col + 64 * pass + j * 8) =
                    stg[r * 8 + (j ^ (r & 7))];
            }
          }
        }
        __syncwarp();
      }
    }
    if (MODE == MODE_DOWN && lane == 0) bulk_wait_group0();  // this warp's TMA stores have completed
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, TMEM_COLS);
  }
}

static bool encode_u8(CUtensorMap* map, const void* base, uint64_t inner, uint64_t outer, uint32_t box_rows) {
  EncodeTiledFn fn = get_encode_tiled();
  if (!fn) return false;
  const cuuint64_t dims[2] = {inner, outer};
  const cuuint64_t strides[1] = {inner};
  const cuuint32_t box[2] = {static_cast<cuuint32_t>(BKB), box_rows};
  const cuuint32_t estr[2] = {1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// o [R][H] bf16 as TMA store boxes of 32 rows x 64 columns (128-byte swizzle).
static bool encode_o(CUtensorMap* map, void* base, uint64_t H, uint64_t R) {
  EncodeTiledFn fn = get_encode_tiled();
  if (!fn) return false;
  const cuuint64_t dims[2] = {H, R};
  const cuuint64_t strides[1] = {H * 2};
  const cuuint32_t box[2] = {64, 32};
  const cuuint32_t estr[2] = {1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, base, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
         CUDA_SUCCESS;
}

template <int MODE>
static cudaError_t smem_attr() {
  static const cudaError_t st = cudaFuncSetAttribute(grouped_blockwise_kernel<MODE>,
                                                     cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SMEM_BYTES);
  return st;
}

}  // namespace gb

cudaError_t launch_gateup_blockwise(const GroupedArgs& a, const float* xs_scale, float* h_scale, cudaStream_t s) {
  using namespace gb;
  if (a.R <= 0) return cudaSuccess;
  cudaError_t err = smem_attr<MODE_GATEUP>();
  if (err != cudaSuccess) return err;
  const int sms = num_sms();
  if (sms <= 0) return cudaErrorNoDevice;
  CUtensorMap tma, tmb, tmbs;
  if (!encode_u8(&tma, a.xs, a.H, a.R, BM) || !encode_u8(&tmb, a.w1, a.H, static_cast<uint64_t>(a.E) * 2 * a.I, 128))
    return cudaErrorInvalidValue;
  tmbs = tmb;
  if (a.S > 0 && !encode_u8(&tmbs, a.w1s, a.H, static_cast<uint64_t>(a.S) * 2 * a.I, 128))
    return cudaErrorInvalidValue;
  Params p{};
  p.tiles = a.tiles;
  p.num_tiles = a.num_tiles;
  p.max_tiles = a.max_tiles;
  p.nN = (a.I + 127) / 128;
  p.K = a.H;
  p.I = a.I;
  p.H = a.H;
  p.a_scale = xs_scale;
  p.w_scale = a.w1_scale;
  p.w_scale2 = a.w1s_scale;
  p.E = a.E;
  p.h = static_cast<uint8_t*>(a.h);
  p.h_scale = h_scale;
  p.hdr = a.hdr;
  const long long items = static_cast<long long>(a.max_tiles) * p.nN;
  const int grid = static_cast<int>(items < sms ? items : sms);
  stage_begin("gateup_gemm", s);
  err = launch_dependent(grouped_blockwise_kernel<MODE_GATEUP>, dim3(grid), dim3(THREADS), SMEM_BYTES, s, tma, tmb,
                         tmbs, tma, p);
  stage_end(s);
  return err;
}

cudaError_t launch_down_blockwise(const GroupedArgs& a, const float* h_scale, cudaStream_t s) {
  using namespace gb;
  if (a.R <= 0) return cudaSuccess;
  cudaError_t err = smem_attr<MODE_DOWN>();
  if (err != cudaSuccess) return err;
  const int sms = num_sms();
  if (sms <= 0) return cudaErrorNoDevice;
  CUtensorMap tma, tmb, tmbs, tmo;
  if (!encode_u8(&tma, a.h, a.I, a.R, BM) || !encode_u8(&tmb, a.w2, a.I, static_cast<uint64_t>(a.E) * a.H, 128) ||
      !encode_o(&tmo, a.o, a.H, a.R))
    return cudaErrorInvalidValue;
  tmbs = tmb;
  if (a.S > 0 && !encode_u8(&tmbs, a.w2s, a.I, static_cast<uint64_t>(a.S) * a.H, 128)) return cudaErrorInvalidValue;
  Params p{};
  p.tiles = a.tiles;
  p.num_tiles = a.num_tiles;
  p.max_tiles = a.max_tiles;
  p.nN = (a.H + BN - 1) / BN;
  p.K = a.I;
  p.I = a.I;
  p.H = a.H;
  p.a_scale = h_scale;
  p.w_scale = a.w2_scale;
  p.w_scale2 = a.w2s_scale;
  p.E = a.E;
  p.out = static_cast<__nv_bfloat16*>(a.o);
  p.hdr = a.hdr;
  const long long units = static_cast<long long>(a.max_tiles) * p.nN;
  const int grid = static_cast<int>(units < sms ? units : sms);
  stage_begin("down_gemm", s);
  err = launch_dependent(grouped_blockwise_kernel<MODE_DOWN>, dim3(grid), dim3(THREADS), SMEM_BYTES, s, tma, tmb, tmbs,
                         tmo, p);
  stage_end(s);
  return err;
}

}  // namespace moe
