// Grouped GEMMs for 128x128-blockwise FP8 ("perf: add small-batch route MMA for
// MoE", Summary: 128x128 blockwise FP8; the grouped path of its Motivation).
//
// The weights carry one fp32 scale per 128x128 block and the activations one
// per (row, 128 columns), so every 128-wide K block has its own scale pair and
// the products cannot be summed inside one accumulator.  Each K block is a
// 128-byte stage of e4m3: the MMA thread writes that block's partial product
// (tcgen05.mma kind::f8f6f4, M=128, N=128, 4 x K=32) into one of four TMEM
// buffers, and eight epilogue warps read it with tcgen05.ld, multiply by
// s_a[row, kb] * s_w[block, kb] and add it into fp32 registers ("promotion")
// while the MMA fills the next buffers.  Two warps share each 32-lane TMEM
// quadrant (one accumulator row per thread), each holding 64 of the 128
// columns, so the loads of one warp overlap the FMAs of the other.
//
// Gate/Up: N = 64 gate + the matching 64 up rows of W1[e] (two 64-row TMA
//   boxes), A = expert-sorted e4m3 x rows with their group scales.  Work items
//   are pairs of units (n = 2g, 2g + 1) of one row tile, processed one after the
//   other by the same CTA, so that the two units together cover the 128-column
//   group g of h: a warp holds 32 gate and the matching 32 up columns of a row
//   and computes a = silu(g) * u; after the first unit it keeps a in shared
//   memory, after the second the two warps of a quadrant exchange their row
//   maxima, and each quantises its 64 values of the row with the group's scale
//   amax / 448 straight into e4m3 h and the fp32 scale (a ragged last group of
//   64 columns is a single unit).
// Down: N = 128 rows of W2[e] (one weight scale block), A = e4m3 h rows with
//   their group scales; the epilogue writes bf16 o for the tile's sorted rows.
#include "common.cuh"
#include "internal.h"

namespace moe {
namespace gb {

constexpr int BM = kGemmBM;  // 128
constexpr int BN = 128;
constexpr int BKB = 128;  // K bytes (= e4m3 elements) per stage, one scale block
constexpr int MAX_STAGES = 6;
// Gate/Up: 6 stages, 32 KB of staging (the first unit's a of a pair) and 1 KB for
// the row maxima; Down: 5 stages and 32 KB of output staging.
__host__ __device__ constexpr int stages_of(int mode) { return mode == 0 ? 6 : 5; }
constexpr int A_BYTES = BM * BKB;
constexpr int B_BYTES = BN * BKB;
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
constexpr int NBUF = 4;           // TMEM partial buffers of 128 columns
constexpr int TMEM_COLS = NBUF * BN;
constexpr int EPI_WARPS = 8;      // warps 4..11
constexpr int THREADS = 32 * (4 + EPI_WARPS);
constexpr int NUM_BARS = 2 * MAX_STAGES + 2 * NBUF + 8;  // + the Gate/Up row-maximum exchange (2 per quadrant)
__host__ __device__ constexpr int staging_offset(int mode) { return (stages_of(mode) * STAGE_BYTES + 256 + 1023) / 1024 * 1024; }
constexpr int STAGING_BYTES = EPI_WARPS * 32 * 128;
constexpr int ROWMAX_BYTES = EPI_WARPS * 32 * 4;
__host__ __device__ constexpr size_t smem_bytes(int mode) {
  return 1024 + staging_offset(mode) + STAGING_BYTES + (mode == 0 ? ROWMAX_BYTES : 0);
}
static_assert(smem_bytes(0) <= 232448 && smem_bytes(1) <= 232448, "shared memory per block");

constexpr int MODE_GATEUP = 0;
constexpr int MODE_DOWN = 1;

struct Params {
  const int32_t* tiles;
  const int32_t* num_tiles;
  int max_tiles;
  const int32_t* perm;
  int nN;          // units per row tile (Gate/Up: 64 h columns each; Down: 128 o columns)
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
// a ragged last group); Down units (row tile, n).
__device__ __forceinline__ int items_per_tile(int mode, int nN) { return mode == 0 ? (nN + 1) / 2 : nN; }
__device__ __forceinline__ int subunits(int mode, int nN, int g) { return mode == 0 ? min(2, nN - 2 * g) : 1; }

template <int MODE>
__global__ void __launch_bounds__(THREADS, 1)
    grouped_blockwise_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                             const __grid_constant__ CUtensorMap tmO, const __grid_constant__ CUtensorMap tmB2,
                             const Params p) {
  constexpr int STAGES = stages_of(MODE);
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + STAGES * STAGE_BYTES);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + NUM_BARS);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t full0 = smem_u32(bars), empty0 = smem_u32(bars + STAGES);
  const uint32_t pfull0 = smem_u32(bars + 2 * STAGES), pempty0 = smem_u32(bars + 2 * STAGES + NBUF);
  // Gate/Up: per quadrant q, xbar0 + 8q (row maxima written) and xbar0 + 8 (4 + q) (read)
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
  const int ipt = items_per_tile(MODE, p.nN);
  const int items = ntiles * ipt;
  const int nk = (p.K + BKB - 1) / BKB;
  const int4* tiles = reinterpret_cast<const int4*>(p.tiles);

  if (warp == 0) {
    // ---------------------------------------------------------------- producer
    uint32_t stage = 0, phase = 0;
    int issued = 0;
    bool ok = true;
    for (int it = blockIdx.x; it < items && ok; it += gridDim.x) {
      const int tile = it / ipt, g = it - tile * ipt;
      const int4 tl = tiles[tile];
      const int row0 = tl.y;
      const bool shx = tl.x >= p.E;  // a shared expert's tile: its own weight tensor
      const int e = shx ? tl.x - p.E : tl.x;
      const CUtensorMap* tb = shx ? &tmB2 : &tmB;
      const int nsub = subunits(MODE, p.nN, g);
      for (int sub = 0; sub < nsub && ok; ++sub) {
        const int n = MODE == MODE_GATEUP ? 2 * g + sub : g;
        for (int kb = 0; kb < nk; ++kb) {
          if (lane == 0) {
            if (!mbar_wait(empty0 + 8 * stage, phase ^ 1, abort_flag, p.hdr, 0x80000u | MODE)) ok = false;
          }
          ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
          if (!ok) break;
          if (lane == 0) {
            const uint32_t full = full0 + 8 * stage;
            const uint32_t a_dst = smem_u32(smem + stage * STAGE_BYTES), b_dst = a_dst + A_BYTES;
            const int kc = kb * BKB;
            mbar_arrive_expect_tx(full, STAGE_BYTES);
            tma_load_2d(a_dst, &tmA, kc, row0, full);
            if (MODE == MODE_GATEUP) {
              const int brow = e * 2 * p.I + n * (BN / 2);
              tma_load_2d(b_dst, tb, kc, brow, full);                   // 64 gate rows
              tma_load_2d(b_dst + B_BYTES / 2, tb, kc, brow + p.I, full);  // the matching 64 up rows
            } else {
              tma_load_2d(b_dst, tb, kc, e * p.H + n * BN, full);
            }
          }
          __syncwarp();
          ++issued;
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1;
          }
        }
      }
    }
    if (!ok && lane == 0) {
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
        const int nsub = subunits(MODE, p.nN, it % ipt);
        for (int kt = 0; kt < nsub * nk; ++kt) {
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
  } else if (warp >= 4) {
    // ---------------------------------------------------------------- epilogue (promotion)
    const int e8 = warp - 4;
    const int q = e8 & 3;   // TMEM lane quadrant (warp % 4)
    const int ch = e8 >> 2; // which 64 of the 128 columns
    const int row = q * 32 + lane;
    // Gate/Up: gate columns [32ch, 32ch+32) and the matching up columns 64 + [32ch, ...);
    // Down: columns [64ch, 64ch+64)
    const int c0 = MODE == MODE_GATEUP ? ch * 32 : ch * 64;
    const int c1 = MODE == MODE_GATEUP ? BN / 2 + ch * 32 : ch * 64 + 32;
    uint32_t pb = 0, pphase = 0;
    const int kblocks = nk;  // scale groups along K: ceil(K / 128)
    float* rowmax = reinterpret_cast<float*>(smem + staging_offset(MODE) + STAGING_BYTES);  // Gate/Up: [8 warps][32]
    uint32_t xphase = 0;  // phase of this quadrant's exchange barriers
    bool ok = true;
    for (int it = blockIdx.x; it < items && ok; it += gridDim.x) {
      const int tile = it / ipt, g = it - tile * ipt;
      const int4 tl = tiles[tile];
      const int row0 = tl.y, nrows = tl.z;
      const bool shx = tl.x >= p.E;
      const int e = shx ? tl.x - p.E : tl.x;
      const float* wsc = shx ? p.w_scale2 : p.w_scale;
      const int arow = row0 + min(row, nrows - 1);
      const float* sa = p.a_scale + static_cast<size_t>(arow) * kblocks;
      const int nsub = subunits(MODE, p.nN, g);
      float mrow = 0.0f;  // Gate/Up: this thread's row maximum of |a| over the group so far
      for (int sub = 0; sub < nsub && ok; ++sub) {
        const int n = MODE == MODE_GATEUP ? 2 * g + sub : g;
        // weight scale rows of this unit's columns (both halves in one block for Down)
        const float* swg;
        const float* swu;
        if (MODE == MODE_GATEUP) {
          const int nblk = 2 * p.I / 128, hblk = p.H / 128;
          swg = wsc + (static_cast<size_t>(e) * nblk + (n * (BN / 2)) / 128) * hblk;
          swu = wsc + (static_cast<size_t>(e) * nblk + (p.I + n * (BN / 2)) / 128) * hblk;
        } else {
          const int hblk = p.H / 128;
          swg = wsc + (static_cast<size_t>(e) * hblk + n) * kblocks;
          swu = swg;
        }
        float acc[64];
#pragma unroll
        for (int i = 0; i < 64; ++i) acc[i] = 0.0f;
        float sa_next = __ldg(sa), sg_next = __ldg(swg), su_next = __ldg(swu);
        for (int kb = 0; kb < nk; ++kb) {
          const float sak = sa_next, sgk = sg_next, suk = su_next;
          if (kb + 1 < nk) {
            sa_next = __ldg(sa + kb + 1);
            sg_next = __ldg(swg + kb + 1);
            su_next = __ldg(swu + kb + 1);
          }
          int good = 1;
          if (lane == 0) good = mbar_wait(pfull0 + 8 * pb, pphase, abort_flag, p.hdr, 0x83000u | MODE);
          if (!__shfl_sync(0xffffffffu, good, 0)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t tbase = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + pb * BN;
          float v0[32], v1[32];
          tmem_ld32(tbase + c0, v0);
          tmem_ld32(tbase + c1, v1);
          tmem_ld_wait();
          // both column ranges are in registers: hand the buffer back before the FMAs
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(pempty0 + 8 * pb);
          const float s0 = sak * sgk, s1 = sak * (MODE == MODE_GATEUP ? suk : sgk);
#pragma unroll
          for (int i = 0; i < 32; i += 2) {  // packed pairs: half the FMA instructions
            fma2(acc[i], acc[i + 1], v0[i], v0[i + 1], s0, s0);
            fma2(acc[32 + i], acc[33 + i], v1[i], v1[i + 1], s1, s1);
          }
          if (++pb == NBUF) {
            pb = 0;
            pphase ^= 1;
          }
        }
        if (!ok) break;
        if (MODE == MODE_GATEUP) {
          // a for 32 h columns of this row; the first unit of a pair parks its values in
          // this warp's staging slot (row-per-lane, 16-byte pieces XOR-swizzled by lane)
          float a[32];
          float m = 0.0f;
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            a[i] = silu_mul_fast(acc[i], acc[32 + i]);
            m = fmaxf(m, fabsf(a[i]));
          }
          mrow = fmaxf(mrow, m);
          float4* stg = reinterpret_cast<float4*>(smem + staging_offset(MODE) + e8 * 4096) + lane * 8;
          if (sub == 0 && nsub == 2) {
#pragma unroll
            for (int i = 0; i < 8; ++i)
              stg[i ^ (lane & 7)] = make_float4(a[4 * i], a[4 * i + 1], a[4 * i + 2], a[4 * i + 3]);
          }
          if (sub == nsub - 1) {
            // the group's scale: row maximum over both warps of the quadrant (64 columns
            // each), exchanged through shared memory between the two warps; bounded
            // mbarrier waits order the write, the partner's read and the next write
            rowmax[e8 * 32 + lane] = row < nrows ? mrow : 0.0f;
            __syncwarp();
            if (lane == 0) mbar_arrive(xbar0 + 8 * q);
            int good = 1;
            if (lane == 0) good = mbar_wait(xbar0 + 8 * q, xphase, abort_flag, p.hdr, 0x84000u);
            if (!__shfl_sync(0xffffffffu, good, 0)) {
              ok = false;
              break;
            }
            const float gm = fmaxf(rowmax[e8 * 32 + lane], rowmax[(e8 ^ 4) * 32 + lane]);
            __syncwarp();
            if (lane == 0) mbar_arrive(xbar0 + 8 * (4 + q));
            if (lane == 0) good = mbar_wait(xbar0 + 8 * (4 + q), xphase, abort_flag, p.hdr, 0x85000u);
            if (!__shfl_sync(0xffffffffu, good, 0)) {
              ok = false;
              break;
            }
            xphase ^= 1;
            if (row < nrows) {
              const float sc = e4m3_scale(gm);
              const float inv = 1.0f / sc;
              const size_t r = static_cast<size_t>(row0 + row);
              uint8_t* hrow = p.h + r * p.I;
              if (nsub == 2) {
                // the first unit's values, 4 at a time from the staging slot
                uint32_t w[8];
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                  const float4 v = stg[i ^ (lane & 7)];
                  w[i] = static_cast<uint32_t>(cvt_e4m3x2(v.x * inv, v.y * inv)) |
                         (static_cast<uint32_t>(cvt_e4m3x2(v.z * inv, v.w * inv)) << 16);
                }
                uint4* d0 = reinterpret_cast<uint4*>(hrow + (2 * g) * 64 + ch * 32);
                d0[0] = make_uint4(w[0], w[1], w[2], w[3]);
                d0[1] = make_uint4(w[4], w[5], w[6], w[7]);
                store_e4m3x32(hrow + (2 * g + 1) * 64 + ch * 32, a, inv);
              } else {
                store_e4m3x32(hrow + (2 * g) * 64 + ch * 32, a, inv);
              }
              if (ch == 0) p.h_scale[r * ((p.I + 127) / 128) + g] = sc;
            }
          }
        } else {
          // Down rows (sorted order, like h): each thread's 64 bf16 outputs are staged
          // in shared memory (16-byte pieces XOR-swizzled by row) and the warp writes
          // four whole 128-byte row segments per store instruction.
          uint4* stg = reinterpret_cast<uint4*>(smem + staging_offset(MODE)) + e8 * (32 * 8);
#pragma unroll
          for (int i = 0; i < 8; ++i) stg[lane * 8 + (i ^ (lane & 7))] = pack_bf16x8(acc + 8 * i);
          __syncwarp();
          const int wrows = min(32, nrows - q * 32);  // valid rows of this warp (may be <= 0)
          const int slot = row0 + row;
#pragma unroll
          for (int it2 = 0; it2 < 8; ++it2) {
            const int r = it2 * 4 + (lane >> 3), j = lane & 7;
            const int rslot = __shfl_sync(0xffffffffu, slot, r);
            if (r < wrows)
              *reinterpret_cast<uint4*>(p.out + static_cast<size_t>(rslot) * p.H + n * BN + ch * 64 + j * 8) =
                  stg[r * 8 + (j ^ (r & 7))];
          }
          __syncwarp();
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 2) {
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

template <int MODE>
static cudaError_t smem_attr() {
  static const cudaError_t st = cudaFuncSetAttribute(grouped_blockwise_kernel<MODE>,
                                                     cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem_bytes(MODE));
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
  if (!encode_u8(&tma, a.xs, a.H, a.R, BM) || !encode_u8(&tmb, a.w1, a.H, static_cast<uint64_t>(a.E) * 2 * a.I, BN / 2))
    return cudaErrorInvalidValue;
  tmbs = tmb;
  if (a.S > 0 && !encode_u8(&tmbs, a.w1s, a.H, static_cast<uint64_t>(a.S) * 2 * a.I, BN / 2))
    return cudaErrorInvalidValue;
  Params p{};
  p.tiles = a.tiles;
  p.num_tiles = a.num_tiles;
  p.max_tiles = a.max_tiles;
  p.perm = a.perm;
  p.nN = a.I / (BN / 2);
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
  const long long items = static_cast<long long>(a.max_tiles) * ((p.nN + 1) / 2);
  const int grid = static_cast<int>(items < sms ? items : sms);
  stage_begin("gateup_gemm", s);
  err = launch_dependent(grouped_blockwise_kernel<MODE_GATEUP>, dim3(grid), dim3(THREADS), smem_bytes(MODE_GATEUP), s,
                         tma, tmb, tma, tmbs, p);
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
  CUtensorMap tma, tmb, tmbs;
  if (!encode_u8(&tma, a.h, a.I, a.R, BM) || !encode_u8(&tmb, a.w2, a.I, static_cast<uint64_t>(a.E) * a.H, BN))
    return cudaErrorInvalidValue;
  tmbs = tmb;
  if (a.S > 0 && !encode_u8(&tmbs, a.w2s, a.I, static_cast<uint64_t>(a.S) * a.H, BN)) return cudaErrorInvalidValue;
  Params p{};
  p.tiles = a.tiles;
  p.num_tiles = a.num_tiles;
  p.max_tiles = a.max_tiles;
  p.perm = a.perm;
  p.nN = a.H / BN;
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
  err = launch_dependent(grouped_blockwise_kernel<MODE_DOWN>, dim3(grid), dim3(THREADS), smem_bytes(MODE_DOWN), s,
                         tma, tmb, tma, tmbs, p);
  stage_end(s);
  return err;
}

}  // namespace moe
