// MXFP8 path of the grouped forward, and the per-group blocked scale layout of
// "[mxfp8 moe training] add per group blocked scale kernels" (Summary: convert
// the MX scales of expert-grouped activations into the blocked, swizzled layout
// per group, with each group's start row in the block-padded output computed on
// the device, without a device-to-host sync).
//
// MXFP8 (OCP Microscaling, E4M3 elements): each run of 32 values along the
// contraction dimension shares one E8M0 scale 2^X, X = floor(log2(amax)) - 8
// (clamped to [-127, 127]; -127 for a zero run); elements e4m3(v / 2^X) rounded
// to nearest even and saturated.  The tensor cores apply the scales themselves
// (tcgen05.mma kind::mxf8f6f4.block_scale), reading them from TMEM, where
// tcgen05.cp puts them from shared memory in exactly the blocked layout: a
// 128-row x 4-chunk block of scales is 512 bytes, line i holding rows i, i+32,
// i+64, i+96, four K chunks each; copied with .32x128b.warpx4, row r's scale
// word lands in TMEM lane r % 32 (of every quadrant), column r / 32.
//
// Kernels:
//   scatter_gather_mx   one block per token: quantises the token's x row to
//                       MXFP8 once and copies codes and scales to its sorted rows
//                       (and its shared-expert rows).
//   mx_blocked          row-major scales -> blocked layout, one 128-row block per
//                       CTA: the blocks of the grouped GEMM's tile map (a group
//                       per expert, padded to whole tiles), the weights' rows, or
//                       caller-given groups (moe_mx_blocked_scales).
//   grouped_mx<0>       Gate/Up: 128 sorted rows x (96 gate + the matching 96 up
//                       rows of W1[e]) per unit; 4 block-scaled MMAs (N = 192) of
//                       K=32 per 128-wide K stage; three epilogue warps per TMEM
//                       quadrant compute a = silu(g) * u and quantise it per run
//                       of 32 straight into e4m3 h and its E8M0 scales (no fp32
//                       round trip).
//   grouped_mx<1>       Down: 128 rows x 128 rows of W2[e]; bf16 o in sorted row
//                       order (staged, TMA tile stores).
#include "common.cuh"
#include "internal.h"

namespace moe {
namespace mx {

constexpr int BM = kGemmBM;      // 128 rows per tile
constexpr int BKB = 128;         // K bytes (= e4m3 values) per stage: 4 scale chunks
constexpr int A_BYTES = BM * BKB;
constexpr int SF_BYTES = 512;    // one blocked scale block (128 rows x 4 chunks)
constexpr int TMEM_COLS = 512;   // 2 accumulators, then the scale slots
// Gate/Up units: 96 gate + the matching 96 up rows of W1[e]; Down units: 192 rows of
// W2[e] (N = 192 for both: two 192-column accumulators and the stages' scale slots
// fit the 512 TMEM columns).
__host__ __device__ constexpr int bn_of(int mode) { return 192; }
__host__ __device__ constexpr int gu_half() { return 96; }
__host__ __device__ constexpr int sfb_blocks(int mode) { return 2; }  // 128-row B scale blocks per unit
__host__ __device__ constexpr int stage_bytes(int mode) {
  return (A_BYTES + bn_of(mode) * BKB + (1 + sfb_blocks(mode)) * SF_BYTES + 1023) / 1024 * 1024;
}
__host__ __device__ constexpr int sf_col0(int mode) { return 2 * bn_of(mode); }
__host__ __device__ constexpr int sf_cols_per_stage(int mode) { return 4 * (1 + sfb_blocks(mode)); }
__host__ __device__ constexpr int stages_of(int mode) { return mode == 0 ? 5 : 4; }
// Gate/Up: three warps per TMEM quadrant, one 32-column run of h each; Down: one.
__host__ __device__ constexpr int epi_warps_of(int mode) { return mode == 0 ? 12 : 4; }
__host__ __device__ constexpr int threads_of(int mode) { return 32 * (4 + epi_warps_of(mode)); }
constexpr int NUM_BARS = 2 * 5 + 4 + 1;
__host__ __device__ constexpr int staging_offset(int mode) {
  return (stages_of(mode) * stage_bytes(mode) + 256 + 1023) / 1024 * 1024;
}
constexpr int STAGING_BYTES = 4 * 32 * 256;  // Down: 32 rows x 256 bytes per epilogue warp
__host__ __device__ constexpr size_t smem_bytes(int mode) {
  return 1024 + staging_offset(mode) + (mode == 1 ? STAGING_BYTES : 0);
}
static_assert(sf_col0(0) + stages_of(0) * sf_cols_per_stage(0) <= TMEM_COLS, "Gate/Up TMEM columns");
static_assert(sf_col0(1) + stages_of(1) * sf_cols_per_stage(1) <= TMEM_COLS, "Down TMEM columns");
static_assert(smem_bytes(0) <= 232448 && smem_bytes(1) <= 232448, "shared memory per block");

// ------------------------------------------------------------------ MX quantisation helpers
// X = floor(log2(amax)) - 8 in [-127, 127]; -127 when amax == 0.
__device__ __forceinline__ int mx_exponent(float amax) {
  if (!(amax > 0.0f)) return -127;
  const uint32_t b = __float_as_uint(amax);
  const int ef = static_cast<int>((b >> 23) & 0xFFu);
  // subnormal amax = m * 2^-149 with m < 2^23: floor(log2) = (bit index of m's top bit) - 149
  const int fl = ef != 0 ? ef - 127 : (31 - __clz(static_cast<int>(b & 0x7FFFFFu))) - 149;
  const int x = fl - 8;
  return x < -127 ? -127 : (x > 127 ? 127 : x);
}

// 2^x as fp32 for x in [-127, 127] (2^-127 is the subnormal 0x00400000).
__device__ __forceinline__ float pow2_exact(int x) {
  return x >= -126 ? __uint_as_float(static_cast<uint32_t>(x + 127) << 23) : __uint_as_float(0x00400000u);
}

// 8 values -> 8 e4m3 codes of v / 2^X (RNE, saturating).  inv = 2^-X is exact for X
// in [-127, 127], so v * inv is the correctly rounded quotient v / 2^X, the same
// value an IEEE division gives, at the cost of a multiplication.
__device__ __forceinline__ uint2 quant8(const float* f, float inv) {
  const uint32_t q0 = static_cast<uint32_t>(cvt_e4m3x2(f[0] * inv, f[1] * inv)) |
                      (static_cast<uint32_t>(cvt_e4m3x2(f[2] * inv, f[3] * inv)) << 16);
  const uint32_t q1 = static_cast<uint32_t>(cvt_e4m3x2(f[4] * inv, f[5] * inv)) |
                      (static_cast<uint32_t>(cvt_e4m3x2(f[6] * inv, f[7] * inv)) << 16);
  return make_uint2(q0, q1);
}

// ------------------------------------------------------------------ scatter + MX quantisation of x
// One block per token: the block quantises the token's x row once into shared
// memory (4 consecutive threads hold one run of 32, 8 values each, and reduce its
// amax), then one warp per route places perm / inv and copies the codes and the
// row's E8M0 scale codes to sorted row p of xs / xs_sc; rows T*k + s*T + t take
// the shared experts' copies.
__global__ void __launch_bounds__(256) scatter_gather_mx_kernel(
    const int32_t* __restrict__ ids, const int32_t* __restrict__ lrank, const int32_t* __restrict__ blockbase, int E,
    int RB, int k, int H, const uint4* __restrict__ x, uint8_t* __restrict__ xs, uint8_t* __restrict__ xs_sc,
    uint8_t* __restrict__ xs_sf, const int32_t* __restrict__ padbase, int32_t* __restrict__ perm,
    int32_t* __restrict__ inv, int S, int T) {
  extern __shared__ __align__(16) uint8_t s_row[];  // [H] e4m3 codes, then [H/32] scale codes
  dep_wait();  // ranks and block bases
  uint8_t* s_sc = s_row + H;
  const int t = blockIdx.x;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int n8 = H / 8;
  const uint4* src = x + static_cast<size_t>(t) * n8;
  for (int base = 0; base < n8; base += blockDim.x) {
    const int c = base + tid;
    const bool act = c < n8;  // whole 4-thread runs are active together (H % 32 == 0)
    const uint4 v = act ? __ldg(src + c) : make_uint4(0, 0, 0, 0);
    float f[8];
    const __nv_bfloat162* b = reinterpret_cast<const __nv_bfloat162*>(&v);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float2 u = __bfloat1622float2(b[j]);
      f[2 * j] = u.x;
      f[2 * j + 1] = u.y;
    }
    float m = 0.0f;
#pragma unroll
    for (int j = 0; j < 8; ++j) m = fmaxf(m, fabsf(f[j]));
    m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 1));
    m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 2));
    const int X = mx_exponent(m);
    if (act) {
      *reinterpret_cast<uint2*>(s_row + 8 * c) = quant8(f, pow2_exact(-X));
      if ((c & 3) == 0) s_sc[c / 4] = static_cast<uint8_t>(X + 127);
    }
  }
  __syncthreads();
  const int row16 = H / 16, nsc = H / 32, ncb = nsc / 4;  // H % 128 == 0: whole 4-chunk blocks
  for (int j = warp; j < k + S; j += blockDim.x >> 5) {
    int p, e;
    if (j < k) {
      const int r = t * k + j;
      const int lr = lrank[r];
      if (lr < 0) {
        if (lane == 0) inv[r] = -1;
        continue;
      }
      e = ids[r];
      p = blockbase[static_cast<size_t>(r / RB) * E + e] + lr;
      if (lane == 0) {
        perm[p] = r;
        inv[r] = p;
      }
    } else {
      e = E + (j - k);
      p = T * k + (j - k) * T + t;
    }
    uint4* dst = reinterpret_cast<uint4*>(xs + static_cast<size_t>(p) * H);
    for (int c = lane; c < row16; c += 32) dst[c] = reinterpret_cast<const uint4*>(s_row)[c];
    for (int c = lane; c < nsc; c += 32) xs_sc[static_cast<size_t>(p) * nsc + c] = s_sc[c];
    // the same scales in the blocked layout: padded row pr, four chunks per 4-byte word
    const int pr = p + __ldg(padbase + e);
    uint8_t* blk = xs_sf + static_cast<size_t>(pr / BM) * ncb * SF_BYTES + (pr % 32) * 16 + ((pr % BM) / 32) * 4;
    for (int cb = lane; cb < ncb; cb += 32)
      *reinterpret_cast<uint32_t*>(blk + cb * SF_BYTES) = reinterpret_cast<const uint32_t*>(s_sc)[cb];
  }
}

// ------------------------------------------------------------------ blocked scale layout
// Where the 128 rows of output block b come from.
//   TILES    block b = tile b of the tile map: rows row0 .. row0 + nrows - 1, the
//            rest padding (a group per expert, each padded to whole 128-row blocks).
//   W1ROWS   block b = (expert e, 64-row chunk n) of W1 [E, 2I, .]: gate rows
//            [64n, 64n + 64) then the matching up rows [I + 64n, I + 64n + 64) of
//            W1[e], the rows of one Gate/Up unit's B operand.
//   CONTIG   block b = rows [128b, 128b + 128) (all valid).
//   W1ROWS96 the B operand of one MXFP8 Gate/Up unit (expert e, unit n): gate rows
//            [96n, 96n + 96) then the matching up rows of W1[e], 192 rows in two
//            blocks (the second half-padded); a row past I is padding.  Output
//            block 2 u + h of unit u = e * units + n is stored at ((u * ncb + cb)
//            * 2 + h) * 512: the two blocks of one column block are adjacent.
//   W2ROWS192 the B operand of one MXFP8 Down unit (expert e, unit n): rows
//            [192n, 192n + 192) of W2[e] ([H rows]), in two blocks stored like
//            W1ROWS96; a row past H is padding.
constexpr int SRC_TILES = 0, SRC_W1ROWS = 1, SRC_CONTIG = 2, SRC_W1ROWS96 = 3, SRC_W2ROWS192 = 4;

// One CTA per output block: thread i of 32 * ncb writes the 16-byte line (i % 32)
// of column block i / 32: scales of rows line, line+32, line+64, line+96 of the
// block, chunks 4cb .. 4cb+3 each (zeros beyond the row or column range).
template <int SRC>
__global__ void __launch_bounds__(256) mx_blocked_kernel(const uint8_t* __restrict__ sc, int C,
                                                         const int4* __restrict__ tiles,
                                                         const int32_t* __restrict__ num_tiles, int I,
                                                         uint8_t* __restrict__ out, int wait_at_end) {
  if (!wait_at_end) dep_wait();  // the scales (and tiles) come from the kernels before
  const int b = blockIdx.x;
  int row0 = 0, nrows = BM, I2 = 0, e = 0, n = 0, half = 0;
  if (SRC == SRC_W2ROWS192) {  // I holds H here
    const int per = (I + 191) / 192;
    half = b & 1;
    e = (b >> 1) / per;
    n = (b >> 1) - e * per;
  } else if (SRC == SRC_W1ROWS96) {
    const int per = (I + gu_half() - 1) / gu_half();
    half = b & 1;
    e = (b >> 1) / per;
    n = (b >> 1) - e * per;
    I2 = 2 * I;
  } else if (SRC == SRC_TILES) {
    if (b >= *num_tiles) return;
    const int4 tl = tiles[b];
    row0 = tl.y;
    nrows = tl.z;
  } else if (SRC == SRC_W1ROWS) {
    const int per = I / 64;
    e = b / per;
    n = b - e * per;
    I2 = 2 * I;
  } else {
    row0 = b * BM;
  }
  const int ncb = (C + 3) / 4;
  uint8_t* blk = out + static_cast<size_t>(b) * ncb * SF_BYTES;
  for (int i = threadIdx.x; i < ncb * 32; i += blockDim.x) {
    const int cb = i >> 5, line = i & 31;
    uint32_t w[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int r = 32 * j + line;  // row of the block
      long long src_row = -1;
      if (SRC == SRC_W2ROWS192) {
        const int br = half * BM + r;
        if (br < 192 && n * 192 + br < I) src_row = static_cast<long long>(e) * I + n * 192 + br;
      } else if (SRC == SRC_W1ROWS96) {
        const int br = half * BM + r;                     // row of the unit's 192-row B operand
        const int col = n * gu_half() + (br < gu_half() ? br : br - gu_half());  // column of h
        if (br < 2 * gu_half() && col < I)
          src_row = static_cast<long long>(e) * I2 + (br < gu_half() ? col : I + col);
      } else if (SRC == SRC_W1ROWS)
        src_row = static_cast<long long>(e) * I2 + (r < 64 ? 64 * n + r : I + 64 * n + (r - 64));
      else if (r < nrows)
        src_row = row0 + r;
      uint32_t word = 0;
      if (src_row >= 0) {
        if ((C & 3) == 0) {  // four whole scale bytes: one aligned 32-bit load
          word = __ldg(reinterpret_cast<const uint32_t*>(sc + src_row * C + 4 * cb));
        } else {
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            const int col = 4 * cb + c;
            if (col < C) word |= static_cast<uint32_t>(__ldg(sc + src_row * C + col)) << (8 * c);
          }
        }
      }
      w[j] = word;
    }
    uint8_t* dst = (SRC == SRC_W1ROWS96 || SRC == SRC_W2ROWS192)
                       ? out + ((static_cast<size_t>(b >> 1) * ncb + cb) * 2 + (b & 1)) * SF_BYTES
                       : blk + cb * SF_BYTES;
    *reinterpret_cast<uint4*>(dst + line * 16) = make_uint4(w[0], w[1], w[2], w[3]);
  }
  if (wait_at_end) dep_wait();  // complete only after the kernel before (keeps the launch chain ordered)
}

// Groups given by row offsets (moe_mx_blocked_scales): tile map of the groups
// (ceil(n_g / 128) blocks each, 128-row blocks, groups in order) and each
// group's start row in the padded output; one block of 1024 threads.
__global__ void __launch_bounds__(1024) mx_group_tiles_kernel(const int32_t* __restrict__ goff, int G, int rows,
                                                              int4* __restrict__ tiles, int32_t* __restrict__ num_tiles,
                                                              int max_tiles, int32_t* __restrict__ starts,
                                                              DeviceHeader* hdr) {
  __shared__ int s_cnt[1024];
  __shared__ int s_pre[1025];
  const int tid = threadIdx.x;
  int carry = 0;  // blocks before this chunk of groups
  for (int g0 = 0; g0 < G; g0 += 1024) {
    const int g = g0 + tid;
    int n = 0;
    if (g < G) {
      const int lo = goff[g], hi = goff[g + 1];
      n = hi - lo;
      if (n < 0 || lo < 0 || hi > rows) {  // a group outside the scale matrix: left out, reported
        record_status(hdr, kStatusBounds, 0x7300000u | static_cast<unsigned>(g));
        n = 0;
      }
    }
    const int nb = (n + BM - 1) / BM;
    s_cnt[tid] = nb;
    __syncthreads();
    if (tid == 0) {  // serial prefix over <= 1024 counts: negligible next to the copy
      int run = carry;
      for (int i = 0; i < 1024; ++i) {
        s_pre[i] = run;
        run += s_cnt[i];
      }
      s_pre[1024] = run;
    }
    __syncthreads();
    if (g < G) {
      starts[g] = s_pre[tid] * BM;
      for (int j = 0; j < nb; ++j) {
        const int idx = s_pre[tid] + j;
        if (idx < max_tiles) tiles[idx] = make_int4(g, goff[g] + j * BM, min(BM, n - j * BM), 0);
      }
    }
    carry = s_pre[1024];
    __syncthreads();
  }
  if (tid == 0) {
    starts[G] = carry * BM;
    *num_tiles = carry;
    if (carry > max_tiles) record_status(hdr, kStatusBounds, 0x7400000u);
  }
}

// ------------------------------------------------------------------ grouped GEMMs
struct Params {
  const int32_t* tiles;
  const int32_t* num_tiles;
  int max_tiles;
  int nN;          // units per row tile
  int K;           // reduction length (bytes = e4m3 values)
  int I, H, E;
  const uint8_t* a_sf;   // blocked A scales: block row = tile index, ncbA column blocks
  const uint8_t* w_sf;   // blocked weight scales of the routed experts
  const uint8_t* w_sf2;  // ... of the shared experts (tiles of expert E + s)
  int ncbA, ncbW;
  uint8_t* h;            // Gate/Up: e4m3 h [R, I]
  uint8_t* h_sc;         // Gate/Up: E8M0 scale codes of h, blocked (block row = tile, ncbH column blocks)
  int ncbH;
  __nv_bfloat16* o;      // Down: o [R, H]
  DeviceHeader* hdr;
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

template <int MODE>
__global__ void __launch_bounds__(threads_of(MODE), 1)
    grouped_mx_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                      const __grid_constant__ CUtensorMap tmO, const __grid_constant__ CUtensorMap tmB2,
                      const Params p) {
  constexpr int STAGES = stages_of(MODE);
  constexpr int EPI = epi_warps_of(MODE);
  constexpr int BN = bn_of(MODE);
  constexpr int STAGE_BYTES = stage_bytes(MODE);
  constexpr int B_BYTES = BN * BKB;
  constexpr int NSFB = sfb_blocks(MODE);
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
      mbar_init(tempty0 + 8 * a, EPI);  // one arrival per epilogue warp
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
  dep_wait();  // tile map, activations and blocked scales come from the kernels before

  const int ntiles = min(*p.num_tiles, p.max_tiles);
  const int total = ntiles * p.nN;
  const int nk = (p.K + BKB - 1) / BKB;
  const int4* tiles = reinterpret_cast<const int4*>(p.tiles);

  if (warp == 0) {
    // ---------------------------------------------------------------- producer
    if (lane == 0) {
      uint32_t stage = 0, phase = 0;
      int issued = 0;
      bool ok = true;
      for (int u = blockIdx.x; u < total && ok; u += gridDim.x) {
        const int tile = u / p.nN, n = u - (u / p.nN) * p.nN;
        const int4 tl = tiles[tile];
        const bool shx = tl.x >= p.E;
        const int e = shx ? tl.x - p.E : tl.x;
        const CUtensorMap* tb = shx ? &tmB2 : &tmB;
        const uint8_t* wsf = shx ? p.w_sf2 : p.w_sf;
        // B rows of this unit and the blocked scale blocks that cover them
        const int brow = MODE == 0 ? e * 2 * p.I + n * gu_half() : e * p.H + n * BN;
        const long long bblk = static_cast<long long>(e) * p.nN + n;
        for (int kb = 0; kb < nk; ++kb) {
          if (!mbar_wait(empty0 + 8 * stage, phase ^ 1, abort_flag, p.hdr, 0xA0000u | MODE)) {
            ok = false;
            break;
          }
          const uint32_t full = full0 + 8 * stage;
          const uint32_t a_dst = smem_u32(smem + stage * STAGE_BYTES);
          const uint32_t b_dst = a_dst + A_BYTES;
          const uint32_t sf_dst = b_dst + B_BYTES;
          mbar_arrive_expect_tx(full, A_BYTES + B_BYTES + (1 + NSFB) * SF_BYTES);
          const int kc = kb * BKB;
          tma_load_2d(a_dst, &tmA, kc, tl.y, full);
          if (MODE == 0) {
            tma_load_2d(b_dst, tb, kc, brow, full);                         // 96 gate rows
            tma_load_2d(b_dst + B_BYTES / 2, tb, kc, brow + p.I, full);  // the matching 96 up rows
          } else {
            tma_load_2d(b_dst, tb, kc, brow, full);
          }
          bulk_load(sf_dst, p.a_sf + (static_cast<size_t>(tile) * p.ncbA + kb) * SF_BYTES, SF_BYTES, full);
          bulk_load(sf_dst + SF_BYTES, wsf + (static_cast<size_t>(bblk) * p.ncbW + kb) * (NSFB * SF_BYTES),
                    NSFB * SF_BYTES, full);
          ++issued;
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1;
          }
        }
      }
      if (!ok) {
        for (int i = 0; i < min(issued, STAGES); ++i) {
          stage = (stage + STAGES - 1) % STAGES;
          if (stage == STAGES - 1) phase ^= 1;
          mbar_wait_quiet(full0 + 8 * stage, phase, 50000000ull);
        }
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ---------------------------------------------------------------- MMA issuer
    if (lane == 0) {
      uint32_t stage = 0, phase = 0, acc = 0, acc_phase = 0;
      bool ok = true;
      for (int u = blockIdx.x; u < total && ok; u += gridDim.x) {
        if (!mbar_wait(tempty0 + 8 * acc, acc_phase ^ 1, abort_flag, p.hdr, 0xA1000u | MODE)) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + acc * BN;
        for (int kb = 0; kb < nk; ++kb) {
          if (!mbar_wait(full0 + 8 * stage, phase, abort_flag, p.hdr, 0xA2000u | MODE)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a_addr = smem_u32(smem + stage * STAGE_BYTES);
          const uint32_t b_addr = a_addr + A_BYTES;
          const uint32_t sf_addr = b_addr + B_BYTES;
          const uint32_t sfa_t = tmem_base + sf_col0(MODE) + stage * sf_cols_per_stage(MODE);
          const uint32_t sfb_t = sfa_t + 4;
          tmem_cp_32x128b_x4(sfa_t, sf_desc(sf_addr));
#pragma unroll
          for (int b = 0; b < NSFB; ++b)  // B rows 128b .. 128b + 127 -> columns 4b .. 4b + 3
            tmem_cp_32x128b_x4(sfb_t + 4 * b, sf_desc(sf_addr + (1 + b) * SF_BYTES));
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)  // K chunk kk of the stage: byte kk of every scale word
            mma_mx(d_tmem, sw128_kmajor_desc(a_addr + kk * 32), sw128_kmajor_desc(b_addr + kk * 32),
                   make_idesc_mx(BM, BN, kk, kk), sfa_t, sfb_t, (kb | kk) != 0);
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
      mma_commit(mma_done);
      mbar_wait_quiet(mma_done, 0, 1000000000ull);
    }
    __syncwarp();
  } else if (warp >= 4) {
    // ---------------------------------------------------------------- epilogue
    const int e8 = warp - 4;
    const int q = e8 & 3;
    const int row = q * 32 + lane;
    uint32_t acc = 0, acc_phase = 0;
    for (int u = blockIdx.x; u < total; u += gridDim.x) {
      const int tile = u / p.nN, n = u - (u / p.nN) * p.nN;
      const int4 tl = tiles[tile];
      const int row0 = tl.y, nrows = tl.z;
      int good = 1;
      if (lane == 0) good = mbar_wait(tfull0 + 8 * acc, acc_phase, abort_flag, p.hdr, 0xA3000u | MODE);
      good = __shfl_sync(0xffffffffu, good, 0);
      if (!good) break;
      tc_fence_after();
      const uint32_t tbase = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + acc * BN;
      if (MODE == 0) {
        // warp run ch of its quadrant: gate columns [32ch, 32ch + 32) and the matching
        // up columns; its 32 h values of a row are exactly one MX run
        const int ch = e8 >> 2;
        float g[32], up[32];
        tmem_ld32(tbase + ch * 32, g);
        tmem_ld32(tbase + gu_half() + ch * 32, up);
        tmem_ld_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(tempty0 + 8 * acc);
        const int col = n * gu_half() + ch * 32;  // first h column of this run
        if (row < nrows && col < p.I) {
          float a[32];
          float m = 0.0f;
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            a[i] = silu_mul(g[i], up[i]);
            m = fmaxf(m, fabsf(a[i]));
          }
          const int X = mx_exponent(m);
          const float inv = pow2_exact(-X);
          uint4 q4[2];
          uint2* q2 = reinterpret_cast<uint2*>(q4);
#pragma unroll
          for (int i = 0; i < 4; ++i) q2[i] = quant8(a + 8 * i, inv);
          const size_t r = static_cast<size_t>(row0 + row);
          uint4* dst = reinterpret_cast<uint4*>(p.h + r * p.I + col);
          dst[0] = q4[0];
          dst[1] = q4[1];
          // the scale straight into the blocked layout of the Down GEMM's A scales
          // (block row = tile, chunk col / 32)
          const int c32 = col / 32;
          p.h_sc[(static_cast<size_t>(tile) * p.ncbH + c32 / 4) * SF_BYTES + (row % 32) * 16 + (row / 32) * 4 + c32 % 4] =
              static_cast<uint8_t>(X + 127);
        }
        // the last unit's last warp zeroes the scale chunks past I up to whole 4-chunk
        // blocks: they meet the Down GEMM's zero-filled K tail
        if (row < nrows && n == p.nN - 1 && ch == 2)
          for (int c32 = (p.I + 31) / 32; c32 < 4 * p.ncbH; ++c32)
            p.h_sc[(static_cast<size_t>(tile) * p.ncbH + c32 / 4) * SF_BYTES + (row % 32) * 16 + (row / 32) * 4 +
                   c32 % 4] = 0;
      } else {
        // Down: the BN output columns of the unit in passes of two 64-column boxes,
        // each staged as [32 rows][128 bytes] (128-byte swizzle) per warp and written
        // by TMA tile stores when all 32 rows belong to the tile, else by 16-byte stores
        uint8_t* stg = smem + staging_offset(MODE) + q * (32 * 256);
        const int wrows = min(32, nrows - q * 32);
        const int wrow0 = row0 + q * 32;
        constexpr int NBOX = BN / 64;
#pragma unroll 1
        for (int b0 = 0; b0 < NBOX; b0 += 2) {
          const int nb = min(2, NBOX - b0);
          if (lane == 0) bulk_wait_group_read0();  // the staging's previous stores have read it
          __syncwarp();
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            if (c < 2 * nb) {
              float v[32];
              tmem_ld32(tbase + b0 * 64 + c * 32, v);
              tmem_ld_wait();
#pragma unroll
              for (int i = 0; i < 4; ++i) {
                const int cc = c * 4 + i;
                *reinterpret_cast<uint4*>(stg + (cc >> 3) * 4096 + lane * 128 + (((cc & 7) ^ (lane & 7)) << 4)) =
                    pack_bf16x8(v + 8 * i);
              }
            }
          }
          if (b0 + 2 >= NBOX) {  // every accumulator column read: hand the buffer back
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(tempty0 + 8 * acc);
          }
          const int col0 = n * BN + b0 * 64;
          if (wrows == 32) {
            fence_proxy_async_shared();
            __syncwarp();
            if (lane == 0) {
              for (int b = 0; b < nb; ++b)
                if (col0 + b * 64 < p.H) tma_store_2d(&tmO, smem_u32(stg + b * 4096), col0 + b * 64, wrow0);
              bulk_commit_group();
            }
            __syncwarp();
          } else {
            __syncwarp();
#pragma unroll 4
            for (int it = 0; it < 16; ++it) {
              const int r = it * 2 + (lane >> 4), j = lane & 15;
              const int col = col0 + j * 8;
              if (r < wrows && (j >> 3) < nb && col < p.H)
                *reinterpret_cast<uint4*>(p.o + static_cast<size_t>(wrow0 + r) * p.H + col) =
                    *reinterpret_cast<const uint4*>(stg + (j >> 3) * 4096 + r * 128 + (((j & 7) ^ (r & 7)) << 4));
            }
            __syncwarp();
          }
        }
      }
      acc ^= 1;
      if (acc == 0) acc_phase ^= 1;
    }
    if (MODE == 1 && lane == 0) bulk_wait_group0();
    __syncwarp();
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

static bool encode_bf16_out(CUtensorMap* map, const void* base, uint64_t inner, uint64_t outer) {
  EncodeTiledFn fn = get_encode_tiled();
  if (!fn) return false;
  const cuuint64_t dims[2] = {inner, outer};
  const cuuint64_t strides[1] = {inner * 2};
  const cuuint32_t box[2] = {64, 32};
  const cuuint32_t estr[2] = {1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int MODE>
static cudaError_t smem_attr() {
  static const cudaError_t st = cudaFuncSetAttribute(grouped_mx_kernel<MODE>,
                                                     cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem_bytes(MODE));
  return st;
}

template <int SRC>
static cudaError_t launch_blocked(const uint8_t* sc, int C, const int32_t* tiles, const int32_t* num_tiles, int I,
                                  uint8_t* out, unsigned nblocks, bool wait_at_end, cudaStream_t s) {
  if (nblocks == 0) return cudaSuccess;
  return launch_dependent(mx_blocked_kernel<SRC>, dim3(nblocks), dim3(256), 0, s, sc, C,
                          reinterpret_cast<const int4*>(tiles), num_tiles, I, out, wait_at_end ? 1 : 0);
}

}  // namespace mx

size_t mx_blocked_bytes(size_t blocks, int C) { return blocks * static_cast<size_t>((C + 3) / 4) * mx::SF_BYTES; }

cudaError_t launch_scatter_gather_mx(const int32_t* ids, const int32_t* lrank, const int32_t* blockbase, int T, int E,
                                     int k, int H, const void* x, void* xs, uint8_t* xs_sc, uint8_t* xs_sf,
                                     const int32_t* padbase, int32_t* perm, int32_t* inv, cudaStream_t s, int S) {
  if (T <= 0) return cudaSuccess;
  const int RB = route_tokens_per_block(k) * k;
  const size_t smem = static_cast<size_t>(H) + static_cast<size_t>(H / 32);
  if (smem > 48 * 1024) return cudaErrorInvalidValue;
  stage_begin("scatter_gather", s);
  const cudaError_t err = launch_dependent(mx::scatter_gather_mx_kernel, dim3(T), dim3(256), smem, s, ids, lrank,
                                           blockbase, E, RB, k, H, static_cast<const uint4*>(x),
                                           static_cast<uint8_t*>(xs), xs_sc, xs_sf, padbase, perm, inv, S, T);
  stage_end(s);
  return err;
}

cudaError_t launch_mx_blocked_weights(const uint8_t* w1_sc, const uint8_t* w2_sc, int E, int H, int I, uint8_t* w1_sf,
                                      uint8_t* w2_sf, cudaStream_t s) {
  stage_begin("mx_weight_scales", s);
  // these read only the caller's weight scales: their work overlaps the kernel
  // before, and they wait for it only at their end so that the chain stays ordered
  const unsigned units = static_cast<unsigned>((I + mx::gu_half() - 1) / mx::gu_half());
  cudaError_t err = mx::launch_blocked<mx::SRC_W1ROWS96>(w1_sc, H / 32, nullptr, nullptr, I, w1_sf,
                                                         static_cast<unsigned>(E) * units * 2, true, s);
  if (err == cudaSuccess)
    err = mx::launch_blocked<mx::SRC_W2ROWS192>(w2_sc, I / 32, nullptr, nullptr, H, w2_sf,
                                                static_cast<unsigned>(E) * ((H + 191) / 192) * 2, true, s);
  stage_end(s);
  return err;
}

cudaError_t launch_mx_group_blocked(const uint8_t* sc, int rows, int C, const int32_t* goff, int G, uint8_t* out,
                                    int32_t* starts, int32_t* tiles, int32_t* num_tiles, int max_tiles,
                                    DeviceHeader* hdr, cudaStream_t s) {
  stage_begin("mx_group_tiles", s);
  mx::mx_group_tiles_kernel<<<1, 1024, 0, s>>>(goff, G, rows, reinterpret_cast<int4*>(tiles), num_tiles, max_tiles,
                                               starts, hdr);
  cudaError_t err = cudaGetLastError();
  stage_end(s);
  if (err != cudaSuccess || max_tiles == 0) return err;
  stage_begin("mx_scales", s);
  err = mx::launch_blocked<mx::SRC_TILES>(sc, C, tiles, num_tiles, 0, out, static_cast<unsigned>(max_tiles), false, s);
  stage_end(s);
  return err;
}

// Gate/Up (MODE 0) and Down (MODE 1) of the MXFP8 grouped path.
static cudaError_t launch_mx_gemm(int mode, const GroupedArgs& a, const uint8_t* a_sf, const uint8_t* w_sf,
                                  const uint8_t* w_sf2, uint8_t* h_sc, cudaStream_t s) {
  using namespace mx;
  if (a.R <= 0) return cudaSuccess;
  cudaError_t err = mode == 0 ? smem_attr<0>() : smem_attr<1>();
  if (err != cudaSuccess) return err;
  const int sms = num_sms();
  if (sms <= 0) return cudaErrorNoDevice;
  CUtensorMap tma, tmb, tmb2, tmo;
  Params p{};
  p.tiles = a.tiles;
  p.num_tiles = a.num_tiles;
  p.max_tiles = a.max_tiles;
  p.I = a.I;
  p.H = a.H;
  p.E = a.E;
  p.a_sf = a_sf;
  p.w_sf = w_sf;
  p.w_sf2 = w_sf2 ? w_sf2 : w_sf;
  p.hdr = a.hdr;
  if (mode == 0) {
    if (!encode_u8(&tma, a.xs, a.H, a.R, BM) ||
        !encode_u8(&tmb, a.w1, a.H, static_cast<uint64_t>(a.E) * 2 * a.I, gu_half()))
      return cudaErrorInvalidValue;
    tmb2 = tmb;
    if (a.S > 0 && !encode_u8(&tmb2, a.w1s, a.H, static_cast<uint64_t>(a.S) * 2 * a.I, gu_half()))
      return cudaErrorInvalidValue;
    tmo = tma;
    p.nN = (a.I + gu_half() - 1) / gu_half();
    p.K = a.H;
    p.ncbA = p.ncbW = (a.H / 32 + 3) / 4;
    p.h = static_cast<uint8_t*>(a.h);
    p.h_sc = h_sc;
    p.ncbH = (a.I / 32 + 3) / 4;
  } else {
    constexpr int BN1 = bn_of(1);
    if (!encode_u8(&tma, a.h, a.I, a.R, BM) || !encode_u8(&tmb, a.w2, a.I, static_cast<uint64_t>(a.E) * a.H, BN1) ||
        !encode_bf16_out(&tmo, a.o, a.H, a.R))
      return cudaErrorInvalidValue;
    tmb2 = tmb;
    if (a.S > 0 && !encode_u8(&tmb2, a.w2s, a.I, static_cast<uint64_t>(a.S) * a.H, BN1)) return cudaErrorInvalidValue;
    p.nN = (a.H + BN1 - 1) / BN1;
    p.K = a.I;
    p.ncbA = p.ncbW = (a.I / 32 + 3) / 4;
    p.o = static_cast<__nv_bfloat16*>(a.o);
  }
  const long long units = static_cast<long long>(a.max_tiles) * p.nN;
  const int grid = static_cast<int>(units < sms ? units : sms);
  if (mode == 0) {
    stage_begin("gateup_gemm", s);
    err = launch_dependent(grouped_mx_kernel<0>, dim3(grid), dim3(threads_of(0)), smem_bytes(0), s, tma, tmb, tmo, tmb2,
                           p);
  } else {
    stage_begin("down_gemm", s);
    err = launch_dependent(grouped_mx_kernel<1>, dim3(grid), dim3(threads_of(1)), smem_bytes(1), s, tma, tmb, tmo, tmb2,
                           p);
  }
  stage_end(s);
  return err;
}

cudaError_t launch_gateup_mx(const GroupedArgs& a, const uint8_t* xs_sf, const uint8_t* w1_sf, const uint8_t* w1s_sf,
                             uint8_t* h_sc, cudaStream_t s) {
  return launch_mx_gemm(0, a, xs_sf, w1_sf, w1s_sf, h_sc, s);
}

cudaError_t launch_down_mx(const GroupedArgs& a, const uint8_t* h_sf, const uint8_t* w2_sf, const uint8_t* w2s_sf,
                           cudaStream_t s) {
  return launch_mx_gemm(1, a, h_sf, w2_sf, w2s_sf, nullptr, s);
}

}  // namespace moe
