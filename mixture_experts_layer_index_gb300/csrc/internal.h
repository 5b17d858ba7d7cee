// Internal (non-ABI) declarations: workspace layout and kernel launchers.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "moe.h"  // include/ is on the include path (build.py)

namespace moe {

struct DeviceHeader;

constexpr int kGemmBM = 128;          // rows (sorted routes) per grouped-GEMM tile
constexpr int kRouteThreads = 1024;   // threads of the route/rank kernel (32 warps: 4 tokens each at k=8)
constexpr int kMaxRoutesPerBlock = 1024;
constexpr int kMaxE = 512;
constexpr int kMaxK = 32;
constexpr int kMaxShared = 16;        // shared experts of moe_forward_ex
constexpr int kRouteDirectMaxRoutes = 1024;

// Tokens handled by one block of the route/rank kernel (its routes are that times k).
inline int route_tokens_per_block(int k) { return k >= kMaxRoutesPerBlock ? 1 : kMaxRoutesPerBlock / k; }

inline size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

// Byte offsets of the regions of a workspace (every region 256-byte aligned).
struct ShuffleLayout {
  size_t header = 0;
  size_t lrank = 0;        // [R] int32: rank of a route among same-expert routes of its block
  size_t blockcounts = 0;  // [nblk, E] int32 (then per-block base rows after the scan)
  size_t tile_scratch = 0; // [E + 1] int32 (tile prefix of the scan kernel)
  size_t total = 0;
  int nblk = 0;
};

ShuffleLayout plan_shuffle(int T, int E, int k, size_t base);

struct ForwardLayout {
  moe_path path = MOE_PATH_AUTO;
  size_t header = 0;
  size_t ids = 0, w = 0;
  ShuffleLayout shuf;
  size_t counts = 0, offsets = 0, perm = 0, inv = 0;
  size_t tiles = 0, num_tiles = 0;
  int max_tiles = 0;
  size_t xs = 0;      // grouped: [R, H] x rows in sorted order (Gate/Up A operand; bf16 or e4m3)
  size_t xs_scale = 0;  // grouped blockwise FP8: [R, H/128] fp32 scales of xs
  size_t abf = 0;     // grouped per-tensor FP8: [R, I] bf16 a before its quantisation
  size_t h = 0;       // grouped: [R, I] h in sorted order (bf16 or e4m3)
  size_t o = 0;       // grouped: [R, H] bf16 (sorted order); route-direct: [R, H] fp32 (route order)
  // route-direct
  size_t xq = 0;      // [T, H] e4m3 x
  size_t sx = 0;      // [T, H/128] fp32 (blockwise) or [1] fp32 (per-tensor) scales of x
  size_t uniq = 0;    // unique-expert table (see decode.cu)
  size_t part = 0;    // [S, R, 2I] fp32 split-K partials of Gate/Up
  size_t act = 0;     // per-tensor: [R, I] fp32 a;  blockwise: [R, I] e4m3 h
  size_t sh = 0;      // blockwise (both paths): [R, I/128] fp32 scales of h
  // MXFP8 (grouped): E8M0 scale codes, row-major and in the blocked layout
  size_t xs_sc = 0, xs_sf = 0;  // x rows [R, H/32]; blocked per tile
  size_t h_sc = 0, h_sf = 0;    // h rows [R, I/32]; blocked per tile
  size_t w1_sf = 0, w2_sf = 0, w1s_sf = 0, w2s_sf = 0;  // blocked weight scales (routed, shared)
  size_t padbase = 0;           // [E + S] int32: padded-row offset of each expert's rows
  int splits = 1;
  size_t total = 0;
};

// S shared experts (moe_forward_ex) add S*T rows to the grouped path's intermediate tensors.
bool plan_forward(const moe_problem& p, ForwardLayout* out, int S = 0);

// ------------------------------------------------------------------ launchers
// All return cudaSuccess or the launch error; none synchronises.
// amax_x (bf16, amax_n values) non-null: the same launch also records the
// per-tensor amax of x in hdr->amax_x (FP8 per-tensor forward).
cudaError_t launch_route_rank(const float* scores, const int32_t* ids_in, int T, int E, int k, int32_t* ids_out,
                              float* w_out, int32_t* lrank, int32_t* blockcounts, DeviceHeader* hdr, bool route,
                              bool rank, cudaStream_t s, const void* amax_x = nullptr, size_t amax_n = 0);
// With tiles: the routed experts' tiles, then (S > 0) ceil(T/BM) tiles per shared
// expert s, numbered expert E + s, over rows [Rr + s*T, Rr + (s+1)*T) (Rr = T*k).
cudaError_t launch_scan_tiles(int32_t* blockcounts, int nblk, int E, int32_t* counts, int32_t* offsets,
                              int32_t* tiles, int32_t* num_tiles, int max_tiles, int BM, int32_t* tile_scratch,
                              DeviceHeader* hdr, cudaStream_t s, int T = 0, int S = 0, int Rr = 0,
                              int32_t* padbase = nullptr);
cudaError_t launch_scatter(const int32_t* ids, const int32_t* lrank, const int32_t* blockbase, int T, int E, int k,
                           int32_t* perm, int32_t* inv, cudaStream_t s);
// The scatter-gather kernels also copy each token's row to rows R + s*T + t of
// xs for the S shared experts.
cudaError_t launch_scatter_gather(const int32_t* ids, const int32_t* lrank, const int32_t* blockbase, int T, int E,
                                  int k, int H, const void* x, void* xs, int32_t* perm, int32_t* inv,
                                  cudaStream_t s, int S = 0);
// Per-tensor e4m3 passes of the grouped FP8 path (quant.cu).
cudaError_t launch_scatter_gather_q(const int32_t* ids, const int32_t* lrank, const int32_t* blockbase, int T, int E,
                                    int k, int H, const void* x, void* xs, int32_t* perm, int32_t* inv,
                                    const DeviceHeader* hdr, cudaStream_t s, int S = 0);
// h = e4m3(a / s) for n values of bf16 a (n % 8 == 0), s = amax_h / 448 from hdr.
cudaError_t launch_quant_rows(const void* a, void* h, size_t n, const DeviceHeader* hdr, cudaStream_t s);
// Blockwise (one scale per row and 128 columns) passes of the grouped FP8 path (quant.cu).
cudaError_t launch_scatter_gather_qb(const int32_t* ids, const int32_t* lrank, const int32_t* blockbase, int T, int E,
                                     int k, int H, const void* x, void* xs, float* xs_scale, int32_t* perm,
                                     int32_t* inv, cudaStream_t s, int S = 0);
cudaError_t launch_tile_map(const int32_t* counts, int E, int BM, int32_t* tiles, int32_t* num_tiles,
                            int max_tiles, int32_t* tile_scratch, DeviceHeader* hdr, cudaStream_t s);
cudaError_t launch_reset_header(DeviceHeader* hdr, cudaStream_t s);

struct GroupedArgs {
  int T, E, k, H, I;
  int R;                 // rows of the intermediate tensors: T*k routed rows + S*T shared-expert rows
  const void* x;
  const void* xs;        // sorted activations [R, H]; NULL = gather x rows with TMA tile::gather4

  const void* w1;
  const void* w2;
  // S shared experts: tiles with expert id E + s read these weights (and scales)
  int S;
  const void* w1s;
  const void* w2s;
  const float* w1s_scale;
  const float* w2s_scale;
  const int32_t* perm;
  const int32_t* tiles;
  const int32_t* num_tiles;
  int max_tiles;
  void* h;               // Down A operand: bf16 h, or e4m3 h (f8)
  void* o;
  DeviceHeader* hdr;
  // per-tensor FP8 (e4m3 operands): xs/h hold e4m3 codes, x's and a's amax live in hdr
  bool f8;
  const float* w1_scale;
  const float* w2_scale;
  void* a_bf16;          // per-tensor FP8 Gate/Up output a [R, I] bf16 (its amax in hdr, taken in fp32)
};
cudaError_t launch_gateup_bf16(const GroupedArgs& a, cudaStream_t s);  // bf16 or e4m3 (a.f8)
cudaError_t launch_down_bf16(const GroupedArgs& a, cudaStream_t s);
// 128x128-blockwise FP8 grouped GEMMs (grouped_blockwise.cu): xs / h hold e4m3
// codes, their scales [R, H/128] / [R, ceil(I/128)] in sorted row order; the
// Gate/Up quantises h and writes its scales itself.
cudaError_t launch_gateup_blockwise(const GroupedArgs& a, const float* xs_scale, float* h_scale, cudaStream_t s);
cudaError_t launch_down_blockwise(const GroupedArgs& a, const float* h_scale, cudaStream_t s);

// MXFP8 grouped path (mx.cu).  Blocked scale tensors hold (C + 3) / 4 blocks of
// 512 bytes per 128-row block (mx_blocked_bytes).
size_t mx_blocked_bytes(size_t blocks, int C);
// Also writes each row's scales straight into the blocked layout xs_sf (row p of
// expert e at padded row p + padbase[e]).
cudaError_t launch_scatter_gather_mx(const int32_t* ids, const int32_t* lrank, const int32_t* blockbase, int T, int E,
                                     int k, int H, const void* x, void* xs, uint8_t* xs_sc, uint8_t* xs_sf,
                                     const int32_t* padbase, int32_t* perm, int32_t* inv, cudaStream_t s, int S = 0);
// W1 scales [E, 2I, H/32] (blocks of 64 gate + the matching 64 up rows) and W2
// scales [E, H, I/32] (blocks of 128 rows) -> blocked layouts.
cudaError_t launch_mx_blocked_weights(const uint8_t* w1_sc, const uint8_t* w2_sc, int E, int H, int I, uint8_t* w1_sf,
                                      uint8_t* w2_sf, cudaStream_t s);
// Groups of rows given by offsets [G+1] -> their tile map (in ws), padded start
// rows [G+1], and the blocked layout.
cudaError_t launch_mx_group_blocked(const uint8_t* sc, int rows, int C, const int32_t* goff, int G, uint8_t* out,
                                    int32_t* starts, int32_t* tiles, int32_t* num_tiles, int max_tiles,
                                    DeviceHeader* hdr, cudaStream_t s);
// Gate/Up writes h's scales straight into the blocked layout h_sf (block row = tile).
cudaError_t launch_gateup_mx(const GroupedArgs& a, const uint8_t* xs_sf, const uint8_t* w1_sf, const uint8_t* w1s_sf,
                             uint8_t* h_sf, cudaStream_t s);
cudaError_t launch_down_mx(const GroupedArgs& a, const uint8_t* h_sf, const uint8_t* w2_sf, const uint8_t* w2s_sf,
                           cudaStream_t s);

struct CombineArgs {
  int T, k, H;
  const void* o;       // [R + S*T, H]
  bool o_is_f32;
  const float* w;      // [R]
  void* y;             // [T, H] bf16, or fp32 when y_f32
  const int32_t* inv;  // row of route r in o (expert-sorted o), or null: o in route order
  int S = 0;           // shared experts: rows T*k + s*T + t of o are added with weight 1
  bool y_f32 = false;  // write the unrounded fp32 sum
};
cudaError_t launch_combine(const CombineArgs& a, cudaStream_t s);
// Same, launched as a programmatic dependent of the previous kernel on the stream.
cudaError_t launch_combine_pdl(const CombineArgs& a, cudaStream_t s);
// y = bf16(y32), n values (round to nearest even).
cudaError_t launch_round_bf16(const float* y32, void* y, size_t n, cudaStream_t s);

struct DecodeArgs {
  int T, E, k, H, I, R;
  moe_quant quant;
  const void* x;
  const float* scores;
  const uint8_t* w1;
  const uint8_t* w2;
  const float* w1_scale;
  const float* w2_scale;
  int32_t* ids;
  float* w;
  uint8_t* xq;
  float* sx;
  int32_t* uniq;
  float* part;
  void* act;
  float* sh;
  float* o;
  int splits;
  DeviceHeader* hdr;
};
cudaError_t launch_route_direct(const DecodeArgs& a, cudaStream_t s);
size_t route_direct_uniq_bytes(int T, int E, int k);

// Launch `kernel` as a programmatic dependent of the previous work on the stream:
// its launch is prepared while the predecessor runs, and it waits for the
// predecessor on the device (dep_wait) before touching its results.
template <typename... KArgs, typename... Args>
cudaError_t launch_dependent(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                             Args... args) {
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

// Stage timing (moe_profile_start/stop): every launcher brackets its kernel with
// stage_begin/stage_end; both are no-ops unless profiling is on.
void stage_begin(const char* name, cudaStream_t s);
void stage_end(cudaStream_t s);

// Driver entry point for cuTensorMapEncodeTiled (resolved once through the runtime).
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn get_encode_tiled();
int num_sms();

}  // namespace moe
